// plan.h -- schedule and workspace structures shared by the host deriver
// (derive.cpp, api.cpp) and the CUDA kernels.  Plain C++ structs, no CUDA
// types, so both compilers see the same layout.
#pragma once

#include <cstddef>
#include <cstdint>

namespace coll {

constexpr int kMaxRanks = 8;

// Readiness encodings (values match COLL_LL8 / COLL_LL128 / COLL_SENT of coll.h).
enum Encoding : int { ENC_LL8 = 0, ENC_LL128 = 1, ENC_SENT = 2 };

// Bytes per line and bf16 payload elements per line of each encoding.
constexpr int kLL8LineBytes = 8, kLL8Elems = 2;
constexpr int kLL128LineBytes = 128, kLL128Elems = 60;
constexpr int kSentLineBytes = 8, kSentElems = 4;  // one sentinel pack
// Lines of one 16-byte LL8 input chunk / one 512-byte LL128 warp row.
constexpr int kLL8GroupLines = 4;
constexpr int kLL128RowLines = 4;

// Work item kinds: fold the same tile of every rank's image in rank order
// ("Atom::reduce" of Purlin Listing 3) or copy one rank's tile ("Atom::copy").
enum ItemKind : uint8_t { IK_REDUCE = 0, IK_COPY = 1 };

enum ItemFlags : uint8_t {
  IF_PUBLISH = 1,        // write the result as lines into the reduced-partition
                         // region of rank `dst` (twoshot reduce-scatter owner)
  IF_RESET_SOLE = 2,     // sole reader: re-arm the lines it read right away
  IF_RESET_COUNTED = 4,  // one of `readers` readers: the last one re-arms
};

// One consume work item: a tile of lines served for one destination rank.
// Lines are counted within a rank image of the source region.  40 bytes.
struct Item {
  uint8_t kind;      // ItemKind
  uint8_t flags;     // ItemFlags
  uint8_t dst;       // rank whose output (or published partition) this writes
  uint8_t src;       // IK_COPY: the source rank image; IK_REDUCE: unused
  uint16_t readers;  // IF_RESET_COUNTED: readers sharing `counter`
  uint16_t pad0;
  uint32_t nlines;   // lines in the tile (a multiple of the group/row size
                     // except at the end of a segment)
  uint32_t nelems;   // payload elements in the tile
  uint64_t src_line; // first line of the tile in the source image
  uint64_t out_off;  // IF_PUBLISH: first line in dst's image of the reduced
                     // region; otherwise first output element in out[dst]
  uint32_t counter;  // reader counter index (IF_RESET_COUNTED)
  uint32_t pad1;
};
static_assert(sizeof(Item) == 40, "Item layout");

// One staging work item: encode a tile of rank `rank`'s input.  32 bytes.
struct StageItem {
  uint16_t rank;
  uint16_t pad0;
  uint32_t nlines;
  uint32_t nelems;
  uint32_t pad1;
  uint64_t dst_line;  // first line in the rank image
  uint64_t in_elem;   // first input element
};
static_assert(sizeof(StageItem) == 32, "StageItem layout");

// Device-resident control block at the start of the workspace.
struct WsHeader {
  uint64_t epoch;          // current epoch; staging slot = epoch & slot_mask
  uint32_t status_code;    // 0 or a coll_status_t latched by a kernel
  uint32_t status_rank;
  int64_t status_line;
  uint32_t abort;          // nonzero after an error: waits give up at once
  uint32_t arrived;        // CTAs of the run's final launch that read the epoch
  uint32_t started[2];     // fused runs: worker CTAs that started, by slot
  uint64_t rejections;     // stale lines observed (diagnostic)
  // composed twoshot: next task of the run's queue, by slot
  uint32_t task_next[2];
  uint32_t pad0[2];
  uint64_t pad1[24];
};
static_assert(sizeof(WsHeader) == 256, "WsHeader layout");

// A staging region: two or four slots (used in turn by consecutive epochs:
// slot = epoch & slot_mask), each holding one image per rank.
struct Region {
  uint64_t base;        // byte offset of slot 0 from the workspace base
  uint64_t slot_bytes;  // bytes between consecutive slots
  uint64_t slot_mask;   // slots - 1 (1 or 3)
  uint64_t rank_bytes;  // bytes between consecutive rank images
};

// MoE dispatch (scatteredV -> transposedV): routing inputs and the device
// tables the routing kernels fill (all inside the workspace).
// Tokens per routing block (per-block counts and prefixes) and, in the
// composed dispatch, per stage task.
constexpr int kMoeBlockTokens = 16;
constexpr int kMoeSubTokens = 2;
constexpr int kMoeSubs = kMoeBlockTokens / kMoeSubTokens;

struct MoeParams {
  const int32_t* topk[kMaxRanks];  // [tokens * k] expert ids per source
  int tokens, hidden, k, experts, el, nblocks;
  int lag;              // composed dispatch: queue steps from a block's stage to its copies
  uint64_t* flag_stage; // composed dispatch: [N][nblocks * kMoeSubs] epoch once staged
  uint32_t row_lines;   // LL128 lines per staged row (a multiple of 4)
  uint32_t max_rows;    // output rows per destination
  uint32_t* entry_rank; // [N][tokens * k] rank among the block's rows of one expert
  uint32_t* block_off;  // [N][nblocks][experts] block counts, then prefixes
  uint32_t* cnt;        // [N][experts]
  uint32_t* tok_rank;   // [N][tokens][N] rank among the block's tokens bound for
                        // one destination, ~0u if none of its choices lives there
  uint32_t* dblock_off; // [N][nblocks][N] the same per destination: counts, then prefixes
  uint32_t* stage_off;  // [N][N] first staged row of (source, destination)
  uint32_t* out_off;    // [N dest][el][N src] first output row of the block
  uint32_t* rows_dest;  // [N]
  int32_t* counts_out;  // [N dest][el][N src] counts, then rows per destination
};

// One piece of an all-to-all (V) exchange, source p's partition x: its
// place in p's rank image and input, its length, and its offset in
// destination x's output.  The composed all-to-all reads table[p * N + x].
struct ExchPiece {
  uint64_t line0;  // first line in rank p's image
  uint64_t elems;  // 16-bit units (V[p][x], or the uniform partition)
  uint64_t in0;    // offset in rank p's input
  uint64_t out0;   // offset in rank x's output: the earlier sources' lengths
};

// The composed launch (Purlin Algorithm 1), by columns or as a queue of
// tasks: the chunking of every partition, the column lengths, the queue's
// lags and per-task completion flags (epoch values, in the workspace).
struct ComposedParams {
  uint32_t chunk_lines;  // lines of one partition per chunk (multiple of 4)
  uint32_t nchunks;
  // columns (unbounded staging): first_cols staggered columns (groups of
  // `stagger` columns of 1/G .. G/G of a chunk) cover each partition's first
  // first_lines lines; then head_chunks chunks of chunk_lines and the rest in
  // chunks of tail_lines.  nchunks counts the chunks after the staggered
  // columns.
  uint32_t first_cols;
  uint32_t first_lines;
  uint32_t stagger;
  uint32_t head_chunks;
  uint32_t tail_lines;
  int lag;               // queue steps between a chunk's stage and its fold
  int lag2;              // queue steps between a chunk's fold and its gather
  int discard;           // drop consumed lines from L2 (no write-back):
                         // 1 = staged and published lines, 2 = staged only
  int variant;           // launch shape (ring depth and CTAs per SM)
  int schedule;          // 0: columns (one CTA runs a column's stage, fold and
                         // gather phases); 1: a queue of tasks with lags
  int mode;              // 0 all-reduce: stage, fold + publish, gather;
                         // 1 reduce-scatter: stage, fold into the outputs;
                         // 2 all-to-all: stage, copy into the outputs;
                         // 3 all-gather: stage, copy every source's chunk
  uint32_t ring;         // chunk slots the staging images cycle through (0: none,
                         // every chunk has its own place); staged and published
                         // lines of chunk c then carry epoch + c
  uint64_t* flag_stage;  // [nchunks][N]: epoch once rank p staged chunk c
  uint64_t* flag_fold;   // [nchunks][N]: epoch once owner r published chunk c
  uint64_t* gather_cnt;  // [nchunks]: (epoch << 8) | gathers of chunk c done
  const ExchPiece* exch; // all-to-all (V), columns: [N][N] pieces
};

// Everything a kernel launch needs; passed by value (captured by graphs).
struct RunParams {
  char* ws;                       // workspace base
  const uint16_t* in[kMaxRanks];  // rank inputs (stage / late producers)
  uint16_t* out[kMaxRanks];       // rank outputs
  int nranks;
  int enc;
  int dtype;                      // kDtBF16 / kDtF32: how folds read a 32-bit word
  int reset_mode;                 // COLL_RESET_* (LL8 only; LL128 needs none)
  int ctas_per_rank;              // fused path: CTAs bound to each rank
  uint64_t timeout_ns;
  Region P;                       // rank images written by stage
  Region AG;                      // reduced partitions (twoshot)
  const StageItem* sitems;        // grouped by rank: [sbeg[r], sbeg[r+1])
  const Item* items1;             // phase 1, grouped by dst rank
  const Item* items2;             // phase 2 (twoshot), grouped by dst rank
  uint32_t* counters;
  int sbeg[kMaxRanks + 1];
  int beg1[kMaxRanks + 1];
  int beg2[kMaxRanks + 1];
  // Segments of a rank image in region P (identical for every rank when the
  // input layout is scattered): used by late producers to find the input
  // elements of an image line.
  int nseg;
  uint64_t seg_line0[kMaxRanks];
  uint64_t seg_elems[kMaxRanks];
  uint64_t seg_in0[kMaxRanks];
  int interleave1, interleave2;   // streamed consume walks ranks interleaved
  int stage_rank;                 // streamed stage of one rank, -1 = all
  int advance_epoch;              // > 0: this launch ends the run and adds
                                  // this much to the epoch (odd; 1 but for
                                  // the composed launch with cycling staging)
  // late producers (fault-injection runs)
  const int64_t* late_order[kMaxRanks];
  int64_t late_n[kMaxRanks];
  int late_ctas;                  // extra CTAs at the end of the grid
  MoeParams moe;
  ComposedParams cp;
  // withheld staging (fault-injection runs)
  const int64_t* wh_lines;
  const int32_t* wh_kind;
  const uint16_t* wh_poison;
  int64_t wh_n;
};

}  // namespace coll
