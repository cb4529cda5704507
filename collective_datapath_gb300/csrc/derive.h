// derive.h -- layout-to-schedule deriver (host only, no CUDA calls).
//
// From (input layout, output layout, op, nranks, count) it derives what the
// pages' orchestration layer derives from a collective's naming (Purlin §3.2
// "Deriving the dependencies from layouts", Listing 2): which rank images
// are staged (one segment per partition of a scattered input, one for a
// packed input), who consumes which segment (a packed output reduces over
// all ranks, a scattered or transposed output copies into rank-ordered
// slots), and for a twoshot all-reduce the composition reduce-scatter ->
// publish -> all-gather (Purlin §3.1 "Composing transformations").  The
// result is a set of per-CTA work lists (tiles of lines) plus the workspace
// layout.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "plan.h"

namespace coll {

enum CollKind { CK_ALLREDUCE, CK_REDUCE_SCATTER, CK_ALLGATHER, CK_ALLTOALL, CK_MOE,
                CK_REDUCE_SCATTER_V, CK_ALLGATHER_V, CK_ALLTOALL_V };

struct Seg {
  uint64_t line0;    // first line in the rank image
  uint64_t lines;    // lines holding payload
  uint64_t elems;    // payload elements
  uint64_t in_elem;  // first element in the rank's input buffer
};

struct DeriveInput {
  int in_layout, out_layout, op, dtype;
  int nranks;
  uint64_t count;
  int encoding, algorithm, reset_mode, path, ctas, tile_lines;
  uint64_t timeout_ns;
  int tokens, hidden, topk, experts, max_rows;
  std::vector<uint64_t> vcounts;  // V collectives (see coll.h)
  int slots;                      // staging slots: 2 or 4 (0 = 2)
  uint64_t staging_bytes;         // per rank image and slot; 0 = whole message
  int sms;             // device SM count (a default when no device is present)
  int fused_capacity;  // co-resident CTAs of the fused kernel
};

struct Plan {
  CollKind kind;
  int dtype = 0;  // COLL_BF16 / COLL_F32; element counts below are 16-bit units
  int algorithm;  // COLL_ONESHOT / COLL_TWOSHOT for all-reduce, else 0
  int enc;
  int n;
  uint64_t count;
  uint64_t shard;  // M: elements per partition
  int path;        // COLL_PATH_FUSED / COLL_PATH_STREAMED (when inputs are given)
  int reset_mode;
  uint64_t timeout_ns;
  int slots = 2;      // staging slots per region
  int ctas_per_rank;  // fused path
  // the run's kernels (fused, or stream-ordered) are launched with
  // programmatic stream serialization, so each one's CTAs are placed while
  // the kernel before it in the stream finishes
  bool dependent_launch = false;
  int consume_grid;   // streamed consume grid
  uint64_t in_elems[kMaxRanks], out_elems[kMaxRanks];
  std::vector<Seg> pseg[kMaxRanks];   // rank images written by stage
  std::vector<Seg> agseg[kMaxRanks];  // reduced partitions (twoshot)
  uint64_t p_rank_lines, ag_rank_lines;
  std::vector<StageItem> sitems;
  std::vector<Item> items1, items2;
  int sbeg[kMaxRanks + 1], beg1[kMaxRanks + 1], beg2[kMaxRanks + 1];
  uint32_t ncounters;
  // MoE dispatch geometry and table offsets
  int moe_tokens = 0, moe_hidden = 0, moe_k = 0, moe_experts = 0, moe_el = 0, moe_nblocks = 0;
  uint32_t moe_row_lines = 0, moe_max_rows = 0;
  uint64_t off_entry_rank = 0, off_block_off = 0, off_cnt = 0, off_tok_rank = 0,
           off_dblock_off = 0, off_stage_off = 0,
           off_out_off = 0, off_rows_dest = 0, off_counts_out = 0, off_moe_flags = 0;
  // workspace layout (byte offsets from the workspace base)
  uint64_t off_sitems, off_items1, off_items2, off_counters;
  // composed twoshot: completion flags for chunks of at least
  // kComposedMinChunk lines (stage, fold: [chunks][N] u64; gather: [chunks] u64)
  uint64_t off_cflags = 0, composed_max_chunks = 0;
  // composed all-to-all (V): the [N][N] exchange pieces
  std::vector<ExchPiece> exch;
  uint64_t off_exch = 0;
  // composed launch with bounded staging: lines of each rank's staging
  // image per slot (chunks cycle through it); 0 = one place per chunk
  uint64_t ring_lines = 0;
  Region P, AG;
  uint64_t ws_bytes;
};

constexpr uint32_t kComposedMinChunk = 16;

// Returns a coll_status_t value (0 = ok).
int derive(const DeriveInput& in, Plan& plan);

int line_bytes(int enc);
int line_elems(int enc);
uint64_t lines_for(int enc, uint64_t elems);
uint64_t shard_elems(uint64_t count, int n);
uint64_t shard_begin(uint64_t count, int n, int r);
uint64_t shard_len(uint64_t count, int n, int r);

}  // namespace coll
