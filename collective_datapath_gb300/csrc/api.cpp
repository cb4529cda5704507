// api.cpp -- the C ABI (include/coll.h): argument checks, workspace binding
// and kernel launches.  No device allocation anywhere in this file.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/coll.h"
#include "derive.h"
#include "launch.h"

using namespace coll;

struct coll_spec {
  Plan plan;
  char* ws = nullptr;
  size_t ws_bytes = 0;
  bool bound = false;
  RunParams base{};
  std::vector<cudaEvent_t> events;  // optional per-launch timing events
  int launches = 0;                 // launches of the current / last run
  const int32_t* topk[kMaxRanks] = {};  // MoE routing per source rank
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cudaStream_t as_stream(coll_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

coll_status_t cuda_status(cudaError_t e) {
  return e == cudaSuccess ? COLL_OK : COLL_ERR_CUDA;
}

// SM count and co-resident fused CTAs of the current device; defaults when
// no device is visible (the deriver is pure host code).
void device_shape(int enc, int* sms, int* cap) {
  int count = 0;
  *sms = 0;
  *cap = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();  // clear the sticky "no device" error
    return;
  }
  *sms = device_sms();
  *cap = fused_capacity(enc);
}

void fill_base(coll_spec* s) {
  const Plan& p = s->plan;
  RunParams& P = s->base;
  P = RunParams{};
  P.ws = s->ws;
  P.nranks = p.n;
  P.enc = p.enc;
  P.reset_mode = p.reset_mode;
  P.dtype = p.dtype;
  P.ctas_per_rank = p.ctas_per_rank;
  P.timeout_ns = p.timeout_ns;
  P.P = p.P;
  P.AG = p.AG;
  P.sitems = reinterpret_cast<const StageItem*>(s->ws + p.off_sitems);
  P.items1 = reinterpret_cast<const Item*>(s->ws + p.off_items1);
  P.items2 = p.items2.empty() ? nullptr : reinterpret_cast<const Item*>(s->ws + p.off_items2);
  P.counters = reinterpret_cast<uint32_t*>(s->ws + p.off_counters);
  for (int r = 0; r <= kMaxRanks; ++r) {
    P.sbeg[r] = p.sbeg[r];
    P.beg1[r] = p.beg1[r];
    P.beg2[r] = p.beg2[r];
  }
  P.nseg = (int)p.pseg[0].size();
  for (int k = 0; k < P.nseg && k < kMaxRanks; ++k) {
    P.seg_line0[k] = p.pseg[0][k].line0;
    P.seg_elems[k] = p.pseg[0][k].elems;
    P.seg_in0[k] = p.pseg[0][k].in_elem;
  }
  auto equal_lists = [&](const int* beg) {
    for (int r = 1; r < p.n; ++r)
      if (beg[r + 1] - beg[r] != beg[1] - beg[0]) return 0;
    return 1;
  };
  P.interleave1 = equal_lists(p.beg1);
  P.interleave2 = equal_lists(p.beg2);
  if (p.kind == CK_MOE) {
    MoeParams& M = P.moe;
    M.tokens = p.moe_tokens;
    M.hidden = p.moe_hidden;
    M.k = p.moe_k;
    M.experts = p.moe_experts;
    M.el = p.moe_el;
    M.nblocks = p.moe_nblocks;
    M.row_lines = p.moe_row_lines;
    M.max_rows = p.moe_max_rows;
    M.entry_rank = reinterpret_cast<uint32_t*>(s->ws + p.off_entry_rank);
    M.block_off = reinterpret_cast<uint32_t*>(s->ws + p.off_block_off);
    M.cnt = reinterpret_cast<uint32_t*>(s->ws + p.off_cnt);
    M.tok_rank = reinterpret_cast<uint32_t*>(s->ws + p.off_tok_rank);
    M.dblock_off = reinterpret_cast<uint32_t*>(s->ws + p.off_dblock_off);
    M.stage_off = reinterpret_cast<uint32_t*>(s->ws + p.off_stage_off);
    M.out_off = reinterpret_cast<uint32_t*>(s->ws + p.off_out_off);
    M.rows_dest = reinterpret_cast<uint32_t*>(s->ws + p.off_rows_dest);
    M.counts_out = reinterpret_cast<int32_t*>(s->ws + p.off_counts_out);
    M.flag_stage = reinterpret_cast<uint64_t*>(s->ws + p.off_moe_flags);
    // composed dispatch: by columns (lag 0), or the queue of stage and copy
    // tasks with this lag in blocks (COLL_MOE_LAG, measurement runs)
    M.lag = 0;
    if (const char* env = std::getenv("COLL_MOE_LAG")) M.lag = std::max(0, std::atoi(env));
    P.sitems = nullptr;
    P.items1 = nullptr;
  }
  P.stage_rank = -1;
  P.advance_epoch = 0;
}

coll_status_t check_outs(const coll_spec* s, void* const* outs) {
  if (outs == nullptr) return COLL_ERR_INVALID;
  for (int r = 0; r < s->plan.n; ++r) {
    if (s->plan.out_elems[r] > 0 && outs[r] == nullptr) return COLL_ERR_INVALID;
    if (!aligned16(outs[r])) return COLL_ERR_ALIGN;
  }
  return COLL_OK;
}

coll_status_t check_ins(const coll_spec* s, const void* const* ins) {
  for (int r = 0; r < s->plan.n; ++r) {
    if (s->plan.in_elems[r] > 0 && ins[r] == nullptr) return COLL_ERR_INVALID;
    if (!aligned16(ins[r])) return COLL_ERR_ALIGN;
  }
  return COLL_OK;
}

// Optional timing: event k is recorded after the k-th launch of a run.
void run_begin(coll_spec* s, cudaStream_t st) {
  s->launches = 0;
  if (!s->events.empty()) cudaEventRecord(s->events[0], st);
}

cudaError_t launched(coll_spec* s, cudaError_t e, cudaStream_t st) {
  if (e != cudaSuccess) return e;
  s->launches += 1;
  if (s->launches < (int)s->events.size()) return cudaEventRecord(s->events[s->launches], st);
  return cudaSuccess;
}

// Shape of the composed launch.  COLL_COMPOSED_SHAPE =
// "chunk_lines,lag,discard,variant,lag2,schedule,tail,tail_hw,stagger"
// overrides the defaults (benchmark sweeps and tests); chunks are a power
// of two of at least kComposedMinChunk lines (the queue counts rows with
// shifts, and its completion flags are laid out for that size).
//
// schedule 0 (default), columns: a column is one chunk of one partition,
// run start to end by one CTA, launch variant 2 (4 warps, 6 CTAs per SM).
// Unbounded staging: the chunk is 64 lines (128 for the all-gather, whose
// column stages one piece and copies it N times), halved down to 32 while
// the co-resident CTAs would get fewer than four columns each, so the last
// round of columns stays a small part of the run.  Measured, 8 ranks, all-
// reduce: 256 MiB 0.89 ms at 64 lines (0.93 at 128, 0.95 at 32); 128 MiB
// 0.46 ms at 64; 32 MiB 0.136-0.139 ms at 32-64; 8 MiB 0.050 ms at 32;
// all-gather 256 MiB 0.396 ms at 128 lines, 0.442 at 64.
// Each CTA's first column is one of a staggered group of `stagger` (8)
// lengths, 1/8 .. 8/8 of a chunk: with equal first columns every CTA staged
// at once (inputs read from HBM while the previous run's outputs were
// written back: the first stage took 16 us against 8.5 later) and the
// phases took three columns to drift apart.  The last columns, over
// `tail_hw` (1) half-rounds of the CTAs' work, are `tail` (16) lines long,
// so that the CTAs run out of work together.  8 ranks, all-reduce, 32 /
// 128 / 256 MiB: 0.1405 / 0.460 / 0.889 ms without, 0.1315 / 0.450 / 0.876
// with both (0.1322 / 0.451 / 0.877 with the stagger alone); all-to-all 32
// / 256 MiB 0.126 / 0.821 ms without, 0.120 / 0.816 with; reduce-scatter
// 0.087 / 0.568 and 0.086 / 0.562.  Not the all-gather.
// Bounded staging: CTA g owns chunk slot g of every rank image, so the
// chunk is the largest of 64 .. 16 lines whose slots cover every co-
// resident CTA, and every column is a chunk.
//
// schedule 1, the queue of tasks (stage, fold, gather per chunk, with lags
// of `lag` and `lag2` steps): defaults measured at 8 x 256 MiB, all-reduce
// 256-line chunks and lag 28, reduce-scatter and all-to-all 128-line chunks
// and lag 40; the all-reduce's chunk is the largest of 256, 128 and 64 lines
// that still gives eight lags' worth of chunks (the queue fills and drains
// over 2 * lag steps).
// CTAs of a launch by columns: the co-resident CTAs, no more than there are
// columns (a short run launches only what it uses), or with bounded staging
// a multiple of N CTAs that each own a chunk slot.  0 if none fit.
int column_grid(const Plan& p, const ComposedParams& q) {
  const int cap = column_capacity(q.variant);
  if (q.ring > 0) {
    int grid = std::min<int>(cap, (int)q.ring);
    grid -= grid % p.n;
    return grid < p.n ? 0 : grid;
  }
  const uint64_t cols = (uint64_t)q.first_cols + (uint64_t)q.nchunks * p.n;
  return (int)std::min<uint64_t>((uint64_t)std::max(cap, 0), cols);
}

ComposedParams composed_shape(const coll_spec* s) {
  const Plan& p = s->plan;
  ComposedParams q{};
  const bool ar = p.kind == CK_ALLREDUCE;
  int chunk = ar ? 256 : 128, lag = ar ? 28 : 40, discard = 1, variant = 0, lag2 = -1,
      schedule = 0, tail = 0, tail_hw = 2, stagger = 0;
  // the longest partition of any rank image (the all-gathers' sources
  // differ in length with V sizes)
  uint64_t most = 0;
  for (int r = 0; r < p.n; ++r)
    for (const Seg& sg : p.pseg[r]) most = std::max<uint64_t>(most, sg.lines);
  const bool gather = p.kind == CK_ALLGATHER || p.kind == CK_ALLGATHER_V;
  const char* env = std::getenv("COLL_COMPOSED_SHAPE");
  if (env != nullptr)
    std::sscanf(env, "%d,%d,%d,%d,%d,%d,%d,%d,%d", &chunk, &lag, &discard, &variant, &lag2,
                &schedule, &tail, &tail_hw, &stagger);
  q.schedule = schedule == 1 ? 1 : 0;
  if (q.schedule == 0 && env == nullptr) {
    variant = 2;
    // the all-gather's columns stage one piece each, and neither form paid
    // there (8 x 256 MiB: 0.392 ms plain, 0.398 with both)
    stagger = gather ? 0 : 8;
    tail = gather ? 0 : 16;
    tail_hw = 1;
  }
  q.variant = variant >= 0 && variant <= 2 ? variant : 0;
  if (q.schedule == 0 && env == nullptr) {
    const uint64_t cap = (uint64_t)std::max(1, column_capacity(q.variant));
    chunk = gather ? 128 : 64;
    if (p.ring_lines > 0) {
      while (chunk > (int)kComposedMinChunk && p.ring_lines / (uint64_t)chunk < cap) chunk /= 2;
    } else {
      while (chunk > 32 && (most + chunk - 1) / chunk * (uint64_t)p.n < 4 * cap) chunk /= 2;
      if ((most + chunk - 1) / chunk * (uint64_t)p.n < cap) {
        // a short run: fewer columns than co-resident CTAs even at 32 lines.
        // 16-line columns, each CTA takes at most one, and no staggered
        // start or short tail (they shape the start and end of long runs)
        chunk = (int)kComposedMinChunk;
        stagger = 0;
        tail = 0;
      }
    }
  } else if (q.schedule == 1 && env == nullptr && ar) {
    while (chunk > 64 && (most + chunk - 1) / chunk < 8ull * (uint64_t)lag) chunk /= 2;
  }
  int c2 = (int)kComposedMinChunk;
  while (c2 * 2 <= chunk && c2 < (1 << 20)) c2 *= 2;
  chunk = c2;
  const uint64_t max_lines = most;
  q.chunk_lines = (uint32_t)chunk;
  q.nchunks = (uint32_t)std::max<uint64_t>(1, (max_lines + chunk - 1) / chunk);
  q.lag = std::max(1, lag);
  q.lag2 = lag2 < 1 ? q.lag : lag2;
  q.ring = 0;
  if (p.ring_lines > 0 && q.schedule == 0) {
    // Bounded staging (Purlin §4.1), columns: ring = chunk slots of each
    // rank image; at least one per partition (the launch takes a multiple
    // of N CTAs, one per slot at most).
    while (q.chunk_lines > kComposedMinChunk && p.ring_lines / q.chunk_lines < (uint64_t)p.n)
      q.chunk_lines /= 2;
    q.nchunks = (uint32_t)std::max<uint64_t>(1, (max_lines + q.chunk_lines - 1) / q.chunk_lines);
    q.ring = (uint32_t)(p.ring_lines / q.chunk_lines);
  } else if (p.ring_lines > 0) {
    // Bounded staging, queue: chunk c uses chunk slot c mod W of the
    // staging images.  A stage waits for the folds (copies) that read the
    // slot's previous chunk, W - lag queue steps back, and a fold for the
    // gathers of its published slot's previous chunk, W - lag2 steps back.
    // Both lags are at most W / 2: every task then waits only for earlier
    // tasks, and no wait is on a task just a few steps back (with lags near
    // W the queue advances one dependent task at a time; 8 x 256 MiB with
    // W = 32 and lags of 28 took 5.0 ms).  The chunk shrinks (to no less
    // than kComposedMinChunk) until the images hold two slots.
    while (q.chunk_lines > kComposedMinChunk &&
           p.ring_lines / ((uint64_t)p.n * q.chunk_lines) < 2)
      q.chunk_lines /= 2;
    // By default the chunk also halves, down to 64 lines, until the images
    // hold 64 chunk slots: longer waits back in the queue pay more than the
    // per-chunk cost (8 x 256 MiB, 4 MiB of staging per rank: 2.92 ms at 256
    // lines, 2.06 at 128, 1.95 at 64; 8 MiB: 1.81, 1.53 and 1.95 ms)
    while (env == nullptr && q.chunk_lines > 64 && q.chunk_lines / 2 >= kComposedMinChunk &&
           p.ring_lines / ((uint64_t)p.n * q.chunk_lines) < 64)
      q.chunk_lines /= 2;
    q.nchunks = (uint32_t)std::max<uint64_t>(1, (max_lines + q.chunk_lines - 1) / q.chunk_lines);
    q.ring = (uint32_t)(p.ring_lines / ((uint64_t)p.n * q.chunk_lines));
    q.lag = std::min(q.lag, std::max(1, (int)q.ring / 2));
    q.lag2 = std::min(q.lag2, std::max(1, (int)q.ring / 2));
  }
  q.first_cols = 0;
  q.first_lines = 0;
  q.stagger = 1;
  q.head_chunks = q.nchunks;
  q.tail_lines = q.chunk_lines;
  if (q.schedule == 0 && q.ring == 0 && ((stagger > 0) || (tail > 0 && tail_hw > 0))) {
    const uint64_t cap = (uint64_t)std::max(1, column_capacity(q.variant));
    const uint64_t CL = q.chunk_lines, cr = CL / kLL128RowLines;
    if (stagger > 0) {
      // one staggered column per CTA of the launch (coll_run's grid): groups
      // of G columns of 1/G .. G/G of a chunk, at least a row each
      const uint64_t G = (uint64_t)std::min(stagger, 64);
      q.stagger = (uint32_t)G;
      q.first_cols = (uint32_t)(cap - cap % (uint64_t)p.n);
      uint64_t rows = 0;
      for (uint64_t j = 0; j < q.first_cols / (uint64_t)p.n; ++j)
        rows += std::max<uint64_t>(1, ((j % G + 1) * cr) / G);
      q.first_lines = (uint32_t)(rows * kLL128RowLines);
    }
    const uint64_t rest = most > q.first_lines ? most - q.first_lines : 0;
    q.head_chunks = (uint32_t)((rest + CL - 1) / CL);
    if (tail > 0 && tail_hw > 0) {
      // columns of `tail` lines for the last `tail_hw` half-rounds of the
      // co-resident CTAs' work
      uint32_t ts = kComposedMinChunk;
      while (ts * 2 <= (uint32_t)tail && ts * 2 < q.chunk_lines) ts *= 2;
      if (ts < q.chunk_lines) {
        const uint64_t tl = (uint64_t)tail_hw * cap * CL / (2 * (uint64_t)p.n);
        q.head_chunks = (uint32_t)((rest > tl ? rest - tl : 0) / CL);
        q.tail_lines = ts;
      }
    }
    const uint64_t after = rest - std::min<uint64_t>(rest, (uint64_t)q.head_chunks * CL);
    q.nchunks = q.head_chunks + (uint32_t)((after + q.tail_lines - 1) / q.tail_lines);
  }
  q.discard = discard;
  q.mode = p.kind == CK_REDUCE_SCATTER || p.kind == CK_REDUCE_SCATTER_V ? 1
           : p.kind == CK_ALLTOALL || p.kind == CK_ALLTOALL_V            ? 2
           : gather                                                      ? 3
                                                                         : 0;
  char* f = s->ws + p.off_cflags;
  q.flag_stage = reinterpret_cast<uint64_t*>(f);
  q.flag_fold = q.flag_stage + p.composed_max_chunks * p.n;
  q.gather_cnt = q.flag_fold + p.composed_max_chunks * p.n;
  q.exch = p.exch.empty() ? nullptr : reinterpret_cast<const ExchPiece*>(s->ws + p.off_exch);
  return q;
}

// One stream-ordered consume phase: phases made only of folds or only of
// plain-output copies run through the
// shared-memory pipelines, when no item re-arms what it read (LL128 lines,
// or the deferred re-arm); anything else through the generic consume kernel.
cudaError_t launch_phase(const Plan& p, const RunParams& P, int phase,
                         const std::vector<Item>& items, cudaStream_t st) {
  const bool pipelined = p.enc == ENC_LL128 ||
                         (p.enc == ENC_LL8 && (p.reset_mode == COLL_RESET_DEFERRED ||
                                               p.reset_mode == COLL_RESET_NONE)) ||
                         (p.enc == ENC_SENT && p.reset_mode == COLL_RESET_DEFERRED);
  if (pipelined && !items.empty()) {
    bool all_fold = true, all_copy = true;
    for (const Item& it : items) {
      all_fold = all_fold && it.kind == IK_REDUCE;
      all_copy = all_copy && it.kind == IK_COPY && !(it.flags & IF_PUBLISH);
    }
    if (all_fold && phase == 1)
      return launch_fold(P, std::min<int>((int)items.size(), device_sms() * 2), st,
                         p.dependent_launch);
    if (all_copy)
      return launch_copy(P, phase, std::min<int>((int)items.size(), device_sms() * 4), st,
                         p.dependent_launch);
  }
  return launch_consume(P, phase, p.consume_grid, st, p.dependent_launch);
}

cudaError_t launch_stager(const Plan& p, const RunParams& P, int items, cudaStream_t st) {
  if (p.enc == ENC_LL128)
    return launch_stage_pipe(P, std::min(items, device_sms() * 4), st, p.dependent_launch);
  return launch_stage(P, std::min(items, device_sms() * 8), st, p.dependent_launch);
}

// Consume phase(s) of a run whose inputs are staged; the last launch
// advances the epoch.
coll_status_t launch_consumers(coll_spec* s, RunParams P, cudaStream_t st) {
  const Plan& p = s->plan;
  const bool rearm_kernel = p.enc != ENC_LL128 && p.reset_mode == COLL_RESET_KERNEL;
  const bool two = !p.items2.empty();
  if (p.items1.empty() && !two) {
    P.advance_epoch = !rearm_kernel;
    if (cudaError_t e = launched(s, launch_advance(P, st), st)) return cuda_status(e);
  } else {
    P.advance_epoch = !two && !rearm_kernel;
    if (cudaError_t e = launched(s, launch_phase(p, P, 1, p.items1, st), st))
      return cuda_status(e);
    if (two) {
      P.advance_epoch = !rearm_kernel;
      if (cudaError_t e = launched(s, launch_phase(p, P, 2, p.items2, st), st))
        return cuda_status(e);
    }
  }
  if (rearm_kernel) {
    P.advance_epoch = 1;
    if (cudaError_t e = launched(s, launch_rearm(P, device_sms() * 4, st), st))
      return cuda_status(e);
  }
  return COLL_OK;
}

}  // namespace

extern "C" {

void coll_options_default(coll_options_t* opt) {
  if (opt == nullptr) return;
  std::memset(opt, 0, sizeof(*opt));
  opt->encoding = COLL_LL8;
  opt->algorithm = COLL_ALGO_AUTO;
  opt->reset_mode = COLL_RESET_DEFERRED;
  opt->path = COLL_PATH_AUTO;
}

coll_status_t coll_spec_create(coll_layout_t in_layout, coll_layout_t out_layout,
                               coll_op_t op, coll_dtype_t dtype, int nranks, size_t count,
                               const coll_options_t* opt, coll_spec_t** spec) {
  if (spec == nullptr) return COLL_ERR_INVALID;
  *spec = nullptr;
  coll_options_t o;
  coll_options_default(&o);
  if (opt != nullptr) o = *opt;
  DeriveInput d{};
  d.in_layout = in_layout;
  d.out_layout = out_layout;
  d.op = op;
  d.dtype = dtype;
  d.nranks = nranks;
  d.count = count;
  d.encoding = o.encoding;
  d.algorithm = o.algorithm;
  d.reset_mode = o.reset_mode;
  d.path = o.path;
  d.ctas = o.ctas;
  d.tile_lines = o.tile_lines;
  d.timeout_ns = o.timeout_ns;
  d.tokens = o.tokens;
  d.hidden = o.hidden;
  d.topk = o.topk;
  d.experts = o.experts;
  d.max_rows = o.max_rows;
  d.slots = o.slots;
  d.staging_bytes = o.staging_bytes;
  if (o.vcounts != nullptr && o.nvcounts > 0)
    d.vcounts.assign(o.vcounts, o.vcounts + o.nvcounts);
  device_shape(o.encoding, &d.sms, &d.fused_capacity);
  coll_spec* s = new (std::nothrow) coll_spec();
  if (s == nullptr) return COLL_ERR_INVALID;
  int st = derive(d, s->plan);
  if (st != COLL_OK) {
    delete s;
    return (coll_status_t)st;
  }
  *spec = s;
  return COLL_OK;
}

coll_status_t coll_workspace_bytes(const coll_spec_t* s, size_t* bytes) {
  if (s == nullptr || bytes == nullptr) return COLL_ERR_INVALID;
  *bytes = (size_t)s->plan.ws_bytes;
  return COLL_OK;
}

coll_status_t coll_buffer_elems(const coll_spec_t* s, int rank, size_t* in_elems,
                                size_t* out_elems) {
  if (s == nullptr || rank < 0 || rank >= s->plan.n) return COLL_ERR_INVALID;
  const uint64_t eu = s->plan.dtype == COLL_F32 ? 2 : 1;  // the plan counts 16-bit units
  if (in_elems) *in_elems = (size_t)(s->plan.in_elems[rank] / eu);
  if (out_elems) *out_elems = (size_t)(s->plan.out_elems[rank] / eu);
  return COLL_OK;
}

coll_status_t coll_bind(coll_spec_t* s, void* dev_workspace, size_t bytes,
                        coll_stream_t stream) {
  if (s == nullptr || dev_workspace == nullptr) return COLL_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(dev_workspace) & 255u) != 0) return COLL_ERR_ALIGN;
  if (bytes < s->plan.ws_bytes) return COLL_ERR_NOMEM;
  cudaStream_t st = as_stream(stream);
  const Plan& p = s->plan;
  s->ws = static_cast<char*>(dev_workspace);
  s->ws_bytes = bytes;
  if (cudaError_t e = cudaMemsetAsync(s->ws, 0, p.ws_bytes, st)) return cuda_status(e);
  if (p.enc == ENC_SENT) {
    // flash-comm §4.2: arrival-checked storage starts out holding the pattern
    for (const Region* R : {&p.P, &p.AG})
      if (R->slot_bytes > 0)
        if (cudaError_t e = cudaMemsetAsync(s->ws + R->base, 0xFF,
                                            (R->slot_mask + 1) * R->slot_bytes, st))
          return cuda_status(e);
  }
  WsHeader h{};
  h.epoch = 1;
  // Pageable sources: the runtime copies them before returning.
  if (cudaError_t e = cudaMemcpyAsync(s->ws, &h, sizeof h, cudaMemcpyHostToDevice, st))
    return cuda_status(e);
  if (!p.sitems.empty())
    if (cudaError_t e = cudaMemcpyAsync(s->ws + p.off_sitems, p.sitems.data(),
                                        p.sitems.size() * sizeof(StageItem),
                                        cudaMemcpyHostToDevice, st))
      return cuda_status(e);
  if (!p.items1.empty())
    if (cudaError_t e = cudaMemcpyAsync(s->ws + p.off_items1, p.items1.data(),
                                        p.items1.size() * sizeof(Item),
                                        cudaMemcpyHostToDevice, st))
      return cuda_status(e);
  if (!p.items2.empty())
    if (cudaError_t e = cudaMemcpyAsync(s->ws + p.off_items2, p.items2.data(),
                                        p.items2.size() * sizeof(Item),
                                        cudaMemcpyHostToDevice, st))
      return cuda_status(e);
  if (!p.exch.empty())
    if (cudaError_t e = cudaMemcpyAsync(s->ws + p.off_exch, p.exch.data(),
                                        p.exch.size() * sizeof(ExchPiece),
                                        cudaMemcpyHostToDevice, st))
      return cuda_status(e);
  if (cudaError_t e = cudaStreamSynchronize(st)) return cuda_status(e);
  fill_base(s);
  s->bound = true;
  return COLL_OK;
}

coll_status_t coll_set_routing(coll_spec_t* s, int rank, const int32_t* dev_topk,
                               coll_stream_t stream) {
  (void)stream;
  if (s == nullptr || dev_topk == nullptr || rank < 0 || rank >= s->plan.n)
    return COLL_ERR_INVALID;
  if (s->plan.kind != CK_MOE) return COLL_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(dev_topk) & 3u) != 0) return COLL_ERR_ALIGN;
  s->topk[rank] = dev_topk;
  return COLL_OK;
}

coll_status_t coll_stage(coll_spec_t* s, int rank, const void* dev_in,
                         coll_stream_t stream) {
  if (s == nullptr || rank < 0 || rank >= s->plan.n) return COLL_ERR_INVALID;
  if (s->plan.ring_lines > 0) return COLL_ERR_UNSUPPORTED;  // staging cycles inside the run
  if (!s->bound) return COLL_ERR_STATE;
  if (s->plan.in_elems[rank] > 0 && dev_in == nullptr) return COLL_ERR_INVALID;
  if (!aligned16(dev_in)) return COLL_ERR_ALIGN;
  RunParams P = s->base;
  P.in[rank] = static_cast<const uint16_t*>(dev_in);
  P.stage_rank = rank;
  if (s->plan.kind == CK_MOE) {
    if (s->topk[rank] == nullptr) return COLL_ERR_STATE;
    for (int r = 0; r < s->plan.n; ++r) P.moe.topk[r] = s->topk[r];
    return cuda_status(launch_moe_stage_all(P, as_stream(stream)));
  }
  const int items = P.sbeg[rank + 1] - P.sbeg[rank];
  return cuda_status(launch_stager(s->plan, P, items, as_stream(stream)));
}

coll_status_t coll_run(coll_spec_t* s, const void* const* dev_ins, void* const* dev_outs,
                       coll_stream_t stream) {
  if (s == nullptr) return COLL_ERR_INVALID;
  if (!s->bound) return COLL_ERR_STATE;
  if (dev_ins == nullptr && s->plan.ring_lines > 0) return COLL_ERR_UNSUPPORTED;
  if (coll_status_t e = check_outs(s, dev_outs)) return e;
  if (dev_ins != nullptr)
    if (coll_status_t e = check_ins(s, dev_ins)) return e;
  const Plan& p = s->plan;
  cudaStream_t st = as_stream(stream);
  RunParams P = s->base;
  for (int r = 0; r < p.n; ++r) {
    P.out[r] = static_cast<uint16_t*>(dev_outs[r]);
    if (dev_ins) P.in[r] = static_cast<const uint16_t*>(dev_ins[r]);
  }
  run_begin(s, st);
  if (p.kind == CK_MOE) {
    for (int r = 0; r < p.n; ++r) {
      if (s->topk[r] == nullptr) return COLL_ERR_STATE;
      P.moe.topk[r] = s->topk[r];
    }
    if (dev_ins != nullptr && p.path == COLL_PATH_COMPOSED) {
      // routing, then stage and copy tasks in one launch
      P.stage_rank = -1;
      if (cudaError_t e = launched(s, launch_moe_routing(P, st), st)) return cuda_status(e);
      P.advance_epoch = 1;
      return cuda_status(launched(s, launch_moe_composed(P, st), st));
    }
    if (dev_ins != nullptr) {
      P.stage_rank = -1;
      if (cudaError_t e = launched(s, launch_moe_stage_all(P, st), st)) return cuda_status(e);
    }
    P.advance_epoch = 1;
    return cuda_status(launched(s, launch_moe_consume(P, st), st));
  }
  const bool empty = p.items1.empty() && p.items2.empty();
  if (dev_ins != nullptr && p.path == COLL_PATH_COMPOSED && !empty) {
    P.cp = composed_shape(s);
    if (P.cp.mode == 3) {
      // all-gather (V): each source stages its own packed segment; the
      // kernel takes source k's segment and its offset in the gathered
      // output, the sum of the earlier sources' lengths
      uint64_t at = 0;
      for (int k = 0; k < p.n; ++k) {
        P.seg_line0[k] = p.pseg[k][0].line0;
        P.seg_elems[k] = p.pseg[k][0].elems;
        P.seg_in0[k] = at;
        at += p.pseg[k][0].elems;
      }
    } else if (P.cp.mode == 2) {
      // all-to-all (V): the pieces come from the exchange table; column x
      // spans the longest source's partition x
      if (P.cp.schedule != 0 && p.kind == CK_ALLTOALL_V) return COLL_ERR_UNSUPPORTED;
      for (int x = 0; x < p.n; ++x) {
        uint64_t most = 0;
        for (int q = 0; q < p.n; ++q) most = std::max<uint64_t>(most, p.pseg[q][x].elems);
        P.seg_elems[x] = most;
      }
    }
    if (P.cp.schedule == 0) {
      const int grid = column_grid(p, P.cp);
      if (grid < 1) return COLL_ERR_CUDA;
      // bounded staging: lines of column q carry epoch + q, so the run moves
      // the epoch past all of them, by an odd step (Purlin §4.2)
      P.advance_epoch =
          P.cp.ring > 0 ? (int)(((uint64_t)P.cp.nchunks * (uint64_t)p.n) | 1u) : 1;
      return cuda_status(launched(s, launch_column(P, grid, st, p.dependent_launch), st));
    }
    const int cap = composed_capacity(P.cp.variant, P.cp.ring > 0);
    if (cap < 3) return COLL_ERR_CUDA;
    // cycling staging: chunk c is notified with epoch + c, so the run moves
    // the epoch past all of them, by an odd step (Purlin §4.2)
    P.advance_epoch = P.cp.ring > 0 ? (int)(P.cp.nchunks | 1u) : 1;
    return cuda_status(launched(s, launch_composed(P, cap, st), st));
  }
  if (dev_ins != nullptr && p.path == COLL_PATH_FUSED && !empty &&
      !(p.enc != ENC_LL128 && p.reset_mode == COLL_RESET_KERNEL)) {
    P.advance_epoch = 1;
    return cuda_status(
        launched(s, launch_fused(P, p.n * p.ctas_per_rank, st, p.dependent_launch), st));
  }
  if (dev_ins != nullptr && !p.sitems.empty()) {
    P.stage_rank = -1;
    if (cudaError_t e = launched(s, launch_stager(p, P, (int)p.sitems.size(), st), st))
      return cuda_status(e);
  }
  return launch_consumers(s, P, st);
}

coll_status_t coll_run_host(coll_spec_t* s, const void* const* host_ins,
                            void* const* dev_ins, void* const* dev_outs,
                            void* const* host_outs, coll_stream_t stream) {
  if (s == nullptr || host_ins == nullptr || dev_ins == nullptr || dev_outs == nullptr ||
      host_outs == nullptr)
    return COLL_ERR_INVALID;
  if (!s->bound) return COLL_ERR_STATE;
  const Plan& p = s->plan;
  cudaStream_t st = as_stream(stream);
  for (int r = 0; r < p.n; ++r) {
    const size_t b = 2 * (size_t)p.in_elems[r];
    if (b && cudaMemcpyAsync(dev_ins[r], host_ins[r], b, cudaMemcpyHostToDevice, st))
      return COLL_ERR_CUDA;
  }
  if (coll_status_t e = coll_run(s, reinterpret_cast<const void* const*>(dev_ins), dev_outs,
                                 stream))
    return e;
  for (int r = 0; r < p.n; ++r) {
    const size_t b = 2 * (size_t)p.out_elems[r];
    if (b && cudaMemcpyAsync(host_outs[r], dev_outs[r], b, cudaMemcpyDeviceToHost, st))
      return COLL_ERR_CUDA;
  }
  return COLL_OK;
}

coll_status_t coll_get_counts(const coll_spec_t* s, int32_t* dev_counts,
                              coll_stream_t stream) {
  if (s == nullptr || dev_counts == nullptr) return COLL_ERR_INVALID;
  if (s->plan.kind != CK_MOE) return COLL_ERR_UNSUPPORTED;
  if (!s->bound) return COLL_ERR_STATE;
  const Plan& p = s->plan;
  const size_t bytes = 4 * ((size_t)p.n * p.moe_el * p.n + p.n);
  return cuda_status(cudaMemcpyAsync(dev_counts, s->ws + p.off_counts_out, bytes,
                                     cudaMemcpyDeviceToDevice, as_stream(stream)));
}

coll_status_t coll_query_status(coll_spec_t* s, coll_stream_t stream, int* code, int* rank,
                                int64_t* line) {
  if (s == nullptr) return COLL_ERR_INVALID;
  if (!s->bound) return COLL_ERR_STATE;
  cudaStream_t st = as_stream(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return COLL_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, s->ws, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
    return COLL_ERR_CUDA;
  if (code) *code = (int)h.status_code;
  if (rank) *rank = (int)h.status_rank;
  if (line) *line = h.status_line;
  if (h.status_code != 0 || h.abort != 0) {
    // Clear status_code .. abort (bytes 8..27) and leave the epoch alone.
    // An aborted run may have skipped items, so the reader counters of the
    // counted re-arm are reset as well.
    char zeros[20] = {0};
    if (cudaMemcpy(s->ws + 8, zeros, sizeof zeros, cudaMemcpyHostToDevice) != cudaSuccess)
      return COLL_ERR_CUDA;
    const size_t cbytes = 4 * (size_t)(s->plan.ncounters ? s->plan.ncounters : 1);
    if (cudaMemset(s->ws + s->plan.off_counters, 0, cbytes) != cudaSuccess)
      return COLL_ERR_CUDA;
  }
  return COLL_OK;
}

coll_status_t coll_get_epoch(coll_spec_t* s, coll_stream_t stream, uint64_t* epoch) {
  if (s == nullptr || epoch == nullptr) return COLL_ERR_INVALID;
  if (!s->bound) return COLL_ERR_STATE;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return COLL_ERR_CUDA;
  if (cudaMemcpy(epoch, s->ws, 8, cudaMemcpyDeviceToHost) != cudaSuccess) return COLL_ERR_CUDA;
  return COLL_OK;
}

coll_status_t coll_get_rejections(coll_spec_t* s, coll_stream_t stream,
                                  uint64_t* rejections) {
  if (s == nullptr || rejections == nullptr) return COLL_ERR_INVALID;
  if (!s->bound) return COLL_ERR_STATE;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return COLL_ERR_CUDA;
  if (cudaMemcpy(rejections, s->ws + offsetof(WsHeader, rejections), 8,
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return COLL_ERR_CUDA;
  return COLL_OK;
}

coll_status_t coll_staging_layout(const coll_spec_t* s, int region, int slot, int rank,
                                  int seg, uint64_t* byte_offset, uint64_t* lines,
                                  int* line_bytes_out) {
  if (s == nullptr || rank < 0 || rank >= s->plan.n || slot < 0 || slot >= s->plan.slots)
    return COLL_ERR_INVALID;
  const Plan& p = s->plan;
  if (p.ring_lines > 0) return COLL_ERR_UNSUPPORTED;  // chunk slots, not segments
  const std::vector<Seg>* segs;
  const Region* R;
  if (region == 0) {
    segs = &p.pseg[rank];
    R = &p.P;
  } else if (region == 1) {
    segs = &p.agseg[rank];
    R = &p.AG;
  } else {
    return COLL_ERR_INVALID;
  }
  if (seg < 0 || seg >= (int)segs->size()) return COLL_ERR_INVALID;
  const int lb = line_bytes(p.enc);
  if (byte_offset)
    *byte_offset = R->base + (uint64_t)slot * R->slot_bytes + (uint64_t)rank * R->rank_bytes +
                   (*segs)[seg].line0 * (uint64_t)lb;
  if (lines) *lines = (*segs)[seg].lines;
  if (line_bytes_out) *line_bytes_out = lb;
  return COLL_OK;
}

coll_status_t coll_stage_withheld(coll_spec_t* s, int rank, const void* dev_in,
                                  const int64_t* dev_lines, const int32_t* dev_kind,
                                  const uint16_t* dev_poison, int64_t n,
                                  coll_stream_t stream) {
  if (n < 0 || (n > 0 && (dev_lines == nullptr || dev_kind == nullptr || dev_poison == nullptr)))
    return COLL_ERR_INVALID;
  if (coll_status_t e = coll_stage(s, rank, dev_in, stream)) return e;
  RunParams P = s->base;
  P.stage_rank = rank;
  P.wh_lines = dev_lines;
  P.wh_kind = dev_kind;
  P.wh_poison = dev_poison;
  P.wh_n = n;
  return cuda_status(launch_withhold(P, as_stream(stream)));
}

coll_status_t coll_run_late(coll_spec_t* s, const void* const* dev_ins, void* const* dev_outs,
                            const int64_t* const* dev_order, const int64_t* n_late,
                            coll_stream_t stream) {
  if (s == nullptr || dev_ins == nullptr || dev_order == nullptr || n_late == nullptr)
    return COLL_ERR_INVALID;
  if (s->plan.ring_lines > 0) return COLL_ERR_UNSUPPORTED;
  if (!s->bound) return COLL_ERR_STATE;
  const Plan& p = s->plan;
  if (p.kind == CK_ALLGATHER || p.kind == CK_ALLGATHER_V || p.kind == CK_ALLTOALL_V ||
      (p.enc != ENC_LL128 && p.reset_mode == COLL_RESET_KERNEL))
    return COLL_ERR_UNSUPPORTED;  // late producers need identical rank images
  if (coll_status_t e = check_outs(s, dev_outs)) return e;
  if (coll_status_t e = check_ins(s, dev_ins)) return e;
  RunParams P = s->base;
  for (int r = 0; r < p.n; ++r) {
    P.out[r] = static_cast<uint16_t*>(dev_outs[r]);
    P.in[r] = static_cast<const uint16_t*>(dev_ins[r]);
    P.late_order[r] = dev_order[r];
    P.late_n[r] = n_late[r];
    if (n_late[r] < 0 || (n_late[r] > 0 && dev_order[r] == nullptr)) return COLL_ERR_INVALID;
  }
  P.sitems = nullptr;  // inputs were staged (with lines withheld)
  P.late_ctas = p.n;
  P.advance_epoch = 1;
  return cuda_status(launch_fused(P, p.n * p.ctas_per_rank + p.n, as_stream(stream), false));
}

coll_status_t coll_debug_items(const coll_spec_t* s, int which, int64_t* buf, size_t cap,
                               size_t* n) {
  if (s == nullptr || n == nullptr || which < 0 || which > 3) return COLL_ERR_INVALID;
  const Plan& p = s->plan;
  if (which == 3) {
    *n = p.exch.size();
    for (size_t i = 0; i < p.exch.size() && i < cap && buf; ++i) {
      const ExchPiece& x = p.exch[i];
      int64_t* o = buf + 10 * i;
      o[0] = (int64_t)(i / p.n); o[1] = (int64_t)(i % p.n);
      o[2] = (int64_t)x.line0; o[3] = (int64_t)x.elems; o[4] = (int64_t)x.in0;
      o[5] = (int64_t)x.out0; o[6] = o[7] = o[8] = o[9] = 0;
    }
    return COLL_OK;
  }
  if (which == 0) {
    *n = p.sitems.size();
    for (size_t i = 0; i < p.sitems.size() && i < cap && buf; ++i) {
      const StageItem& it = p.sitems[i];
      int64_t* o = buf + 10 * i;
      o[0] = it.rank; o[1] = o[2] = o[3] = o[4] = 0;
      o[5] = it.nlines; o[6] = it.nelems; o[7] = (int64_t)it.dst_line;
      o[8] = (int64_t)it.in_elem; o[9] = 0;
    }
    return COLL_OK;
  }
  const std::vector<Item>& v = which == 1 ? p.items1 : p.items2;
  *n = v.size();
  for (size_t i = 0; i < v.size() && i < cap && buf; ++i) {
    const Item& it = v[i];
    int64_t* o = buf + 10 * i;
    o[0] = it.kind; o[1] = it.flags; o[2] = it.dst; o[3] = it.src; o[4] = it.readers;
    o[5] = it.nlines; o[6] = it.nelems; o[7] = (int64_t)it.src_line;
    o[8] = (int64_t)it.out_off; o[9] = it.counter;
  }
  return COLL_OK;
}

coll_status_t coll_debug_plan(const coll_spec_t* s, int* algorithm, int* path,
                              int* ctas_per_rank, int* encoding, int* dependent_launch) {
  if (s == nullptr) return COLL_ERR_INVALID;
  if (dependent_launch) *dependent_launch = s->plan.dependent_launch ? 1 : 0;
  if (algorithm) *algorithm = s->plan.algorithm;
  if (path) *path = s->plan.path;
  if (ctas_per_rank) *ctas_per_rank = s->plan.ctas_per_rank;
  if (encoding) *encoding = s->plan.enc;
  return COLL_OK;
}

coll_status_t coll_set_profile_events(coll_spec_t* s, void* const* events, int n) {
  if (s == nullptr || n < 0 || (n > 0 && events == nullptr)) return COLL_ERR_INVALID;
  s->events.clear();
  for (int i = 0; i < n; ++i) s->events.push_back(static_cast<cudaEvent_t>(events[i]));
  return COLL_OK;
}

coll_status_t coll_launch_floor(coll_spec_t* s, coll_stream_t stream) {
  if (s == nullptr) return COLL_ERR_INVALID;
  const Plan& p = s->plan;
  const bool empty = p.items1.empty() && p.items2.empty();
  if (p.kind != CK_MOE && p.path == COLL_PATH_COMPOSED && !empty) {
    // the launch by columns: its grid, block and attributes
    if (!s->bound) return COLL_ERR_STATE;
    const ComposedParams q = composed_shape(s);
    if (q.schedule != 0) return COLL_ERR_UNSUPPORTED;
    const int grid = column_grid(p, q);
    if (grid < 1) return COLL_ERR_CUDA;
    return cuda_status(launch_floor(grid, as_stream(stream), p.dependent_launch, true,
                                    column_threads(q.variant)));
  }
  if (p.kind == CK_MOE || p.path != COLL_PATH_FUSED || empty ||
      (p.enc != ENC_LL128 && p.reset_mode == COLL_RESET_KERNEL))
    return COLL_ERR_UNSUPPORTED;
  return cuda_status(launch_floor(p.n * p.ctas_per_rank, as_stream(stream), p.dependent_launch));
}

coll_status_t coll_last_launches(const coll_spec_t* s, int* launches) {
  if (s == nullptr || launches == nullptr) return COLL_ERR_INVALID;
  *launches = s->launches;
  return COLL_OK;
}

coll_status_t coll_destroy(coll_spec_t* s) {
  delete s;
  return COLL_OK;
}

const char* coll_status_string(coll_status_t st) {
  switch (st) {
    case COLL_OK: return "ok";
    case COLL_ERR_INVALID: return "invalid argument";
    case COLL_ERR_UNSUPPORTED: return "unsupported collective, type or option";
    case COLL_ERR_ALIGN: return "pointer or count not 16-byte aligned";
    case COLL_ERR_NOMEM: return "workspace smaller than coll_workspace_bytes";
    case COLL_ERR_CUDA: return "CUDA runtime error";
    case COLL_ERR_TIMEOUT: return "a device wait exceeded its time bound";
    case COLL_ERR_STATE: return "call out of sequence";
  }
  return "unknown status";
}

}  // extern "C"
