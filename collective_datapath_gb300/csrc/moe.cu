// moe.cu -- layout-derived all-to-all for MoE dispatch (scatteredV ->
// transposedV copy).
//
// Source rank p holds T token rows of H bf16 and a top-K routing (expert ids,
// distinct per token).  Expert e lives on destination d = e / EL as local
// expert le = e % EL (EL = E / N).  Destination d receives, in the order
// (le, source rank, token), every row routed to one of its experts, plus the
// counts[d][le][p].  Purlin §3.1: a transposed output holds what every
// source sent to this rank in source-rank order, and the V variants take
// their partition sizes at runtime; the order inside a destination is this
// library's reading (local expert first, so each expert's rows are
// contiguous).
//
// Steps, all on the device:
//  k_moe_count    per (source, block of 16 tokens): per-expert counts and
//                 the stable rank of every (token, choice) among the block's
//                 tokens routed to the same expert; per destination, the rank
//                 of every token with a choice there among the block's tokens
//  k_moe_scan_src per source (two CTAs: expert columns, destination columns):
//                 block prefixes, cnt[p][e], and stage_off[p][d]
//                 (the source's staging image = rows ordered by destination,
//                 then token: one contiguous partition per destination, each
//                 token staged once for every destination it is routed to)
//  k_moe_stage    per token row: one 1-D TMA bulk copy of the row into shared
//                 memory, then one LL128 copy of it per destination
//  k_moe_scan_dst per destination: out_off[d][le][p], counts, rows
//  k_moe_copy     one warp per staged row: validate its LL128 lines through a
//                 cp.async ring and unpack them into each of the token's
//                 output rows on that destination (one per choice there)
//  k_moe_column   the stage and copy steps in one launch (after the routing
//                 kernels) by columns: one CTA stages a source's token
//                 sub-block and copies those rows into their destinations,
//                 so staged rows are read back from L2 and dropped there
//  k_moe_composed the same launch as a queue of stage and copy tasks with a
//                 lag (selected with COLL_MOE_LAG, measurement runs)
#include <cuda_runtime.h>

#include "launch.h"
#include "ll128.cuh"
#include "pipe.cuh"
#include "tma.cuh"

namespace coll {

constexpr int kMoeThreads = 256;
constexpr uint32_t kStatusInvalid = 1, kStatusNoMem = 4;

// ---- routing ---------------------------------------------------------------------

__global__ void __launch_bounds__(kMoeThreads) k_moe_count(RunParams P) {
  extern __shared__ int32_t s_topk[];
  const MoeParams& M = P.moe;
  const int p = P.stage_rank >= 0 ? P.stage_rank : (int)blockIdx.y;
  const int t0 = blockIdx.x * kMoeBlockTokens;
  const int nt = min(kMoeBlockTokens, M.tokens - t0);
  if (nt <= 0) return;
  const int ne = nt * M.k;
  const int32_t* topk = M.topk[p] + (size_t)t0 * M.k;
  for (int i = threadIdx.x; i < ne; i += blockDim.x) {
    int32_t e = topk[i];
    if (e < 0 || e >= M.experts) {
      latch_error(P.ws, kStatusInvalid, p, (int64_t)t0 * M.k + i);
      e = -1;
    }
    s_topk[i] = e;
  }
  __syncthreads();
  // per (token, destination): does one of the token's choices live there
  const int n = P.nranks;
  __shared__ uint8_t s_on[kMoeBlockTokens * kMaxRanks];
  for (int i = threadIdx.x; i < nt * n; i += blockDim.x) {
    const int tok = i / n, d = i % n;
    bool on = false;
    for (int j = 0; j < M.k; ++j) {
      const int32_t e = s_topk[tok * M.k + j];
      on |= e >= 0 && e / M.el == d;
    }
    s_on[i] = on;
  }
  __syncthreads();
  uint32_t* rank_out = M.entry_rank + (size_t)p * M.tokens * M.k + (size_t)t0 * M.k;
  uint32_t* bcnt = M.block_off + ((size_t)p * M.nblocks + blockIdx.x) * M.experts;
  for (int e = threadIdx.x; e < M.experts; e += blockDim.x) {
    uint32_t c = 0;
    for (int i = 0; i < ne; ++i)
      if (s_topk[i] == e) rank_out[i] = c++;
    bcnt[e] = c;
  }
  // per destination: the block's tokens with at least one choice there, in
  // token order (each is staged once for that destination)
  uint32_t* trank = M.tok_rank + ((size_t)p * M.tokens + t0) * n;
  uint32_t* dcnt = M.dblock_off + ((size_t)p * M.nblocks + blockIdx.x) * n;
  const int d = (int)blockDim.x - 1 - (int)threadIdx.x;  // the last threads: n <= blockDim
  if (d < n) {
    uint32_t c = 0;
    for (int i = 0; i < nt; ++i) trank[(size_t)i * n + d] = s_on[i * n + d] ? c++ : ~0u;
    dcnt[d] = c;
  }
}

// Exclusive prefix over the blocks of one column of a [nblocks][stride]
// table of block counts, in place; returns the column's total.
__device__ uint32_t prefix_blocks(uint32_t* col, size_t stride, int nblocks) {
  constexpr int kBatch = 16;  // block counts loaded before any is rewritten
  uint32_t run = 0;
  for (int b0 = 0; b0 < nblocks; b0 += kBatch) {
    uint32_t v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) v[j] = b0 + j < nblocks ? col[(size_t)(b0 + j) * stride] : 0u;
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      if (b0 + j < nblocks) {
        col[(size_t)(b0 + j) * stride] = run;
        run += v[j];
      }
  }
  return run;
}

__global__ void __launch_bounds__(kMoeThreads) k_moe_scan_src(RunParams P) {
  __shared__ uint32_t s_dcnt[kMaxRanks];
  const MoeParams& M = P.moe;
  const int p = P.stage_rank >= 0 ? P.stage_rank : (int)blockIdx.x;
  const int n = P.nranks;
  if (blockIdx.y == 0) {  // a thread per expert column
    for (int c = threadIdx.x; c < M.experts; c += blockDim.x)
      M.cnt[(size_t)p * M.experts + c] =
          prefix_blocks(M.block_off + (size_t)p * M.nblocks * M.experts + c, M.experts, M.nblocks);
    return;
  }
  // a second CTA per source: a thread per destination column
  for (int d = threadIdx.x; d < n; d += blockDim.x)
    s_dcnt[d] = prefix_blocks(M.dblock_off + (size_t)p * M.nblocks * n + d, n, M.nblocks);
  __syncthreads();
  if (threadIdx.x == 0) {
    // the staging image: one partition per destination, in rank order
    uint32_t run = 0;
    for (int d = 0; d < n; ++d) {
      M.stage_off[(size_t)p * n + d] = run;
      run += s_dcnt[d];
    }
  }
}

__global__ void __launch_bounds__(kMoeThreads) k_moe_scan_dst(RunParams P) {
  extern __shared__ uint32_t s_cnt[];  // [el * n], (le, p) order
  const MoeParams& M = P.moe;
  const int d = blockIdx.x;
  const int n = P.nranks;
  const int m = M.el * n;
  // every count loaded in parallel, then one thread's running sum
  for (int i = threadIdx.x; i < m; i += blockDim.x) {
    const int le = i / n, p = i % n;
    s_cnt[i] = M.cnt[(size_t)p * M.experts + d * M.el + le];
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  uint32_t run = 0;
  for (int i = 0; i < m; ++i) {
    const uint32_t c = s_cnt[i];
    M.out_off[(size_t)d * m + i] = run;
    M.counts_out[(size_t)d * m + i] = (int32_t)c;
    run += c;
  }
  M.counts_out[(size_t)n * m + d] = (int32_t)run;
  M.rows_dest[d] = run;
  if (run > M.max_rows) latch_error(P.ws, kStatusNoMem, d, (int64_t)run);
}

// ---- gather-stage with a TMA bulk load per token row ----------------------------

size_t moe_stage_smem_bytes(int hidden) {
  return 2 * (((size_t)hidden * 2 + 127) / 128 * 128);
}

// First staged row of (source p, token t) for destination d in p's staging
// image, or -1 when none of the token's choices lives on d.
__device__ __forceinline__ int64_t moe_staged_row(const MoeParams& M, int n, int p, int t, int d) {
  const uint32_t r = M.tok_rank[((size_t)p * M.tokens + t) * n + d];
  if (r == ~0u) return -1;
  return (int64_t)M.stage_off[(size_t)p * n + d] +
         M.dblock_off[((size_t)p * M.nblocks + t / kMoeBlockTokens) * n + d] + r;
}

// Writes the token row at `row` (shared memory, row_bytes) as one staged
// LL128 row at `dst`: every 128-byte line holds 60 16-bit units and the
// epoch; a warp writes four lines per step, one 16-byte store per lane,
// steps r0 .. r1-1 of the row.
__device__ __forceinline__ void moe_write_row(char* dst, uint32_t row, uint32_t row_bytes,
                                              uint32_t r0, uint32_t r1, int lane, uint64_t e) {
  const int li = lane >> 3, kk = lane & 7;
  for (uint32_t r = r0; r < r1; ++r) {
    const uint32_t off = (uint32_t)kRowElems * 2 * r + 120 * li + 16 * kk;
    const uint2 a = off < row_bytes ? lds_v2(row + off) : make_uint2(0, 0);
    const uint2 b = (kk < 7 && off + 8 < row_bytes) ? lds_v2(row + off + 8) : make_uint2(0, 0);
    uint4 v = make_uint4(a.x, a.y, b.x, b.y);
    if (kk == 7) {
      v.z = (uint32_t)e;
      v.w = (uint32_t)(e >> 32);
    }
    st_v4(dst + (size_t)r * kRowBytes + 16 * lane, v);
  }
}

__global__ void __launch_bounds__(kMoeThreads) k_moe_stage(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t mbar[2];
  __shared__ int ok_all;
  const uint64_t e = begin_run(P);
  const MoeParams& M = P.moe;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint32_t row_bytes = (uint32_t)M.hidden * 2;
  const uint32_t buf_stride = (row_bytes + 127) / 128 * 128;
  const uint32_t sbuf = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t sbar = (uint32_t)__cvta_generic_to_shared(mbar);
  const int nsrc = P.stage_rank >= 0 ? 1 : P.nranks;
  const int64_t units = (int64_t)nsrc * M.tokens;
  auto unit_src = [&](int64_t u, int& p, int& t) {
    p = P.stage_rank >= 0 ? P.stage_rank : (int)(u / M.tokens);
    t = (int)(u % M.tokens);
  };
  if (threadIdx.x == 0) {
    mbar_init(sbar, 1);
    mbar_init(sbar + 8, 1);
    fence_mbarrier_init();
    ok_all = 1;
  }
  __syncthreads();
  auto issue = [&](int64_t u, int b) {
    int p, t;
    unit_src(u, p, t);
    fence_proxy_async_smem();
    mbar_expect_tx(sbar + 8 * b, row_bytes);
    tma_load_1d(sbuf + b * buf_stride, P.in[p] + (size_t)t * M.hidden, row_bytes, sbar + 8 * b);
  };
  if (threadIdx.x == 0 && (int64_t)blockIdx.x < units) issue(blockIdx.x, 0);
  int it = 0;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x, ++it) {
    const int cur = it & 1;
    if (threadIdx.x == 0 && u + gridDim.x < units) issue(u + gridDim.x, cur ^ 1);
    // bounded wait for this row; after a timeout the prefetch of the other
    // buffer (if any) is waited for too, also bounded, before the CTA leaves
    if (threadIdx.x == 0) {
      if (!mbar_wait_bounded(sbar + 8 * cur, (it >> 1) & 1, P.timeout_ns)) {
        latch_error(P.ws, kStatusTimeout, 0, (int64_t)u);
        ok_all = 0;
        if (u + gridDim.x < units)
          mbar_wait_bounded(sbar + 8 * (cur ^ 1), ((it + 1) >> 1) & 1, P.timeout_ns);
      }
    }
    __syncthreads();
    if (!ok_all) break;
    int p, t;
    unit_src(u, p, t);
    const uint32_t row = sbuf + cur * buf_stride;
    char* img = P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes + (uint64_t)p * P.P.rank_bytes;
    for (int d = warp; d < P.nranks; d += nwarps) {  // one staged row per destination
      const int64_t srow = moe_staged_row(M, P.nranks, p, t, d);
      if (srow >= 0)
        moe_write_row(img + (uint64_t)srow * M.row_lines * kLL128LineBytes, row, row_bytes, 0,
                      M.row_lines / kLL128RowLines, lane, e);
    }
    __syncthreads();  // the buffer is free for the load after next
  }
  finish_run(P, e);
}

// ---- copy: one warp per staged row ---------------------------------------------

constexpr int kMoeRing = 8;

// The output rows of destination d that (source p, token t) fills: lane j
// holds the row of choice j in o0 (choice j + 32 in o1), and the warp-uniform
// masks name the choices that live on d.  Rows past the capacity are left
// out (the routing latched that error).
struct MoeFan {
  uint32_t mask0, mask1, o0, o1;
};

__device__ __forceinline__ MoeFan moe_dest_rows(const MoeParams& M, int n, int p, int t, int d,
                                                int lane) {
  uint32_t o[2] = {0, 0};
  bool on[2] = {false, false};
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int j = lane + 32 * c;
    if (j >= M.k) continue;
    const size_t ent = (size_t)t * M.k + j;
    const int ex = M.topk[p][ent];
    if (ex < 0 || ex >= M.experts || ex / M.el != d) continue;
    const int le = ex - d * M.el;
    o[c] = M.out_off[((size_t)d * M.el + le) * n + p] +
           M.block_off[((size_t)p * M.nblocks + t / kMoeBlockTokens) * M.experts + ex] +
           M.entry_rank[(size_t)p * M.tokens * M.k + ent];
    on[c] = o[c] < M.max_rows;
  }
  MoeFan f;
  f.mask0 = __ballot_sync(0xFFFFFFFFu, on[0]);
  f.mask1 = __ballot_sync(0xFFFFFFFFu, on[1]);
  f.o0 = o[0];
  f.o1 = o[1];
  return f;
}

// Validates steps r0 .. r1-1 (512 bytes, four lines each) of one staged row
// (src: epoch-e LL128 lines staged by source p, the first of them line0 of
// p's image) through the warp's cp.async ring at wbase, and stores each
// step's 240 units into every output row of f.  discard: the row has no
// other reader, so each step's lines leave L2 once read.  false: a line's
// wait ran out (error latched).
template <int kRing>
__device__ __forceinline__ bool moe_copy_row(const RunParams& P, const char* src, int64_t line0,
                                             int p, uint16_t* out_d, int r0, int r1, const MoeFan& f,
                                             uint32_t wbase, int lane, uint64_t e, bool discard) {
  const int hidden = P.moe.hidden;
  const uint64_t pol = l2_evict_first_policy();  // output rows are written once
  const int q = lane < 30 ? lane : 29;
  const uint32_t g0off = 128 * ((2 * q) / 15) + 8 * ((2 * q) % 15);
  const uint32_t g1off = 128 * ((2 * q + 1) / 15) + 8 * ((2 * q + 1) % 15);
  auto issue = [&](int r) {
    if (r < r1)
      cp_async16(wbase + ((r - r0) % kRing) * kRowBytes + 16 * lane,
                 src + (size_t)r * kRowBytes + 16 * lane, true);
    cp_async_commit();
  };
#pragma unroll
  for (int i = 0; i < kRing; ++i) issue(r0 + i);
  bool ok = true;
  for (int r = r0; r < r1; ++r) {
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint32_t slot = wbase + ((r - r0) % kRing) * kRowBytes;
    const bool ready = (lane & 7) != 7 || lds_u64(slot + 16 * lane + 8) == e;
    if (!__all_sync(0xFFFFFFFFu, ready)) {
      const char* grow = src + (size_t)r * kRowBytes;
      if (!ll128_wait_chunk(P, grow, lane, ready, e, p, line0 + (int64_t)r * kLL128RowLines)) {
        ok = false;
        break;
      }
      sts_v4(slot + 16 * lane, ld_v4(grow + 16 * lane));
      __syncwarp();
    }
    const uint2 a = lds_v2(slot + g0off), c = lds_v2(slot + g1off);
    __syncwarp();
    issue(r + kRing);
    if (discard && lane < 4)
      asm volatile("discard.global.L2 [%0], 128;" ::"l"(src + (size_t)r * kRowBytes + 128 * lane)
                   : "memory");
    const int64_t left = (int64_t)hidden - (int64_t)r * kRowElems;
    const bool mine = lane < 30 && 8 * lane < left;
    const uint4 v = make_uint4(a.x, a.y, c.x, c.y);
    uint16_t* col = out_d + (size_t)r * kRowElems + 8 * lane;
    for (uint32_t m = f.mask0; m; m &= m - 1) {
      const uint32_t o = __shfl_sync(0xFFFFFFFFu, f.o0, __ffs(m) - 1);
      if (mine) st_v4_hint(col + (uint64_t)o * hidden, v, pol);
    }
    for (uint32_t m = f.mask1; m; m &= m - 1) {
      const uint32_t o = __shfl_sync(0xFFFFFFFFu, f.o1, __ffs(m) - 1);
      if (mine) st_v4_hint(col + (uint64_t)o * hidden, v, pol);
    }
  }
  cp_async_wait<0>();
  __syncwarp();
  return ok;
}

size_t moe_copy_smem_bytes() { return (size_t)(kMoeThreads / 32) * kMoeRing * kRowBytes; }

// One warp per (source, destination, token) unit, in that order, so each
// warp takes the staged rows of one partition in token order; units whose
// token has no choice on the destination are skipped.
__global__ void __launch_bounds__(kMoeThreads, 4) k_moe_copy(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const MoeParams& M = P.moe;
  const int n = P.nranks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(smem) +
                         (uint32_t)(warp * kMoeRing * kRowBytes);
  const int nrows_w = (int)(M.row_lines / kLL128RowLines);
  const char* img0 = P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes;
  const uint64_t units = (uint64_t)n * n * M.tokens;
  for (uint64_t v = (uint64_t)blockIdx.x * nwarps + warp; v < units; v += (uint64_t)gridDim.x * nwarps) {
    if (aborted(P.ws)) break;
    const int t = (int)(v % (uint64_t)M.tokens);
    const int pd = (int)(v / (uint64_t)M.tokens), p = pd / n, d = pd % n;
    const int64_t srow = moe_staged_row(M, n, p, t, d);
    if (srow < 0) continue;
    const MoeFan f = moe_dest_rows(M, n, p, t, d, lane);
    const char* src = img0 + (uint64_t)p * P.P.rank_bytes + (uint64_t)srow * M.row_lines * kLL128LineBytes;
    if (!moe_copy_row<kMoeRing>(P, src, srow * M.row_lines, p, P.out[d], 0, nrows_w, f, wbase, lane,
                                e, false))
      break;
  }
  finish_run(P, e);
}

// ---- composed dispatch: stage and copy tasks in one launch ---------------------
// The queue of the composed twoshot (composed.cu) applied to the dispatch:
// step b holds the stage tasks of routing block b (source p, kMoeSubTokens
// tokens each: one TMA row load, one LL128 copy per destination) and the copy
// tasks of block b - lag (destination d, source p: the staged rows of source
// p's block for d, one warp per staged row, each unpacked into all of the
// token's output rows on d).  A copy task waits for the flags of its block's
// stage tasks; each staged row has exactly that one reader, which drops it
// from L2 once copied.
constexpr int kMcWarps = 8, kMcRing = 8;
// Each staged row is written and copied as kMcSplit ranges of its 512-byte
// steps, so a task's warps get near-equal shares (the task ends at a CTA
// barrier, where its busiest warp sets the pace).
constexpr int kMcSplit = 2;

// Token-row buffers of the composed and column kernels: one per token of a
// sub-block (the stage kernel's double buffer when sub-blocks are smaller),
// then each warp's copy ring.  Both kernels place the rings after
// kMcRowBufs buffers, so a different sub-block size resizes them together.
constexpr int kMcRowBufs = kMoeSubTokens > 2 ? kMoeSubTokens : 2;
size_t moe_composed_smem_bytes(int hidden) {
  return (size_t)kMcRowBufs * (((size_t)hidden * 2 + 127) / 128 * 128) +
         (size_t)kMcWarps * kMcRing * kRowBytes;
}

__global__ void __launch_bounds__(kMcWarps * 32, 3) k_moe_composed(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t mbar[kMcRowBufs];  // one per token row buffer
  __shared__ int s_task[2], s_ok;
  __shared__ int s_tok[kMoeBlockTokens];        // copy task: its staged rows' tokens
  const uint64_t e = begin_run(P);
  const MoeParams& M = P.moe;
  WsHeader* h = header(P.ws);
  const int n = P.nranks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t row_bytes = (uint32_t)M.hidden * 2;
  const uint32_t buf_stride = (row_bytes + 127) / 128 * 128;
  const uint32_t sbuf = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t sbar = (uint32_t)__cvta_generic_to_shared(mbar);
  const uint32_t wbase = sbuf + kMcRowBufs * buf_stride + (uint32_t)(warp * kMcRing * kRowBytes);
  const int slot = (int)(e & 1);
  const int per_step = n * kMoeSubs + n * n;
  const int ntasks = (M.nblocks + M.lag) * per_step;
  const int nsub_total = M.nblocks * kMoeSubs;
  const size_t img_stride = P.P.rank_bytes;
  char* img0 = P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes;
  uint32_t uses[kMcRowBufs] = {};                // thread 0: loads into each buffer so far
  if (threadIdx.x == 0) {
    for (int k = 0; k < kMcRowBufs; ++k) mbar_init(sbar + 8 * k, 1);
    fence_mbarrier_init();
    s_task[0] = (int)atomicAdd(&h->task_next[slot], 1u);
    s_ok = 1;
  }
  __syncthreads();
  const int nrows_w = (int)(M.row_lines / kLL128RowLines);
  for (int it = 0;; ++it) {
    const int t = s_task[it & 1];
    if (t >= ntasks) break;
    if (threadIdx.x == 0)
      s_task[(it + 1) & 1] = aborted(P.ws) ? ntasks : (int)atomicAdd(&h->task_next[slot], 1u);
    const int step = t / per_step, rem = t % per_step;
    if (rem < n * kMoeSubs) {
      // ---- stage: source p, tokens of sub-block sb of block `step` ---------------
      const int b = step, p = rem / kMoeSubs, sb = rem % kMoeSubs;
      const int t0 = b * kMoeBlockTokens + sb * kMoeSubTokens;
      const int nt = b < M.nblocks ? max(0, min(kMoeSubTokens, M.tokens - t0)) : 0;
      if (nt == 0) {
        __syncthreads();
        continue;
      }
      if (threadIdx.x == 0) {
        const uint64_t in_pol = l2_evict_first_policy();  // token rows are read once
        for (int k = 0; k < nt; ++k) {
          fence_proxy_async_smem();
          mbar_expect_tx(sbar + 8 * k, row_bytes);
          tma_load_1d_hint(sbuf + k * buf_stride, P.in[p] + (size_t)(t0 + k) * M.hidden, row_bytes,
                           sbar + 8 * k, in_pol);
        }
      }
      char* img = img0 + (uint64_t)p * img_stride;
      if (threadIdx.x == 0) {
        for (int k = 0; k < nt; ++k) {  // every load is waited for (bounded), even after a timeout
          if (!mbar_wait_bounded(sbar + 8 * k, uses[k] & 1, P.timeout_ns)) {
            latch_error(P.ws, kStatusTimeout, p, (int64_t)(t0 + k));
            s_ok = 0;
          }
          uses[k] += 1;
        }
      }
      __syncthreads();
      if (s_ok) {
        // the sub-block's staged rows, one per (token, destination with a
        // choice of it), spread over the warps: warp w writes the w-th, the
        // (w + kMcWarps)-th ... of them
        static_assert(kMoeSubTokens * kMaxRanks <= 32, "a lane per (token, destination)");
        int64_t srow = -1;
        if (lane < nt * n) srow = moe_staged_row(M, n, p, t0 + lane / n, lane % n);
        uint32_t real = __ballot_sync(0xFFFFFFFFu, srow >= 0);
        for (int i = 0; real; ++i, real &= real - 1) {
          const int q = __ffs(real) - 1;
          const int64_t sr = __shfl_sync(0xFFFFFFFFu, srow, q);
          for (int part = 0; part < kMcSplit; ++part)
            if ((i * kMcSplit + part) % kMcWarps == warp)
              moe_write_row(img + (uint64_t)sr * M.row_lines * kLL128LineBytes,
                            sbuf + (q / n) * buf_stride, row_bytes, part * nrows_w / kMcSplit,
                            (part + 1) * nrows_w / kMcSplit, lane, e);
        }
      }
      // release: every row of the sub-block is written
      __syncthreads();
      if (threadIdx.x == 0 && s_ok) {
        fence_acq_rel_gpu();
        st_relaxed_u64(M.flag_stage + (size_t)p * nsub_total + b * kMoeSubs + sb, e);
      }
      __syncthreads();
      if (!s_ok) break;
      continue;
    }
    // ---- copy: destination d, source p, block step - lag ---------------------------
    const int idx = rem - n * kMoeSubs, d = idx / n, p = idx % n;
    const int b = step - M.lag;
    if (b < 0 || b >= M.nblocks) {
      __syncthreads();
      continue;
    }
    // acquire: the block's stage tasks of source p
    if ((int)threadIdx.x < kMoeSubs) {
      const int sb = threadIdx.x;
      if (b * kMoeBlockTokens + sb * kMoeSubTokens < M.tokens) {
        const uint64_t* f = M.flag_stage + (size_t)p * nsub_total + b * kMoeSubs + sb;
        if (ld_relaxed_u64(f) != e) {
          Waiter w;
          while (ld_relaxed_u64(f) != e) {
            if (w.expired(P.ws, P.timeout_ns)) {
              latch_error(P.ws, kStatusTimeout, p, -5);
              s_ok = 0;
              break;
            }
            __nanosleep(64);
          }
        }
        fence_acq_rel_gpu();
      }
    }
    // the block's tokens bound for d: consecutive staged rows, in token order
    bool mine = false;
    if ((int)threadIdx.x < kMoeBlockTokens) {
      const int t = b * kMoeBlockTokens + threadIdx.x;
      if (t < M.tokens) {
        const uint32_t r = M.tok_rank[((size_t)p * M.tokens + t) * n + d];
        if (r != ~0u) {
          s_tok[r] = t;
          mine = true;
        }
      }
    }
    const int rows = __syncthreads_count(mine);
    if (!s_ok) break;
    const int64_t row0 = (int64_t)M.stage_off[(size_t)p * n + d] +
                         M.dblock_off[((size_t)p * M.nblocks + b) * n + d];
    for (int u = warp; u < rows * kMcSplit; u += kMcWarps) {
      const int j = u / kMcSplit, part = u % kMcSplit;
      const MoeFan f = moe_dest_rows(M, n, p, s_tok[j], d, lane);
      const int64_t srow = row0 + j;
      const char* src = img0 + (uint64_t)p * img_stride + (uint64_t)srow * M.row_lines * kLL128LineBytes;
      if (!moe_copy_row<kMcRing>(P, src, srow * M.row_lines, p, P.out[d], part * nrows_w / kMcSplit,
                                 (part + 1) * nrows_w / kMcSplit, f, wbase, lane, e, true)) {
        s_ok = 0;
        break;
      }
    }
    __syncthreads();  // s_tok, s_task and s_ok are final
    if (!s_ok) break;
  }
  finish_run(P, e);
}

// ---- dispatch by columns -----------------------------------------------------------
// A column is (source p, one sub-block of kMoeSubTokens tokens), and one CTA
// runs all of it: thread 0 loads the sub-block's token rows into shared
// memory with TMA; the warps stage one LL128 row per (token, destination
// holding one of its experts) -- source p's stage -- and, after a CTA
// barrier, copy each staged row, validated, into every output row of its
// token on that destination -- destination d's copy of what p sent it --
// dropping the staged lines from L2 once read.  The next column's rows load
// while the current one is copied.  CTAs take columns from one counter and
// never wait for each other, and a staged row is read back a few
// microseconds after it was written, by the same SM, before L2 writes it
// back.
__global__ void __launch_bounds__(kMcWarps * 32, 3) k_moe_column(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t mbar[kMcRowBufs];
  __shared__ int s_col[2], s_ok;
  const uint64_t e = begin_run(P);
  const MoeParams& M = P.moe;
  WsHeader* h = header(P.ws);
  const int n = P.nranks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t row_bytes = (uint32_t)M.hidden * 2;
  const uint32_t buf_stride = (row_bytes + 127) / 128 * 128;
  const uint32_t sbuf = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t sbar = (uint32_t)__cvta_generic_to_shared(mbar);
  const uint32_t wbase =
      sbuf + kMcRowBufs * buf_stride + (uint32_t)(warp * kMcRing * kRowBytes);
  const int slot = (int)(e & 1);
  const int ncols = M.nblocks * kMoeSubs * n;
  const int nrows_w = (int)(M.row_lines / kLL128RowLines);
  char* img0 = P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes;
  // column q: source q % n, tokens [t0, t0 + nt) of sub-block q / n
  auto col_src = [&](int q, int& p, int& t0, int& nt) {
    p = q % n;
    t0 = (q / n) * kMoeSubTokens;
    nt = max(0, min(kMoeSubTokens, M.tokens - t0));
  };
  uint32_t uses[kMcRowBufs] = {};  // thread 0: loads waited for, per buffer
  int issued = -1;                    // thread 0: the column whose loads are in flight
  auto load = [&](int q) {            // thread 0
    int p, t0, nt;
    col_src(q, p, t0, nt);
    const uint64_t in_pol = l2_evict_first_policy();  // token rows are read once
    for (int k = 0; k < nt; ++k) {
      fence_proxy_async_smem();
      mbar_expect_tx(sbar + 8 * k, row_bytes);
      tma_load_1d_hint(sbuf + k * buf_stride, P.in[p] + (size_t)(t0 + k) * M.hidden, row_bytes,
                       sbar + 8 * k, in_pol);
    }
    issued = q;
  };
  auto wait_loads = [&](int q) -> bool {  // thread 0, bounded
    int p, t0, nt;
    col_src(q, p, t0, nt);
    bool ok = true;
    for (int k = 0; k < nt; ++k) {
      if (!mbar_wait_bounded(sbar + 8 * k, uses[k] & 1, P.timeout_ns)) {
        latch_error(P.ws, kStatusTimeout, p, (int64_t)(t0 + k));
        ok = false;
      }
      uses[k] += 1;
    }
    issued = -1;
    return ok;
  };
  if (threadIdx.x == 0) {
    for (int k = 0; k < kMcRowBufs; ++k) mbar_init(sbar + 8 * k, 1);
    fence_mbarrier_init();
    s_col[0] = (int)atomicAdd(&h->task_next[slot], 1u);
    s_ok = 1;
    if (s_col[0] < ncols) load(s_col[0]);
  }
  __syncthreads();
  for (int it = 0;; ++it) {
    const int q = s_col[it & 1];
    if (q >= ncols) break;
    int p, t0, nt;
    col_src(q, p, t0, nt);
    if (threadIdx.x == 0 && !wait_loads(q)) s_ok = 0;
    __syncthreads();
    if (!s_ok) break;
    // stage: the sub-block's rows, one per (token, destination with a choice
    // of it); lane j of every warp looks up pair j, warp w writes the parts
    // w, w + kMcWarps, ... of the list
    static_assert(kMoeSubTokens * kMaxRanks <= 32, "a lane per (token, destination)");
    char* img = img0 + (uint64_t)p * P.P.rank_bytes;
    int64_t srow = -1;
    if (lane < nt * n) srow = moe_staged_row(M, n, p, t0 + lane / n, lane % n);
    const uint32_t real = __ballot_sync(0xFFFFFFFFu, srow >= 0);
    {
      uint32_t m = real;
      for (int i = 0; m; ++i, m &= m - 1) {
        const int j = __ffs(m) - 1;
        const int64_t sr = __shfl_sync(0xFFFFFFFFu, srow, j);
        for (int part = 0; part < kMcSplit; ++part)
          if ((i * kMcSplit + part) % kMcWarps == warp)
            moe_write_row(img + (uint64_t)sr * M.row_lines * kLL128LineBytes,
                          sbuf + (j / n) * buf_stride, row_bytes, part * nrows_w / kMcSplit,
                          (part + 1) * nrows_w / kMcSplit, lane, e);
      }
    }
    // the staged rows are written (the barrier orders them before the
    // copies' loads at CTA scope) and the row buffers are free again
    __syncthreads();
    if (threadIdx.x == 0) {
      const int qn = aborted(P.ws) ? ncols : (int)atomicAdd(&h->task_next[slot], 1u);
      s_col[(it + 1) & 1] = qn;
      if (qn < ncols) load(qn);
    }
    // copy: every staged row into its token's output rows on its destination
    {
      uint32_t m = real;
      for (int i = 0; m; ++i, m &= m - 1) {
        const int j = __ffs(m) - 1;
        const int64_t sr = __shfl_sync(0xFFFFFFFFu, srow, j);
        const int t = t0 + j / n, d = j % n;
        bool any = false;
        for (int part = 0; part < kMcSplit; ++part)
          any = any || (i * kMcSplit + part) % kMcWarps == warp;
        if (!any) continue;
        const MoeFan f = moe_dest_rows(M, n, p, t, d, lane);
        const char* src = img + (uint64_t)sr * M.row_lines * kLL128LineBytes;
        for (int part = 0; part < kMcSplit; ++part)
          if ((i * kMcSplit + part) % kMcWarps == warp &&
              !moe_copy_row<kMcRing>(P, src, sr * M.row_lines, p, P.out[d],
                                     part * nrows_w / kMcSplit, (part + 1) * nrows_w / kMcSplit,
                                     f, wbase, lane, e, true))
            s_ok = 0;
      }
    }
    __syncthreads();  // s_col and s_ok are final
    if (!s_ok) break;
  }
  // a column whose rows were requested but that this CTA leaves unprocessed
  // (after an error): wait (bounded) for its loads before the CTA exits
  if (threadIdx.x == 0 && issued >= 0) wait_loads(issued);
  finish_run(P, e);
}

// ---- launchers ------------------------------------------------------------------

cudaError_t launch_moe_stage_all(const RunParams& P, cudaStream_t s) {
  const MoeParams& M = P.moe;
  const int nsrc = P.stage_rank >= 0 ? 1 : P.nranks;
  if (M.tokens > 0) {
    const size_t smem = (size_t)kMoeBlockTokens * M.k * sizeof(int32_t);
    k_moe_count<<<dim3(M.nblocks, nsrc), kMoeThreads, smem, s>>>(P);
    if (cudaError_t e = cudaGetLastError()) return e;
  }
  k_moe_scan_src<<<dim3(nsrc, 2), kMoeThreads, 0, s>>>(P);
  if (cudaError_t e = cudaGetLastError()) return e;
  const size_t bytes = moe_stage_smem_bytes(M.hidden);
  static size_t memo[kMaxDevices];
  if (bytes > 48 * 1024)
    if (cudaError_t e = raise_smem_limit(k_moe_stage, bytes, memo)) return e;
  const int64_t units = (int64_t)nsrc * M.tokens;
  const int grid = (int)std::min<int64_t>(std::max<int64_t>(units, 1), device_sms() * 8);
  k_moe_stage<<<grid, kMoeThreads, bytes, s>>>(P);
  return cudaGetLastError();
}

// Routing only (counts, source and destination prefixes): the composed
// dispatch stages inside its own launch.
cudaError_t launch_moe_routing(const RunParams& P, cudaStream_t s) {
  const MoeParams& M = P.moe;
  if (M.tokens > 0) {
    const size_t smem = (size_t)kMoeBlockTokens * M.k * sizeof(int32_t);
    k_moe_count<<<dim3(M.nblocks, P.nranks), kMoeThreads, smem, s>>>(P);
    if (cudaError_t e = cudaGetLastError()) return e;
  }
  k_moe_scan_src<<<dim3(P.nranks, 2), kMoeThreads, 0, s>>>(P);
  if (cudaError_t e = cudaGetLastError()) return e;
  k_moe_scan_dst<<<P.nranks, kMoeThreads, sizeof(uint32_t) * M.el * P.nranks, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_moe_composed(const RunParams& P, cudaStream_t s) {
  const size_t bytes = moe_composed_smem_bytes(P.moe.hidden);
  const bool columns = P.moe.lag <= 0;
  auto* kernel = columns ? k_moe_column : k_moe_composed;
  static size_t memo[2][kMaxDevices];
  if (cudaError_t e = raise_smem_limit(kernel, bytes, memo[columns ? 1 : 0])) return e;
  int per_sm = 0;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel,
                                                                    kMcWarps * 32, bytes))
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(per_sm * device_sms());
  cfg.blockDim = dim3(kMcWarps * 32);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, P);
}

cudaError_t launch_moe_consume(const RunParams& P, cudaStream_t s) {
  const MoeParams& M = P.moe;
  k_moe_scan_dst<<<P.nranks, kMoeThreads, sizeof(uint32_t) * M.el * P.nranks, s>>>(P);
  if (cudaError_t e = cudaGetLastError()) return e;
  const size_t bytes = moe_copy_smem_bytes();
  static size_t memo[kMaxDevices];
  if (bytes > 48 * 1024)
    if (cudaError_t e = raise_smem_limit(k_moe_copy, bytes, memo)) return e;
  k_moe_copy<<<device_sms() * 4, kMoeThreads, bytes, s>>>(P);
  return cudaGetLastError();
}

}  // namespace coll
