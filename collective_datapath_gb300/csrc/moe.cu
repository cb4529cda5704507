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
//                 tokens routed to the same expert
//  k_moe_scan_src per source: block prefixes, cnt[p][e], and stage_off[p][e]
//                 (the source's staging image = rows ordered by expert, then
//                 token: one contiguous partition per destination)
//  k_moe_stage    per token row: one 1-D TMA bulk copy of the row into shared
//                 memory, then K LL128 copies of it into the staging image
//  k_moe_scan_dst per destination: out_off[d][le][p], counts, rows
//  k_moe_copy     one warp per output row: validate the row's LL128 lines
//                 through a cp.async ring and unpack them
//  k_moe_composed the stage and copy steps as tasks of one launch (after the
//                 routing kernels), staged rows read back mostly from L2
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
  uint32_t* rank_out = M.entry_rank + (size_t)p * M.tokens * M.k + (size_t)t0 * M.k;
  uint32_t* bcnt = M.block_off + ((size_t)p * M.nblocks + blockIdx.x) * M.experts;
  for (int e = threadIdx.x; e < M.experts; e += blockDim.x) {
    uint32_t c = 0;
    for (int i = 0; i < ne; ++i)
      if (s_topk[i] == e) rank_out[i] = c++;
    bcnt[e] = c;
  }
}

__global__ void __launch_bounds__(kMoeThreads) k_moe_scan_src(RunParams P) {
  const MoeParams& M = P.moe;
  const int p = P.stage_rank >= 0 ? P.stage_rank : (int)blockIdx.x;
  uint32_t* cnt = M.cnt + (size_t)p * M.experts;
  constexpr int kBatch = 16;  // block counts loaded before any is rewritten
  for (int e = threadIdx.x; e < M.experts; e += blockDim.x) {
    uint32_t run = 0;
    uint32_t* col = M.block_off + (size_t)p * M.nblocks * M.experts + e;
    for (int b0 = 0; b0 < M.nblocks; b0 += kBatch) {
      uint32_t v[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        v[j] = b0 + j < M.nblocks ? col[(size_t)(b0 + j) * M.experts] : 0u;
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        if (b0 + j < M.nblocks) {
          col[(size_t)(b0 + j) * M.experts] = run;  // exclusive prefix over blocks
          run += v[j];
        }
    }
    cnt[e] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t run = 0;
    uint32_t* off = M.stage_off + (size_t)p * M.experts;
    for (int e = 0; e < M.experts; ++e) {
      off[e] = run;
      run += cnt[e];
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

__global__ void __launch_bounds__(kMoeThreads) k_moe_stage(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t mbar[2];
  __shared__ int ok_all;
  const uint64_t e = begin_run(P);
  const MoeParams& M = P.moe;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int li = lane >> 3, kk = lane & 7;
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
    for (int j = warp; j < M.k; j += nwarps) {
      const size_t ent = (size_t)t * M.k + j;
      const int ex = M.topk[p][ent];
      if (ex < 0 || ex >= M.experts) continue;
      const uint32_t s = M.stage_off[(size_t)p * M.experts + ex] +
                         M.block_off[((size_t)p * M.nblocks + t / kMoeBlockTokens) * M.experts + ex] +
                         M.entry_rank[(size_t)p * M.tokens * M.k + ent];
      char* dst = img + (uint64_t)s * M.row_lines * kLL128LineBytes;
      for (uint32_t r = 0; r < M.row_lines / kLL128RowLines; ++r) {
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
    __syncthreads();  // the buffer is free for the load after next
  }
  finish_run(P, e);
}

// ---- copy: one warp per output row ----------------------------------------------

constexpr int kMoeRing = 8;

size_t moe_copy_smem_bytes(int nranks, int experts) {
  const int el = experts / nranks;
  return (size_t)(kMoeThreads / 32) * kMoeRing * kRowBytes +
         sizeof(uint32_t) * ((size_t)nranks * el * nranks + (size_t)nranks * experts +
                             kMaxRanks + 1);
}

__global__ void __launch_bounds__(kMoeThreads, 4) k_moe_copy(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const MoeParams& M = P.moe;
  const int n = P.nranks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int ntab = n * M.el * n;
  uint32_t* s_out = reinterpret_cast<uint32_t*>(smem + (size_t)nwarps * kMoeRing * kRowBytes);
  uint32_t* s_stage = s_out + ntab;
  uint32_t* s_pre = s_stage + n * M.experts;
  for (int i = threadIdx.x; i < ntab; i += blockDim.x) s_out[i] = M.out_off[i];
  for (int i = threadIdx.x; i < n * M.experts; i += blockDim.x) s_stage[i] = M.stage_off[i];
  if (threadIdx.x == 0) {
    uint32_t run = 0;
    for (int d = 0; d < n; ++d) {
      s_pre[d] = run;
      run += min(M.rows_dest[d], M.max_rows);
    }
    s_pre[n] = run;
  }
  __syncthreads();
  const uint32_t total = s_pre[n];
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(smem) +
                         (uint32_t)(warp * kMoeRing * kRowBytes);
  const int q = lane < 30 ? lane : 29;
  const uint32_t g0off = 128 * ((2 * q) / 15) + 8 * ((2 * q) % 15);
  const uint32_t g1off = 128 * ((2 * q + 1) / 15) + 8 * ((2 * q + 1) % 15);
  const int nrows = (int)(M.row_lines / kLL128RowLines);
  for (uint32_t v = blockIdx.x * nwarps + warp; v < total; v += gridDim.x * nwarps) {
    if (aborted(P.ws)) break;
    int d = 0;
    while (d + 1 < n && v >= s_pre[d + 1]) ++d;
    const uint32_t o = v - s_pre[d];
    // last (le, p) block whose first row is <= o: it holds row o
    const uint32_t* tab = s_out + (size_t)d * M.el * n;
    int lo = 0, hi = M.el * n;  // upper_bound
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (tab[mid] <= o) lo = mid + 1; else hi = mid;
    }
    const int idx = lo - 1;
    const int le = idx / n, p = idx % n;
    const int ex = d * M.el + le;
    const uint32_t s = s_stage[p * M.experts + ex] + (o - tab[idx]);
    const char* src = P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes + (uint64_t)p * P.P.rank_bytes +
                      (uint64_t)s * M.row_lines * kLL128LineBytes;
    uint16_t* dst = P.out[d] + (uint64_t)o * M.hidden;
    auto issue = [&](int j) {
      if (j < nrows)
        cp_async16(wbase + (j % kMoeRing) * kRowBytes + 16 * lane,
                   src + (size_t)j * kRowBytes + 16 * lane, true);
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kMoeRing; ++j) issue(j);
    bool ok = true;
    for (int j = 0; j < nrows; ++j) {
      cp_async_wait<kMoeRing - 1>();
      __syncwarp();
      const uint32_t slot = wbase + (j % kMoeRing) * kRowBytes;
      const bool ready =
          (lane & 7) != 7 || lds_u64(slot + 16 * lane + 8) == e;
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        const char* grow = src + (size_t)j * kRowBytes;
        if (!ll128_wait_chunk(P, grow, lane, ready, e, p,
                              (int64_t)s * M.row_lines + (int64_t)j * kLL128RowLines)) {
          ok = false;
          break;
        }
        sts_v4(slot + 16 * lane, ld_v4(grow + 16 * lane));
        __syncwarp();
      }
      const uint2 a = lds_v2(slot + g0off), b = lds_v2(slot + g1off);
      __syncwarp();
      issue(j + kMoeRing);
      const int64_t left = (int64_t)M.hidden - (int64_t)j * kRowElems;
      if (lane < 30 && 8 * lane < left)
        st_v4(dst + (size_t)j * kRowElems + 8 * lane, make_uint4(a.x, a.y, b.x, b.y));
    }
    cp_async_wait<0>();
    __syncwarp();
    if (!ok) break;
  }
  finish_run(P, e);
}

// ---- composed dispatch: stage and copy tasks in one launch ---------------------
// The queue of the composed twoshot (composed.cu) applied to the dispatch:
// step b holds the stage tasks of routing block b (source p, kMoeSubTokens
// tokens each: one TMA row load, K LL128 copies) and the copy tasks of block
// b - lag (destination d, source p: every row source p's block routed to an
// expert of d, one warp per row).  A copy task waits for the flags of its
// block's stage tasks; each staged row has exactly that one reader, which
// drops it from L2 once copied, so staged rows rarely reach HBM.
constexpr int kMcWarps = 8, kMcRing = 8;

// Two row buffers, the warps' copy rings, and a prefix table of the local
// experts' row counts (up to 1024 local experts).
size_t moe_composed_smem_bytes(int hidden) {
  return moe_stage_smem_bytes(hidden) + (size_t)kMcWarps * kMcRing * kRowBytes + 4 * 1028;
}

// K LL128 copies of one token row (in shared memory at `row`) into the
// source's staging image; warp j writes choice j.
__device__ __forceinline__ void moe_write_copies(const RunParams& P, const MoeParams& M, int p,
                                                 int t, uint32_t row, uint32_t row_bytes,
                                                 char* img, int lane, int warp, uint64_t e) {
  const int li = lane >> 3, kk = lane & 7;
  for (int j = warp; j < M.k; j += kMcWarps) {
    const size_t ent = (size_t)t * M.k + j;
    const int ex = M.topk[p][ent];
    if (ex < 0 || ex >= M.experts) continue;
    const uint32_t srow = M.stage_off[(size_t)p * M.experts + ex] +
                          M.block_off[((size_t)p * M.nblocks + t / kMoeBlockTokens) * M.experts + ex] +
                          M.entry_rank[(size_t)p * M.tokens * M.k + ent];
    char* dst = img + (uint64_t)srow * M.row_lines * kLL128LineBytes;
    for (uint32_t r = 0; r < M.row_lines / kLL128RowLines; ++r) {
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
}

__global__ void __launch_bounds__(kMcWarps * 32, 3) k_moe_composed(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t mbar[2];
  __shared__ int s_task[2], s_ok;
  __shared__ uint32_t s_rows;                   // rows of the current copy task
  const uint64_t e = begin_run(P);
  const MoeParams& M = P.moe;
  WsHeader* h = header(P.ws);
  const int n = P.nranks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t row_bytes = (uint32_t)M.hidden * 2;
  const uint32_t buf_stride = (row_bytes + 127) / 128 * 128;
  const uint32_t sbuf = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t sbar = (uint32_t)__cvta_generic_to_shared(mbar);
  const uint32_t wbase = sbuf + 2 * buf_stride + (uint32_t)(warp * kMcRing * kRowBytes);
  uint32_t* s_pre = reinterpret_cast<uint32_t*>(smem + 2 * buf_stride +
                                                 (size_t)kMcWarps * kMcRing * kRowBytes);
  const int slot = (int)(e & 1);
  const int per_step = n * kMoeSubs + n * n;
  const int ntasks = (M.nblocks + M.lag) * per_step;
  const int nsub_total = M.nblocks * kMoeSubs;
  const size_t img_stride = P.P.rank_bytes;
  char* img0 = P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes;
  uint32_t uses[2] = {0, 0};                     // thread 0: loads into each buffer so far
  if (threadIdx.x == 0) {
    mbar_init(sbar, 1);
    mbar_init(sbar + 8, 1);
    fence_mbarrier_init();
    s_task[0] = (int)atomicAdd(&h->task_next[slot], 1u);
    s_ok = 1;
  }
  __syncthreads();
  const int q = lane < 30 ? lane : 29;
  const uint32_t g0off = 128 * ((2 * q) / 15) + 8 * ((2 * q) % 15);
  const uint32_t g1off = 128 * ((2 * q + 1) / 15) + 8 * ((2 * q + 1) % 15);
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
        for (int k = 0; k < nt; ++k) {
          fence_proxy_async_smem();
          mbar_expect_tx(sbar + 8 * k, row_bytes);
          tma_load_1d(sbuf + k * buf_stride, P.in[p] + (size_t)(t0 + k) * M.hidden, row_bytes,
                      sbar + 8 * k);
        }
      }
      char* img = img0 + (uint64_t)p * img_stride;
      for (int k = 0; k < nt; ++k) {
        if (threadIdx.x == 0) {
          if (!mbar_wait_bounded(sbar + 8 * k, uses[k] & 1, P.timeout_ns)) {
            latch_error(P.ws, kStatusTimeout, p, (int64_t)(t0 + k));
            s_ok = 0;
            for (int k2 = k + 1; k2 < nt; ++k2)   // let the other load land, bounded
              mbar_wait_bounded(sbar + 8 * k2, uses[k2] & 1, P.timeout_ns);
          }
        }
        __syncthreads();
        if (!s_ok) break;
        moe_write_copies(P, M, p, t0 + k, sbuf + k * buf_stride, row_bytes, img, lane, warp, e);
      }
      if (threadIdx.x == 0)
        for (int k = 0; k < nt; ++k) uses[k] += 1;
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
    // rows of each local expert of d in this block, prefix-summed
    for (int le = threadIdx.x; le < M.el; le += blockDim.x) {
      const int ex = d * M.el + le;
      const uint32_t b0 = M.block_off[((size_t)p * M.nblocks + b) * M.experts + ex];
      const uint32_t b1 = b + 1 < M.nblocks
                              ? M.block_off[((size_t)p * M.nblocks + b + 1) * M.experts + ex]
                              : M.cnt[(size_t)p * M.experts + ex];
      s_pre[le + 1] = b1 - b0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      s_pre[0] = 0;
      for (int le = 0; le < M.el; ++le) s_pre[le + 1] += s_pre[le];
      s_rows = s_pre[M.el];
    }
    __syncthreads();
    if (!s_ok) break;
    const uint32_t rows = s_rows;
    for (uint32_t j = warp; j < rows; j += kMcWarps) {
      int lo = 0, hi = M.el;  // last le with s_pre[le] <= j
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pre[mid] <= j) lo = mid; else hi = mid;
      }
      const int le = lo, ex = d * M.el + le;
      const uint32_t i = j - s_pre[le];
      const uint32_t boff = M.block_off[((size_t)p * M.nblocks + b) * M.experts + ex];
      const uint32_t o = M.out_off[((size_t)d * M.el + le) * n + p] + boff + i;
      if (o >= M.max_rows) continue;  // capacity error, latched by the routing
      const uint32_t srow = M.stage_off[(size_t)p * M.experts + ex] + boff + i;
      const char* src = img0 + (uint64_t)p * img_stride + (uint64_t)srow * M.row_lines * kLL128LineBytes;
      uint16_t* dst = P.out[d] + (uint64_t)o * M.hidden;
      auto issue = [&](int r) {
        if (r < nrows_w)
          cp_async16(wbase + (r % kMcRing) * kRowBytes + 16 * lane, src + (size_t)r * kRowBytes + 16 * lane,
                     true);
        cp_async_commit();
      };
#pragma unroll
      for (int r = 0; r < kMcRing; ++r) issue(r);
      bool ok = true;
      for (int r = 0; r < nrows_w; ++r) {
        cp_async_wait<kMcRing - 1>();
        __syncwarp();
        const uint32_t ring = wbase + (r % kMcRing) * kRowBytes;
        const bool ready = (lane & 7) != 7 || lds_u64(ring + 16 * lane + 8) == e;
        if (!__all_sync(0xFFFFFFFFu, ready)) {
          const char* grow = src + (size_t)r * kRowBytes;
          if (!ll128_wait_chunk(P, grow, lane, ready, e, p,
                                (int64_t)srow * M.row_lines + (int64_t)r * kLL128RowLines)) {
            ok = false;
            break;
          }
          sts_v4(ring + 16 * lane, ld_v4(grow + 16 * lane));
          __syncwarp();
        }
        const uint2 a = lds_v2(ring + g0off), c = lds_v2(ring + g1off);
        __syncwarp();
        issue(r + kMcRing);
        if (lane < 4)  // the row's four lines have no other reader
          asm volatile("discard.global.L2 [%0], 128;" ::"l"(src + (size_t)r * kRowBytes + 128 * lane)
                       : "memory");
        const int64_t left = (int64_t)M.hidden - (int64_t)r * kRowElems;
        if (lane < 30 && 8 * lane < left)
          st_v4(dst + (size_t)r * kRowElems + 8 * lane, make_uint4(a.x, a.y, c.x, c.y));
      }
      cp_async_wait<0>();
      __syncwarp();
      if (!ok) {
        s_ok = 0;
        break;
      }
    }
    __syncthreads();  // s_pre, s_task and s_ok are final
    if (!s_ok) break;
  }
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
  k_moe_scan_src<<<nsrc, kMoeThreads, 0, s>>>(P);
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
  k_moe_scan_src<<<P.nranks, kMoeThreads, 0, s>>>(P);
  if (cudaError_t e = cudaGetLastError()) return e;
  k_moe_scan_dst<<<P.nranks, kMoeThreads, sizeof(uint32_t) * M.el * P.nranks, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_moe_composed(const RunParams& P, cudaStream_t s) {
  const size_t bytes = moe_composed_smem_bytes(P.moe.hidden);
  static size_t memo[kMaxDevices];
  if (cudaError_t e = raise_smem_limit(k_moe_composed, bytes, memo)) return e;
  int per_sm = 0;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_moe_composed,
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
  return cudaLaunchKernelEx(&cfg, k_moe_composed, P);
}

cudaError_t launch_moe_consume(const RunParams& P, cudaStream_t s) {
  const MoeParams& M = P.moe;
  k_moe_scan_dst<<<P.nranks, kMoeThreads, sizeof(uint32_t) * M.el * P.nranks, s>>>(P);
  if (cudaError_t e = cudaGetLastError()) return e;
  const size_t bytes = moe_copy_smem_bytes(P.nranks, M.experts);
  static size_t memo[kMaxDevices];
  if (bytes > 48 * 1024)
    if (cudaError_t e = raise_smem_limit(k_moe_copy, bytes, memo)) return e;
  k_moe_copy<<<device_sms() * 4, kMoeThreads, bytes, s>>>(P);
  return cudaGetLastError();
}

}  // namespace coll
