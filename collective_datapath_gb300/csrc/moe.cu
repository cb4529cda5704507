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
//  k_moe_count    per (source, block of 128 tokens): per-expert counts and
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
#include <cuda_runtime.h>

#include "launch.h"
#include "ll128.cuh"
#include "pipe.cuh"

namespace coll {

constexpr int kMoeThreads = 256;
constexpr int kMoeBlockTokens = 128;
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
  for (int e = threadIdx.x; e < M.experts; e += blockDim.x) {
    uint32_t run = 0;
    for (int b = 0; b < M.nblocks; ++b) {
      uint32_t* c = M.block_off + ((size_t)p * M.nblocks + b) * M.experts + e;
      const uint32_t v = *c;
      *c = run;  // exclusive prefix over blocks
      run += v;
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
  const MoeParams& M = P.moe;
  const int d = blockIdx.x;
  if (threadIdx.x != 0) return;
  uint32_t run = 0;
  const int n = P.nranks;
  for (int le = 0; le < M.el; ++le)
    for (int p = 0; p < n; ++p) {
      const uint32_t c = M.cnt[(size_t)p * M.experts + d * M.el + le];
      M.out_off[((size_t)d * M.el + le) * n + p] = run;
      M.counts_out[((size_t)d * M.el + le) * n + p] = (int32_t)c;
      run += c;
    }
  M.counts_out[(size_t)n * M.el * n + d] = (int32_t)run;
  M.rows_dest[d] = run;
  if (run > M.max_rows) latch_error(P.ws, kStatusNoMem, d, (int64_t)run);
}

// ---- gather-stage with a TMA bulk load per token row ----------------------------

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t mbar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(mbar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of an mbarrier, giving up after timeout_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t mbar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(mbar, parity))
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  return true;
}
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const void* src, uint32_t bytes,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
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
  static size_t configured = 0;
  if (bytes > 48 * 1024 && bytes > configured) {
    if (cudaError_t e = cudaFuncSetAttribute(k_moe_stage,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes))
      return e;
    configured = bytes;
  }
  const int64_t units = (int64_t)nsrc * M.tokens;
  const int grid = (int)std::min<int64_t>(std::max<int64_t>(units, 1), device_sms() * 8);
  k_moe_stage<<<grid, kMoeThreads, bytes, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_moe_consume(const RunParams& P, cudaStream_t s) {
  const MoeParams& M = P.moe;
  k_moe_scan_dst<<<P.nranks, 32, 0, s>>>(P);
  if (cudaError_t e = cudaGetLastError()) return e;
  const size_t bytes = moe_copy_smem_bytes(P.nranks, M.experts);
  static size_t configured = 0;
  if (bytes > 48 * 1024 && bytes > configured) {
    if (cudaError_t e = cudaFuncSetAttribute(k_moe_copy,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes))
      return e;
    configured = bytes;
  }
  k_moe_copy<<<device_sms() * 4, kMoeThreads, bytes, s>>>(P);
  return cudaGetLastError();
}

}  // namespace coll
