// composed.cu -- the twoshot all-reduce as one persistent cooperative launch.
//
// Purlin §3.2 ("Extending the execution to AllReduce", Figure 5, Algorithm 1):
// three CTA groups run concurrently at the granularity of a chunk -- staging
// CTAs, reducer CTAs that fold partition r of every rank and publish it, and
// gather CTAs that copy every published partition into every output.  Here
// the notification between the groups is the LL128 sequence number carried
// by every line (flash-comm §3.1), so the groups need no counters to be
// correct; two counters only keep each group within `window` chunks of the
// next one, so that a chunk's staged and published lines are still in L2 when
// their reader comes (the 126 MiB L2 stands in for the interconnect).
//
// Units (c = chunk, one chunk = chunk_lines lines of every partition):
//   stage  (c, p): rank p's input -> the chunk's lines of its N partitions
//   fold   (c, r): partition r's chunk lines of all N ranks -> folded, published
//   gather (c, d): every owner's published chunk lines -> rank d's output
// Memory ordering per unit: a producer CTA stores all data, __syncthreads,
// every thread fence.acq_rel.gpu, then the sequence numbers (a release
// pattern); a consumer CTA polls every sequence number of the unit, every
// thread fence.acq_rel.gpu, __syncthreads, then reads the data (an acquire
// pattern).  Each line is still checked; the fence is paid once per unit.
// A staged line has exactly one reader (its fold unit), which drops it from
// L2 after reading it (discard.global.L2), so staging never reaches HBM.
#include <cuda_runtime.h>

#include "launch.h"
#include "ll128.cuh"
#include "pipe.cuh"

namespace coll {

constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;
constexpr int kCFoldStages = 3;                      // rows of all N images per warp
constexpr int kCRing = kCFoldStages * kMaxRanks;     // rows per warp (stage / gather)

size_t composed_smem_bytes() { return (size_t)kCWarps * kCRing * kRowBytes; }

__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ int seg_lines_of(const RunParams& P, int k) {
  return (int)((P.seg_elems[k] + kLL128Elems - 1) / kLL128Elems);
}

// Bounded wait for a counter to reach `target` (flow control).
__device__ __forceinline__ bool wait_counter(const RunParams& P, const uint32_t* ctr,
                                             uint32_t target) {
  if (ld_relaxed_u32(ctr) >= target) return true;
  Waiter w;
  while (ld_relaxed_u32(ctr) < target) {
    if (w.expired(P.ws, P.timeout_ns)) {
      latch_error(P.ws, kStatusTimeout, 0xFFFFFFFEu, -3);
      return false;
    }
    __nanosleep(200);
  }
  return true;
}

// Every thread polls its share of a unit's sequence numbers -- all loads
// issued before any is checked -- then fences; the caller's __syncthreads
// completes the acquire for the whole CTA.  `line_addr(i)` gives line i of
// the unit (i < total); at most kPollPerThread lines per thread per batch.
constexpr int kPollPerThread = 8;

template <class F>
__device__ __forceinline__ bool poll_unit(const RunParams& P, int total, uint64_t seq, F line_addr) {
  bool ok = true;
  for (int base = 0; base < total; base += kPollPerThread * (int)blockDim.x) {
    uint64_t v[kPollPerThread];
#pragma unroll
    for (int j = 0; j < kPollPerThread; ++j) {
      const int i = base + j * (int)blockDim.x + (int)threadIdx.x;
      v[j] = i < total ? ld_relaxed_u64(line_addr(i) + 120) : seq;
    }
#pragma unroll
    for (int j = 0; j < kPollPerThread; ++j) {
      const int i = base + j * (int)blockDim.x + (int)threadIdx.x;
      if (ok && v[j] != seq) ok = ll128_wait_seq(P, line_addr(i) + 120, seq, 0, i);
    }
  }
  return ok;
}

__global__ void __launch_bounds__(kCThreads, 2) k_composed_ll128(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  __shared__ int s_ok;
  const uint64_t e = begin_run(P);
  const ComposedParams& Q = P.cp;
  WsHeader* h = header(P.ws);
  const int n = P.nranks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int li = lane >> 3, kk = lane & 7;
  const uint32_t Lc = Q.chunk_lines;
  const int units = (int)Q.nchunks * n;
  const int slot = (int)(e & 1);
  const uint32_t wbase =
      (uint32_t)__cvta_generic_to_shared(smem) + (uint32_t)(warp * kCRing * kRowBytes);
  int role, first, stride;
  if ((int)blockIdx.x < Q.n_stage) {
    role = 0; first = blockIdx.x; stride = Q.n_stage;
  } else if ((int)blockIdx.x < Q.n_stage + Q.n_fold) {
    role = 1; first = blockIdx.x - Q.n_stage; stride = Q.n_fold;
  } else {
    role = 2; first = blockIdx.x - Q.n_stage - Q.n_fold;
    stride = gridDim.x - Q.n_stage - Q.n_fold;
  }
  // payload granules of output chunk q (gather) and of line chunk (li, kk) (stage)
  const int q = lane < 30 ? lane : 29;
  const uint32_t g0off = 128 * ((2 * q) / 15) + 8 * ((2 * q) % 15);
  const uint32_t g1off = 128 * ((2 * q + 1) / 15) + 8 * ((2 * q + 1) % 15);
  const int G = 15 * li + 2 * kk;

  for (int u = first; u < units; u += stride) {
    if (aborted(P.ws)) break;
    const int c = u / n, x = u % n;  // x = rank p (stage), owner r (fold), rank d (gather)
    const uint32_t t0 = (uint32_t)c * Lc;
    if (role == 0) {
      // ---- stage (c, p = x) ------------------------------------------------------
      if (threadIdx.x == 0) {
        s_ok = c < Q.window ||
               wait_counter(P, &h->fold_done[slot], (uint32_t)(c - Q.window + 1) * n);
      }
      __syncthreads();
      if (!s_ok) break;
      // the unit's rows (all N partition tiles) as one stream per warp
      int rows_before[kMaxRanks + 1];
      rows_before[0] = 0;
      for (int k = 0; k < n; ++k) {
        const int nl = max(0, min((int)Lc, seg_lines_of(P, k) - (int)t0));
        rows_before[k + 1] = rows_before[k] + (nl + kLL128RowLines - 1) / kLL128RowLines;
      }
      const int nrows = rows_before[n];
      const int nj = warp < nrows ? (nrows - warp + kCWarps - 1) / kCWarps : 0;
      auto locate = [&](int gr, int& k, int& r) {
        k = 0;
        while (k + 1 < n && gr >= rows_before[k + 1]) ++k;
        r = gr - rows_before[k];
      };
      auto issue = [&](int j) {
        if (j < nj) {
          int k, r;
          locate(warp + j * kCWarps, k, r);
          const int64_t left =
              (int64_t)P.seg_elems[k] - ((int64_t)t0 * kLL128Elems + (int64_t)r * kRowElems);
          const bool valid = lane < 30 && 8 * lane < left;
          const uint16_t* src = P.in[x] + P.seg_in0[k] + (uint64_t)t0 * kLL128Elems +
                                (uint64_t)r * kRowElems + (valid ? 8 * lane : 0);
          cp_async16(wbase + (j % kCRing) * kRowBytes + 16 * lane, src, valid);
        }
        cp_async_commit();
      };
#pragma unroll 1
      for (int j = 0; j < kCRing; ++j) issue(j);
      for (int j = 0; j < nj; ++j) {
        cp_async_wait<kCRing - 1>();
        __syncwarp();
        const uint32_t row = wbase + (j % kCRing) * kRowBytes;
        const uint2 a = lds_v2(row + 8 * G);
        const uint2 b = kk == 7 ? make_uint2(0, 0) : lds_v2(row + 8 * (G + 1));
        __syncwarp();
        issue(j + kCRing);
        int k, r;
        locate(warp + j * kCWarps, k, r);
        const int nl = min((int)Lc, seg_lines_of(P, k) - (int)t0);
        const int nl_row = min((int)kLL128RowLines, nl - r * kLL128RowLines);
        if (li < nl_row) {
          char* dst = image_bytes(P, P.P, e, x) +
                      (P.seg_line0[k] + t0 + (uint64_t)r * kLL128RowLines) * kLL128LineBytes +
                      16 * lane;
          if (kk == 7)
            st_v2u32(dst, a.x, a.y);
          else
            st_v4(dst, make_uint4(a.x, a.y, b.x, b.y));
        }
      }
      cp_async_wait<0>();
      // release: every data store of the CTA, then the numbers
      __syncthreads();
      fence_acq_rel_gpu();
      for (int k = 0; k < n; ++k) {
        const int nl = min((int)Lc, seg_lines_of(P, k) - (int)t0);
        char* img = image_bytes(P, P.P, e, x) + (P.seg_line0[k] + t0) * kLL128LineBytes;
        for (int j = threadIdx.x; j < nl; j += blockDim.x)
          st_relaxed_u64(img + (size_t)j * kLL128LineBytes + 120, e);
      }
    } else if (role == 1) {
      // ---- fold (c, r = x) ---------------------------------------------------------
      const int r = x;
      const int nl = min((int)Lc, seg_lines_of(P, r) - (int)t0);
      if (threadIdx.x == 0) {
        s_ok = c < Q.window ||
               wait_counter(P, &h->gather_done[slot], (uint32_t)(c - Q.window + 1) * n);
      }
      __syncthreads();
      if (!s_ok) break;
      if (nl > 0) {
        const uint64_t src_line = P.seg_line0[r] + t0;
        // acquire every line of the unit
        const bool ok = poll_unit(P, n * nl, e, [&](int idx) {
          return (const char*)image_bytes(P, P.P, e, idx / nl) +
                 (src_line + (uint64_t)(idx % nl)) * kLL128LineBytes;
        });
        fence_acq_rel_gpu();
        if (threadIdx.x == 0) s_ok = 1;
        __syncthreads();
        if (!ok) s_ok = 0;
        __syncthreads();
        if (!s_ok) break;
        const int nrows = (nl + kLL128RowLines - 1) / kLL128RowLines;
        const int nj = warp < nrows ? (nrows - warp + kCWarps - 1) / kCWarps : 0;
        auto issue = [&](int j) {
          if (j < nj) {
            const int rr = warp + j * kCWarps;
            const int nl_row = min((int)kLL128RowLines, nl - rr * kLL128RowLines);
            const uint64_t off =
                (src_line + (uint64_t)rr * kLL128RowLines) * kLL128LineBytes + 16 * lane;
            const uint32_t sl = wbase + (uint32_t)((j % kCFoldStages) * n * kRowBytes);
            for (int p = 0; p < n; ++p)
              cp_async16(sl + p * kRowBytes + 16 * lane, image_bytes(P, P.P, e, p) + off,
                         li < nl_row);
          }
          cp_async_commit();
        };
#pragma unroll
        for (int j = 0; j < kCFoldStages; ++j) issue(j);
        char* ag = image_bytes(P, P.AG, e, r) + (uint64_t)t0 * kLL128LineBytes;
        for (int j = 0; j < nj; ++j) {
          cp_async_wait<kCFoldStages - 1>();
          const uint32_t sl = wbase + (uint32_t)((j % kCFoldStages) * n * kRowBytes);
          uint4 s[kMaxRanks];
#pragma unroll
          for (int p = 0; p < kMaxRanks; ++p)
            if (p < n) s[p] = lds_v4(sl + p * kRowBytes + 16 * lane);
          issue(j + kCFoldStages);
          const int rr = warp + j * kCWarps;
          const int nl_row = min((int)kLL128RowLines, nl - rr * kLL128RowLines);
          // the staged lines of this row have no other reader: drop them
          if (Q.discard && lane < 4 * n && (lane & 3) < nl_row)
            discard_l2_line(image_bytes(P, P.P, e, lane >> 2) +
                            (src_line + (uint64_t)rr * kLL128RowLines + (lane & 3)) *
                                kLL128LineBytes);
          const uint4 res = ll128_fold(s, n);
          if (li < nl_row) {
            char* dst = ag + (size_t)rr * kRowBytes + 16 * lane;
            if (kk == 7)
              st_v2u32(dst, res.x, res.y);
            else
              st_v4(dst, res);
          }
        }
        cp_async_wait<0>();
        __syncthreads();
        fence_acq_rel_gpu();
        for (int j = threadIdx.x; j < nl; j += blockDim.x)
          st_relaxed_u64(ag + (size_t)j * kLL128LineBytes + 120, e);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(&h->fold_done[slot], 1u);
      }
    } else {
      // ---- gather (c, d = x) -------------------------------------------------------
      const int d = x;
      int rows_before[kMaxRanks + 1];
      rows_before[0] = 0;
      for (int r = 0; r < n; ++r) {
        const int nl = max(0, min((int)Lc, seg_lines_of(P, r) - (int)t0));
        rows_before[r + 1] = rows_before[r] + (nl + kLL128RowLines - 1) / kLL128RowLines;
      }
      // owners' chunk tiles have Lc lines except in the last chunk; lines
      // past a shorter tile are skipped by pointing them at a ready line
      const bool ok = poll_unit(P, n * (int)Lc, e, [&](int idx) {
        const int r = idx / (int)Lc, j = idx % (int)Lc;
        const int nl = min((int)Lc, seg_lines_of(P, r) - (int)t0);
        const int jj = j < nl ? j : 0;
        return (const char*)image_bytes(P, P.AG, e, nl > 0 ? r : 0) +
               ((uint64_t)(nl > 0 ? t0 : 0) + jj) * kLL128LineBytes;
      });
      fence_acq_rel_gpu();
      if (threadIdx.x == 0) s_ok = 1;
      __syncthreads();
      if (!ok) s_ok = 0;
      __syncthreads();
      if (!s_ok) break;
      const int nrows = rows_before[n];
      const int nj = warp < nrows ? (nrows - warp + kCWarps - 1) / kCWarps : 0;
      auto locate = [&](int gr, int& r, int& rr) {
        r = 0;
        while (r + 1 < n && gr >= rows_before[r + 1]) ++r;
        rr = gr - rows_before[r];
      };
      auto issue = [&](int j) {
        if (j < nj) {
          int r, rr;
          locate(warp + j * kCWarps, r, rr);
          const int nl = min((int)Lc, seg_lines_of(P, r) - (int)t0);
          const int nl_row = min((int)kLL128RowLines, nl - rr * kLL128RowLines);
          const char* src = image_bytes(P, P.AG, e, r) +
                            ((uint64_t)t0 + (uint64_t)rr * kLL128RowLines) * kLL128LineBytes;
          cp_async16(wbase + (j % kCRing) * kRowBytes + 16 * lane, src + 16 * lane,
                     li < nl_row);
        }
        cp_async_commit();
      };
#pragma unroll 1
      for (int j = 0; j < kCRing; ++j) issue(j);
      for (int j = 0; j < nj; ++j) {
        cp_async_wait<kCRing - 1>();
        __syncwarp();
        const uint32_t row = wbase + (j % kCRing) * kRowBytes;
        const uint2 a = lds_v2(row + g0off), b = lds_v2(row + g1off);
        __syncwarp();
        issue(j + kCRing);
        int r, rr;
        locate(warp + j * kCWarps, r, rr);
        const int64_t left = (int64_t)P.seg_elems[r] - (int64_t)(t0 + rr * kLL128RowLines) * kLL128Elems;
        if (lane < 30 && 8 * lane < left)
          st_v4(P.out[d] + P.seg_in0[r] + (uint64_t)(t0 + rr * kLL128RowLines) * kLL128Elems +
                    8 * lane,
                make_uint4(a.x, a.y, b.x, b.y));
      }
      cp_async_wait<0>();
      __syncthreads();
      if (threadIdx.x == 0) atomicAdd(&h->gather_done[slot], 1u);
    }
  }
  finish_run(P, e);
}

int composed_capacity() {
  int per_sm = 0;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(k_composed_ll128, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)composed_smem_bytes()) != cudaSuccess)
      return 0;
    configured = true;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_composed_ll128, kCThreads,
                                                    composed_smem_bytes()) != cudaSuccess)
    return 0;
  return per_sm * device_sms();
}

cudaError_t launch_composed(const RunParams& P, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = composed_smem_bytes();
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_composed_ll128, P);
}

}  // namespace coll
