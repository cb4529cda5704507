// kernels.cu -- the datapath kernels and their host-side launchers.
//
//  k_stage     stream-ordered staging of rank inputs into LL lines
//  k_consume   stream-ordered validate + unpack + (fold) + write, per phase
//  k_fold_ll128 / k_copy_ll128 / k_stage_ll128
//              the LL128 fold, copy and stage through per-warp cp.async
//              rings of 512-byte rows (stream-ordered path)
//  k_fold_ll8 / k_copy_ll8
//              the same rings for LL8 lines (stream-ordered path with the
//              deferred or no re-arm)
//  k_fused     one cooperative launch: each CTA serves one emulated rank,
//              stages its tiles, then polls and consumes; optional late
//              producer CTAs publish withheld lines while consumers poll
//  k_withhold  fault injection: overwrite listed lines with stale content
//  k_rearm     LL8 / sentinel re-arm of a whole slot by a separate kernel
//  k_advance   an empty run: only the epoch advances
#include <cuda_runtime.h>

#include "launch.h"
#include "ll128.cuh"
#include "ll8.cuh"
#include "pipe.cuh"
#include "sent.cuh"

namespace coll {

constexpr int kThreads = 256;

template <int ENC, bool kConc>
__device__ __forceinline__ void stage_item(const RunParams& P, const StageItem& it,
                                           uint64_t e) {
  if (ENC == ENC_LL8)
    ll8_stage_tile(P, it, e);
  else if (ENC == ENC_SENT)
    sent_stage_tile(P, it, e);
  else
    ll128_stage_tile<kConc>(P, it, e);
}

template <int ENC, bool kConc>
__device__ __forceinline__ void consume_item(const RunParams& P, const Region& R,
                                             const Item& it, uint64_t e) {
  if (ENC == ENC_LL8)
    ll8_consume_item(P, R, it, e);
  else if (ENC == ENC_SENT)
    sent_consume_item(P, R, it, e);
  else
    ll128_consume_item<kConc>(P, R, it, e);
}

template <int ENC>
__global__ void __launch_bounds__(kThreads) k_stage(RunParams P) {
  const uint64_t e = begin_run(P);
  const int lo = P.stage_rank < 0 ? 0 : P.stage_rank;
  const int hi = P.stage_rank < 0 ? P.nranks : P.stage_rank + 1;
  for (int i = P.sbeg[lo] + blockIdx.x; i < P.sbeg[hi]; i += gridDim.x)
    stage_item<ENC, false>(P, P.sitems[i], e);
}

// Stream-ordered consume.  When every rank has the same item list shape the
// launch walks the items rank-interleaved (item j of rank 0, of rank 1, ...)
// so the ranks that read the same source tile run together and share L2.
template <int ENC>
__global__ void __launch_bounds__(kThreads, 2) k_consume(RunParams P, int phase) {
  const uint64_t e = begin_run(P);
  const Item* items = phase == 1 ? P.items1 : P.items2;
  const int* beg = phase == 1 ? P.beg1 : P.beg2;
  const int n_items = beg[P.nranks];
  const bool inter = phase == 1 ? P.interleave1 : P.interleave2;
  const Region& R = phase == 1 ? P.P : P.AG;
  for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
    if (aborted(P.ws)) break;
    const int i = inter ? beg[v % P.nranks] + v / P.nranks : v;
    consume_item<ENC, false>(P, R, items[i], e);
  }
  finish_run(P, e);
}

// ---- LL128 fold with a cp.async shared-memory pipeline ------------------------
// The unified pipeline of Purlin §3.3 (Algorithm 2) applied to the fold: each
// warp keeps kFoldStages rows of all n rank images in flight in shared memory
// (prime; steady state: wait for the oldest row, read it into registers,
// refetch the slot, validate, fold, write; drain).  A lane only ever copies
// and reads its own 16-byte chunks, so the per-thread cp.async groups need no
// warp synchronisation.  Stream-ordered launches only.
constexpr int kFoldStages = 3;

size_t fold_smem_bytes(int nranks) {
  return (size_t)(kThreads / 32) * kFoldStages * nranks * kRowBytes;
}

__global__ void __launch_bounds__(kThreads, 2) k_fold_ll128(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int n = P.nranks;
  const int li = lane >> 3;
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(smem) +
                         (uint32_t)(warp * kFoldStages * n * kRowBytes + 16 * lane);
  const int n_items = P.beg1[P.nranks];
  for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
    if (aborted(P.ws)) break;
    const int i = P.interleave1 ? P.beg1[v % P.nranks] + v / P.nranks : v;
    const Item it = P.items1[i];
    const bool publish = (it.flags & IF_PUBLISH) != 0;
    const uint32_t nrows = (it.nlines + kLL128RowLines - 1) / kLL128RowLines;
    const int nj = (uint32_t)warp < nrows ? (int)((nrows - warp + nwarps - 1) / nwarps) : 0;
    auto issue = [&](int j) {
      if (j < nj) {
        const uint32_t r = warp + j * nwarps;
        const int nl = min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines));
        const uint64_t off =
            (it.src_line + (uint64_t)r * kLL128RowLines) * kLL128LineBytes + 16 * lane;
        const uint32_t slot = wbase + (uint32_t)((j % kFoldStages) * n * kRowBytes);
        for (int p = 0; p < n; ++p)
          cp_async16(slot + p * kRowBytes, image_bytes(P, P.P, e, p) + off, li < nl);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kFoldStages; ++j) issue(j);
    for (int j = 0; j < nj; ++j) {
      cp_async_wait<kFoldStages - 1>();
      const uint32_t slot = wbase + (uint32_t)((j % kFoldStages) * n * kRowBytes);
      uint4 s[kMaxRanks];
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p)
        if (p < n) s[p] = lds_v4(slot + p * kRowBytes);
      issue(j + kFoldStages);
      const uint32_t r = warp + j * nwarps;
      const int nl = min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines));
      const bool valid = li < nl;
      const uint64_t row_line = it.src_line + (uint64_t)r * kLL128RowLines;
      bool ready = true;
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p)
        if (p < n) ready = ready && ll128_chunk_ready(s[p], lane, valid, e);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        bool ok = true;
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p) {
          if (p < n && ok) {
            const bool rp = ll128_chunk_ready(s[p], lane, valid, e);
            if (!__all_sync(0xFFFFFFFFu, rp)) {
              const char* row = image_bytes(P, P.P, e, p) + row_line * kLL128LineBytes;
              ok = ll128_wait_chunk(P, row, lane, rp, e, p, (int64_t)row_line);
              if (ok && valid) s[p] = ld_v4(row + 16 * lane);
            }
          }
        }
        if (!ok) break;
      }
      const uint4 res = ll128_fold(s, n, P.dtype);
      if (publish) {
        char* dst = image_bytes(P, P.AG, e, it.dst) +
                    (it.out_off + (uint64_t)r * kLL128RowLines) * kLL128LineBytes;
        ll128_store_row<false>(dst, res, lane, nl, e);
      } else {
        const int64_t left = (int64_t)it.nelems - (int64_t)r * kRowElems;
        ll128_write_payload(P.out[it.dst] + it.out_off + (uint64_t)r * kRowElems, res, lane,
                            left);
      }
    }
    cp_async_wait<0>();
  }
  finish_run(P, e);
}

// ---- LL128 copy and stage through cp.async rings --------------------------------
// Copy (all-gather, all-to-all, twoshot phase 2): each warp keeps kCopyStages
// source rows (512 bytes of lines) in flight in shared memory; after a row
// lands the warp validates its sequence numbers and every lane q < 30 gathers
// the two 8-byte payload granules of output chunk q straight from shared
// memory (payload granule G of a row sits in line G / 15 at byte 8 (G % 15)).
// Stage: the same ring holds input rows (480 payload bytes); lane L gathers
// the granules of its line chunk and adds the sequence number.
constexpr int kCopyStages = 8;

size_t copy_smem_bytes() { return (size_t)(kThreads / 32) * kCopyStages * kRowBytes; }

__global__ void __launch_bounds__(kThreads, 4) k_copy_ll128(RunParams P, int phase) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int li = lane >> 3;
  const Item* items = phase == 1 ? P.items1 : P.items2;
  const int* beg = phase == 1 ? P.beg1 : P.beg2;
  const bool inter = phase == 1 ? P.interleave1 : P.interleave2;
  const Region& R = phase == 1 ? P.P : P.AG;
  const int n_items = beg[P.nranks];
  const uint32_t wbase =
      (uint32_t)__cvta_generic_to_shared(smem) + (uint32_t)(warp * kCopyStages * kRowBytes);
  // output chunk q = lane: its two granules
  const int q = lane < 30 ? lane : 29;
  const uint32_t g0off = 128 * ((2 * q) / 15) + 8 * ((2 * q) % 15);
  const uint32_t g1off = 128 * ((2 * q + 1) / 15) + 8 * ((2 * q + 1) % 15);
  for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
    if (aborted(P.ws)) break;
    const int i = inter ? beg[v % P.nranks] + v / P.nranks : v;
    const Item it = items[i];
    const char* src = image_bytes(P, R, e, it.src) + it.src_line * kLL128LineBytes;
    const uint32_t nrows = (it.nlines + kLL128RowLines - 1) / kLL128RowLines;
    const int nj = (uint32_t)warp < nrows ? (int)((nrows - warp + nwarps - 1) / nwarps) : 0;
    auto issue = [&](int j) {
      if (j < nj) {
        const uint32_t r = warp + j * nwarps;
        const int nl = min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines));
        cp_async16(wbase + (j % kCopyStages) * kRowBytes + 16 * lane,
                   src + (size_t)r * kRowBytes + 16 * lane, li < nl);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kCopyStages; ++j) issue(j);
    for (int j = 0; j < nj; ++j) {
      cp_async_wait<kCopyStages - 1>();
      __syncwarp();
      const uint32_t row = wbase + (j % kCopyStages) * kRowBytes;
      const uint32_t r = warp + j * nwarps;
      const int nl = min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines));
      const bool valid = li < nl;
      const bool ready = !(valid && (lane & 7) == 7) || lds_u64(row + 16 * lane + 8) == e;
      if (!__all_sync(0xFFFFFFFFu, ready)) {
        const char* grow = src + (size_t)r * kRowBytes;
        if (!ll128_wait_chunk(P, grow, lane, ready, e, it.src,
                              (int64_t)(it.src_line + r * kLL128RowLines)))
          break;
        if (valid) sts_v4(row + 16 * lane, ld_v4(grow + 16 * lane));
        __syncwarp();
      }
      const uint2 a = lds_v2(row + g0off), b = lds_v2(row + g1off);
      __syncwarp();  // every lane read the slot before it is refilled
      issue(j + kCopyStages);
      const int64_t left = (int64_t)it.nelems - (int64_t)r * kRowElems;
      if (lane < 30 && 8 * lane < left)
        st_v4(P.out[it.dst] + it.out_off + (uint64_t)r * kRowElems + 8 * lane,
              make_uint4(a.x, a.y, b.x, b.y));
    }
    cp_async_wait<0>();
    __syncwarp();
  }
  finish_run(P, e);
}

__global__ void __launch_bounds__(kThreads, 4) k_stage_ll128(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int li = lane >> 3, k = lane & 7;
  const int lo = P.stage_rank < 0 ? 0 : P.stage_rank;
  const int hi = P.stage_rank < 0 ? P.nranks : P.stage_rank + 1;
  const uint32_t wbase =
      (uint32_t)__cvta_generic_to_shared(smem) + (uint32_t)(warp * kCopyStages * kRowBytes);
  const int G = 15 * li + 2 * k;  // first payload granule of this lane's line chunk
  for (int v = P.sbeg[lo] + blockIdx.x; v < P.sbeg[hi]; v += gridDim.x) {
    const StageItem it = P.sitems[v];
    const uint16_t* in = P.in[it.rank] + it.in_elem;
    char* img = image_bytes(P, P.P, e, it.rank) + it.dst_line * kLL128LineBytes;
    const uint32_t nrows = (it.nlines + kLL128RowLines - 1) / kLL128RowLines;
    const int nj = (uint32_t)warp < nrows ? (int)((nrows - warp + nwarps - 1) / nwarps) : 0;
    auto issue = [&](int j) {
      if (j < nj) {
        const uint32_t r = warp + j * nwarps;
        const int64_t left = (int64_t)it.nelems - (int64_t)r * kRowElems;
        const bool valid = lane < 30 && 8 * lane < left;
        cp_async16(wbase + (j % kCopyStages) * kRowBytes + 16 * lane,
                   in + (size_t)r * kRowElems + (valid ? 8 * lane : 0), valid);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kCopyStages; ++j) issue(j);
    for (int j = 0; j < nj; ++j) {
      cp_async_wait<kCopyStages - 1>();
      __syncwarp();
      const uint32_t row = wbase + (j % kCopyStages) * kRowBytes;
      // lanes 30, 31 hold no input: their slot bytes [480, 512) stay unread
      const uint2 a = lds_v2(row + 8 * G);
      const uint2 b = k == 7 ? make_uint2(0, 0) : lds_v2(row + 8 * (G + 1));
      __syncwarp();
      issue(j + kCopyStages);
      const uint32_t r = warp + j * nwarps;
      const int nl = min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines));
      ll128_store_row<false>(img + (size_t)r * kRowBytes, make_uint4(a.x, a.y, b.x, b.y), lane,
                             nl, e);
    }
    cp_async_wait<0>();
    __syncwarp();
  }
}

// ---- LL8 fold and copy through cp.async rings ------------------------------------
// The same pipelines for 8-byte lines: a warp row is 512 bytes = 64 lines =
// 128 elements; lane L holds lines 2L and 2L+1 (elements 4L..4L+3).  Used on
// the stream-ordered path when re-arming is deferred or off (the last-reader
// re-arm needs the generic kernel's counters).

__device__ __forceinline__ bool ll8_pair_ready(const uint4& v, uint32_t flag) {
  return v.y == flag && v.w == flag;
}

constexpr int kLL8RowLines = 64;

__global__ void __launch_bounds__(kThreads, 2) k_fold_ll8(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const uint32_t flag = (uint32_t)e;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int n = P.nranks;
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(smem) +
                         (uint32_t)(warp * kFoldStages * n * kRowBytes + 16 * lane);
  const bool deferred = P.reset_mode == kResetDeferred;
  const int n_items = P.beg1[P.nranks];
  for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
    if (aborted(P.ws)) break;
    const int i = P.interleave1 ? P.beg1[v % P.nranks] + v / P.nranks : v;
    const Item it = P.items1[i];
    const bool publish = (it.flags & IF_PUBLISH) != 0;
    const uint32_t nrows = (it.nlines + kLL8RowLines - 1) / kLL8RowLines;
    const int nj = (uint32_t)warp < nrows ? (int)((nrows - warp + nwarps - 1) / nwarps) : 0;
    auto issue = [&](int j) {
      if (j < nj) {
        const uint32_t r = warp + j * nwarps;
        const bool valid = r * kLL8RowLines + 2 * lane < it.nlines;
        const uint64_t off = (it.src_line + (uint64_t)r * kLL8RowLines) * kLL8LineBytes + 16 * lane;
        const uint32_t slot = wbase + (uint32_t)((j % kFoldStages) * n * kRowBytes);
        for (int p = 0; p < n; ++p)
          cp_async16(slot + p * kRowBytes, P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes +
                                               (uint64_t)p * P.P.rank_bytes + off,
                     valid);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kFoldStages; ++j) issue(j);
    bool ok = true;
    for (int j = 0; j < nj; ++j) {
      cp_async_wait<kFoldStages - 1>();
      const uint32_t slot = wbase + (uint32_t)((j % kFoldStages) * n * kRowBytes);
      uint4 s[kMaxRanks];
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p)
        if (p < n) s[p] = lds_v4(slot + p * kRowBytes);
      issue(j + kFoldStages);
      const uint32_t r = warp + j * nwarps;
      const uint64_t line = it.src_line + (uint64_t)r * kLL8RowLines + 2 * lane;
      const bool valid = r * kLL8RowLines + 2 * lane < it.nlines;
      if (valid) {
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p) {
          if (p < n && ok && !ll8_pair_ready(s[p], flag)) {
            const uint64_t* g = reinterpret_cast<const uint64_t*>(
                                    P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes +
                                    (uint64_t)p * P.P.rank_bytes) + line;
            ok = ll8_wait_lines(P, g, 2, flag, p, (int64_t)line);
            uint64_t a, b;
            ld_relaxed_v2u64(g, a, b);
            s[p] = make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
          }
        }
        uint64_t lo[kMaxRanks], hi[kMaxRanks];
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p) {
          lo[p] = s[p].x;   // payload words of the two lines
          hi[p] = s[p].z;
        }
        uint32_t w0, w1;
        ll8_fold_pair(lo, hi, n, P.dtype, w0, w1);
        if (publish) {
          uint64_t* dst = reinterpret_cast<uint64_t*>(P.ws + P.AG.base + (e & P.AG.slot_mask) * P.AG.slot_bytes +
                                                      (uint64_t)it.dst * P.AG.rank_bytes) +
                          it.out_off + (uint64_t)r * kLL8RowLines + 2 * lane;
          const uint64_t f = (uint64_t)flag << 32;
          st_relaxed_v2u64(dst, (uint64_t)w0 | f, (uint64_t)w1 | f);
          if (deferred) {
            uint64_t* other = reinterpret_cast<uint64_t*>(
                                  P.ws + P.AG.base + ((e + 1) & P.AG.slot_mask) * P.AG.slot_bytes +
                                  (uint64_t)it.dst * P.AG.rank_bytes) +
                              it.out_off + (uint64_t)r * kLL8RowLines + 2 * lane;
            st_relaxed_v2u64(other, 0ull, 0ull);
          }
        } else {
          st_v2u32(P.out[it.dst] + it.out_off + (uint64_t)r * 2 * kLL8RowLines + 4 * lane, w0, w1);
        }
      }
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
    }
    cp_async_wait<0>();
    if (!ok) break;
  }
  finish_run(P, e);
}

__global__ void __launch_bounds__(kThreads, 4) k_copy_ll8(RunParams P, int phase) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const uint32_t flag = (uint32_t)e;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const Item* items = phase == 1 ? P.items1 : P.items2;
  const int* beg = phase == 1 ? P.beg1 : P.beg2;
  const bool inter = phase == 1 ? P.interleave1 : P.interleave2;
  const Region& R = phase == 1 ? P.P : P.AG;
  const int n_items = beg[P.nranks];
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(smem) +
                         (uint32_t)(warp * kCopyStages * kRowBytes + 16 * lane);
  for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
    if (aborted(P.ws)) break;
    const int i = inter ? beg[v % P.nranks] + v / P.nranks : v;
    const Item it = items[i];
    const uint64_t* src = reinterpret_cast<const uint64_t*>(
                              P.ws + R.base + (e & R.slot_mask) * R.slot_bytes +
                              (uint64_t)it.src * R.rank_bytes) +
                          it.src_line;
    const uint32_t nrows = (it.nlines + kLL8RowLines - 1) / kLL8RowLines;
    const int nj = (uint32_t)warp < nrows ? (int)((nrows - warp + nwarps - 1) / nwarps) : 0;
    auto issue = [&](int j) {
      if (j < nj) {
        const uint32_t r = warp + j * nwarps;
        cp_async16(wbase + (j % kCopyStages) * kRowBytes, src + (size_t)r * kLL8RowLines + 2 * lane,
                   r * kLL8RowLines + 2 * lane < it.nlines);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kCopyStages; ++j) issue(j);
    bool ok = true;
    for (int j = 0; j < nj; ++j) {
      cp_async_wait<kCopyStages - 1>();
      uint4 s = lds_v4(wbase + (j % kCopyStages) * kRowBytes);
      issue(j + kCopyStages);
      const uint32_t r = warp + j * nwarps;
      if (r * kLL8RowLines + 2 * lane < it.nlines) {
        if (!ll8_pair_ready(s, flag)) {
          const uint64_t* g = src + (size_t)r * kLL8RowLines + 2 * lane;
          ok = ll8_wait_lines(P, g, 2, flag, it.src,
                              (int64_t)(it.src_line + r * kLL8RowLines + 2 * lane));
          uint64_t a, b;
          ld_relaxed_v2u64(g, a, b);
          s = make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
        }
        st_v2u32(P.out[it.dst] + it.out_off + (uint64_t)r * 2 * kLL8RowLines + 4 * lane, s.x, s.z);
      }
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
    }
    cp_async_wait<0>();
    if (!ok) break;
  }
  finish_run(P, e);
}

// Fold of sentinel packs (deferred re-arm: the fold re-arms only the other
// slot of what it publishes).  The ring of k_fold_ll8: each lane takes a
// pair of packs (8 elements) of every rank's image per warp row of 64 packs;
// a pair that still holds the all-ones pattern is polled (bounded) and
// reloaded; sent_fold8 folds them in rank order.
__global__ void __launch_bounds__(kThreads, 2) k_fold_sent(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int n = P.nranks;
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(smem) +
                         (uint32_t)(warp * kFoldStages * n * kRowBytes + 16 * lane);
  const int n_items = P.beg1[P.nranks];
  const char* img = P.ws + P.P.base + (e & P.P.slot_mask) * P.P.slot_bytes;
  for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
    if (aborted(P.ws)) break;
    const int i = P.interleave1 ? P.beg1[v % P.nranks] + v / P.nranks : v;
    const Item it = P.items1[i];
    const bool publish = (it.flags & IF_PUBLISH) != 0;
    const uint32_t ngroups = it.nlines / kSentGroupLines;
    const uint32_t nrows = (ngroups + 31) / 32;
    const int nj = (uint32_t)warp < nrows ? (int)((nrows - warp + nwarps - 1) / nwarps) : 0;
    auto issue = [&](int j) {
      if (j < nj) {
        const uint32_t g = (warp + j * nwarps) * 32 + lane;
        const uint64_t off = (it.src_line + 2 * (uint64_t)g) * kSentLineBytes;
        const uint32_t slot = wbase + (uint32_t)((j % kFoldStages) * n * kRowBytes);
        for (int p = 0; p < n; ++p)
          cp_async16(slot + p * kRowBytes, img + (uint64_t)p * P.P.rank_bytes + off, g < ngroups);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kFoldStages; ++j) issue(j);
    bool ok = true;
    for (int j = 0; j < nj; ++j) {
      cp_async_wait<kFoldStages - 1>();
      const uint32_t slot = wbase + (uint32_t)((j % kFoldStages) * n * kRowBytes);
      uint64_t lo[kMaxRanks], hi[kMaxRanks];
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p)
        if (p < n) {
          const uint4 w = lds_v4(slot + p * kRowBytes);
          lo[p] = (uint64_t)w.x | ((uint64_t)w.y << 32);
          hi[p] = (uint64_t)w.z | ((uint64_t)w.w << 32);
        }
      issue(j + kFoldStages);
      const uint32_t g = (warp + j * nwarps) * 32 + lane;
      const uint64_t line = it.src_line + 2 * (uint64_t)g;
      if (g < ngroups) {
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p)
          if (p < n && ok && (lo[p] == kSentPack || hi[p] == kSentPack)) {
            const uint64_t* q =
                reinterpret_cast<const uint64_t*>(img + (uint64_t)p * P.P.rank_bytes) + line;
            ok = sent_wait_pair(P, q, p, (int64_t)line);
            ld_relaxed_v2u64(q, lo[p], hi[p]);
          }
        if (ok) {
          const uint4 res = sent_fold8(lo, hi, n, P.dtype);
          if (publish) {
            uint64_t* dst = reinterpret_cast<uint64_t*>(P.ws + P.AG.base +
                                                        (e & P.AG.slot_mask) * P.AG.slot_bytes +
                                                        (uint64_t)it.dst * P.AG.rank_bytes) +
                            it.out_off + 2 * (uint64_t)g;
            st_relaxed_v2u64(dst, (uint64_t)res.x | ((uint64_t)res.y << 32),
                             (uint64_t)res.z | ((uint64_t)res.w << 32));
            uint64_t* other = reinterpret_cast<uint64_t*>(
                                  P.ws + P.AG.base + ((e + 1) & P.AG.slot_mask) * P.AG.slot_bytes +
                                  (uint64_t)it.dst * P.AG.rank_bytes) +
                              it.out_off + 2 * (uint64_t)g;
            sent_rearm(other);
          } else {
            st_v4(P.out[it.dst] + it.out_off + 8 * (uint64_t)g, res);
          }
        }
      }
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
    }
    cp_async_wait<0>();
    if (!ok) break;
  }
  finish_run(P, e);
}

// Validated copy of sentinel packs (deferred re-arm: a copy item re-arms
// nothing).  The ring of k_copy_ll8: each warp row is 32 groups of two packs
// (512 bytes), a lane's group arrives through a cp.async stage; a group that
// still holds the all-ones pattern is polled (bounded) and reloaded, and the
// 8 elements are stored as they are.
__global__ void __launch_bounds__(kThreads, 4) k_copy_sent(RunParams P, int phase) {
  extern __shared__ __align__(128) char smem[];
  const uint64_t e = begin_run(P);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const Item* items = phase == 1 ? P.items1 : P.items2;
  const int* beg = phase == 1 ? P.beg1 : P.beg2;
  const bool inter = phase == 1 ? P.interleave1 : P.interleave2;
  const Region& R = phase == 1 ? P.P : P.AG;
  const int n_items = beg[P.nranks];
  const uint32_t wbase = (uint32_t)__cvta_generic_to_shared(smem) +
                         (uint32_t)(warp * kCopyStages * kRowBytes + 16 * lane);
  for (int v = blockIdx.x; v < n_items; v += gridDim.x) {
    if (aborted(P.ws)) break;
    const int i = inter ? beg[v % P.nranks] + v / P.nranks : v;
    const Item it = items[i];
    const uint64_t* src = reinterpret_cast<const uint64_t*>(
                              P.ws + R.base + (e & R.slot_mask) * R.slot_bytes +
                              (uint64_t)it.src * R.rank_bytes) +
                          it.src_line;
    const uint32_t ngroups = it.nlines / kSentGroupLines;
    const uint32_t nrows = (ngroups + 31) / 32;
    const int nj = (uint32_t)warp < nrows ? (int)((nrows - warp + nwarps - 1) / nwarps) : 0;
    auto issue = [&](int j) {
      if (j < nj) {
        const uint32_t g = (warp + j * nwarps) * 32 + lane;
        cp_async16(wbase + (j % kCopyStages) * kRowBytes, src + 2 * (size_t)g, g < ngroups);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int j = 0; j < kCopyStages; ++j) issue(j);
    bool ok = true;
    for (int j = 0; j < nj; ++j) {
      cp_async_wait<kCopyStages - 1>();
      uint4 s = lds_v4(wbase + (j % kCopyStages) * kRowBytes);
      issue(j + kCopyStages);
      const uint32_t g = (warp + j * nwarps) * 32 + lane;
      if (g < ngroups) {
        const uint64_t a = (uint64_t)s.x | ((uint64_t)s.y << 32);
        const uint64_t b = (uint64_t)s.z | ((uint64_t)s.w << 32);
        if (a == kSentPack || b == kSentPack) {
          const uint64_t* q = src + 2 * (size_t)g;
          ok = sent_wait_pair(P, q, it.src, (int64_t)(it.src_line + 2 * (uint64_t)g));
          uint64_t a2, b2;
          ld_relaxed_v2u64(q, a2, b2);
          s = make_uint4((uint32_t)a2, (uint32_t)(a2 >> 32), (uint32_t)b2, (uint32_t)(b2 >> 32));
        }
        if (ok) st_v4(P.out[it.dst] + it.out_off + 8 * (uint64_t)g, s);
      }
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
    }
    cp_async_wait<0>();
    if (!ok) break;
  }
  finish_run(P, e);
}

// Late producer: publish rank p's withheld lines in the given order, after
// every consumer CTA has started polling.  One warp publishes, in order.
template <int ENC>
__device__ void late_producer(const RunParams& P, uint64_t e, int p, int workers) {
  WsHeader* h = header(P.ws);
  __shared__ int go;
  if (threadIdx.x == 0) {
    Waiter w;
    go = 1;
    while (ld_relaxed_u32(&h->started[e & 1]) < (uint32_t)workers) {
      if (w.expired(P.ws, P.timeout_ns)) {
        latch_error(P.ws, kStatusTimeout, p, -1);
        go = 0;
        break;
      }
      __nanosleep(200);
    }
  }
  __syncthreads();
  if (!go || threadIdx.x >= 32) return;
  __nanosleep(2000);  // consumers are polling the stale lines by now
  const int lane = threadIdx.x;
  const int64_t n = P.late_n[p];
  const int64_t* order = P.late_order[p];
  const uint16_t* in = P.in[p];
  auto locate = [&](int64_t line, uint64_t& elem0, int64_t& elems) {
    // segment containing `line` (segments are in image order)
    int k = 0;
    while (k + 1 < P.nseg && (uint64_t)line >= P.seg_line0[k + 1]) ++k;
    const int epl = ENC == ENC_LL8 ? kLL8Elems : (ENC == ENC_SENT ? kSentElems : kLL128Elems);
    const uint64_t off = ((uint64_t)line - P.seg_line0[k]) * epl;
    elem0 = P.seg_in0[k] + off;
    elems = (int64_t)P.seg_elems[k] - (int64_t)off;  // elements left in segment
  };
  if (ENC == ENC_SENT) {
    uint64_t* img = image_lines(P, P.P, e, p);
    for (int64_t j = 0; j < n; j += 32) {
      if (j + lane < n) {
        const int64_t line = order[j + lane];
        uint64_t elem0;
        int64_t left;
        locate(line, elem0, left);
        const uint2 d = *reinterpret_cast<const uint2*>(in + elem0);
        st_relaxed_u64(img + line, (uint64_t)sent_word(d.x, P.dtype) |
                                       ((uint64_t)sent_word(d.y, P.dtype) << 32));
      }
      __syncwarp();
      __nanosleep(500);
    }
  } else if (ENC == ENC_LL8) {
    uint64_t* img = image_lines(P, P.P, e, p);
    for (int64_t j = 0; j < n; j += 32) {
      if (j + lane < n) {
        const int64_t line = order[j + lane];
        uint64_t elem0;
        int64_t left;
        locate(line, elem0, left);
        const uint32_t data = *reinterpret_cast<const uint32_t*>(in + elem0);
        st_relaxed_u64(img + line, (uint64_t)data | ((uint64_t)(uint32_t)e << 32));
      }
      __syncwarp();
      __nanosleep(500);
    }
  } else {
    char* img = image_bytes(P, P.P, e, p);
    const int i = lane >> 3, k = lane & 7;
    for (int64_t j = 0; j < n; j += 4) {
      const bool valid = j + i < n;
      char* dst = nullptr;
      if (valid) {
        const int64_t line = order[j + i];
        uint64_t elem0;
        int64_t left;
        locate(line, elem0, left);
        dst = img + (uint64_t)line * kLL128LineBytes + 16 * k;
        // this lane's 8 (k < 7) or 4 (k = 7) elements; zero past the segment
        uint16_t v[8];
        for (int q = 0; q < 8; ++q) {
          const int64_t idx = 8 * k + q;
          v[q] = (q < (k == 7 ? 4 : 8) && idx < left) ? in[elem0 + idx] : 0;
        }
        const uint64_t lo = (uint64_t)v[0] | ((uint64_t)v[1] << 16) |
                            ((uint64_t)v[2] << 32) | ((uint64_t)v[3] << 48);
        const uint64_t hi = (uint64_t)v[4] | ((uint64_t)v[5] << 16) |
                            ((uint64_t)v[6] << 32) | ((uint64_t)v[7] << 48);
        if (k == 7)
          st_relaxed_u64(dst, lo);
        else
          st_relaxed_v2u64(dst, lo, hi);
      }
      __syncwarp();
      if (valid && k == 7) {
        fence_acq_rel_gpu();
        st_relaxed_u64(dst + 8, e);
      }
      __syncwarp();
      __nanosleep(500);
    }
  }
}

// A run in one launch is a chain of dependent global-memory round trips, so
// the prologue overlaps the ones that do not depend on each other: this
// CTA's first stage and consume items are read before the wait for the
// previous kernel (the plan's items are written when the workspace is bound
// and never change), and the first input load of the stage is issued while
// the epoch is in flight.  The grid's last CTA reads the arrival count
// before its consume phase, so the end of the run need not wait on it.
template <int ENC>
__global__ void __launch_bounds__(kThreads, 2) k_fused(RunParams P) {
  const int B = P.ctas_per_rank;
  const int workers = P.nranks * B;
  const bool worker = (int)blockIdx.x < workers;
  const int d = worker ? (int)blockIdx.x / B : 0, b = worker ? (int)blockIdx.x % B : 0;
  const int s0 = P.sbeg[d] + b, i0 = P.beg1[d] + b;
  const bool has_s = worker && P.sitems != nullptr && s0 < P.sbeg[d + 1];
  const bool has_i = worker && i0 < P.beg1[d + 1];
  __shared__ uint64_t s_epoch;
  StageItem si{};
  Item it1{};
  if (has_s) si = P.sitems[s0];
  if (has_i) it1 = P.items1[i0];
  // The epoch is read once per CTA (thread 0) and handed over in shared
  // memory: a read by every warp of every CTA at once is a hot spot on one
  // L2 line.  The first input load is in flight meanwhile.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) s_epoch = ld_relaxed_u64(&header(P.ws)->epoch);
  uint2 first8 = make_uint2(0, 0);
  uint4 firsts = make_uint4(0, 0, 0, 0);
  if (has_s) {
    if (ENC == ENC_LL8) first8 = ll8_stage_first(P, si);
    if (ENC == ENC_SENT) firsts = sent_stage_first(P, si);
  }
  __syncthreads();
  const uint64_t e = s_epoch;
  run_arrive(P, e);
  if (!worker) {
    late_producer<ENC>(P, e, ((int)blockIdx.x - workers) % P.nranks, workers);
    finish_run(P, e);
    return;
  }
  if (has_s) {
    if (ENC == ENC_LL8)
      ll8_stage_tile(P, si, e, true, first8);
    else if (ENC == ENC_SENT)
      sent_stage_tile(P, si, e, true, firsts);
    else
      stage_item<ENC, true>(P, si, e);
    for (int i = s0 + B; i < P.sbeg[d + 1]; i += B) stage_item<ENC, true>(P, P.sitems[i], e);
  }
  if (threadIdx.x == 0) atomicAdd(&header(P.ws)->started[e & 1], 1u);
  const uint32_t seen = early_arrivals(P);
  // The first item is consumed without reading the abort word first: that
  // read, made by every thread of every CTA at once, sat on the critical
  // path of a small run, and a wait inside the item still gives up once an
  // error is latched.  Later items check it as before.
  if (has_i) {
    consume_item<ENC, true>(P, P.P, it1, e);
    for (int i = i0 + B; i < P.beg1[d + 1]; i += B) {
      if (aborted(P.ws)) break;
      consume_item<ENC, true>(P, P.P, P.items1[i], e);
    }
  }
  if (P.items2 != nullptr)
    for (int i = P.beg2[d] + b; i < P.beg2[d + 1]; i += B) {
      if (aborted(P.ws)) break;
      consume_item<ENC, true>(P, P.AG, P.items2[i], e);
    }
  finish_run(P, e, seen);
}

// Overwrite the listed lines of rank `stage_rank`'s image with stale
// content: readiness value e-1 / e-2 / 0 (by kind) and a poison payload.
template <int ENC>
__global__ void k_withhold(RunParams P) {
  const uint64_t e = begin_run(P);
  const int p = P.stage_rank;
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < P.wh_n;
       j += (int64_t)gridDim.x * blockDim.x) {
    const int64_t line = P.wh_lines[j];
    const int kind = P.wh_kind[j];
    const uint64_t stale = kind == 0 ? e - 1 : (kind == 1 ? e - 2 : 0);
    const uint64_t pz = P.wh_poison[j];
    const uint64_t pw = pz | (pz << 16) | (pz << 32) | (pz << 48);
    if (ENC == ENC_SENT) {
      // a pack that was never published still holds the pattern
      st_relaxed_u64(image_lines(P, P.P, e, p) + line, kSentPack);
    } else if (ENC == ENC_LL8) {
      uint64_t* img = image_lines(P, P.P, e, p);
      st_relaxed_u64(img + line, (pw & 0xFFFFFFFFull) | ((uint64_t)(uint32_t)stale << 32));
    } else {
      char* l = image_bytes(P, P.P, e, p) + (uint64_t)line * kLL128LineBytes;
      for (int q = 0; q < 15; ++q) st_relaxed_u64(l + 8 * q, pw);
      st_relaxed_u64(l + 120, stale);
    }
  }
}

// Re-arm every LL8 line (flag 0) or sentinel pack (the pattern) of the
// current slot (both regions), then end the run.
__global__ void __launch_bounds__(kThreads) k_rearm(RunParams P) {
  const uint64_t e = begin_run(P);
  const uint64_t fill = P.enc == ENC_SENT ? kSentPack : 0ull;
  for (int region = 0; region < 2; ++region) {
    const Region& R = region == 0 ? P.P : P.AG;
    if (R.rank_bytes == 0) continue;
    const uint64_t words = (uint64_t)P.nranks * R.rank_bytes / 16;
    uint4* base = reinterpret_cast<uint4*>(P.ws + R.base + (e & R.slot_mask) * R.slot_bytes);
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < words;
         i += (uint64_t)gridDim.x * blockDim.x)
      st_relaxed_v2u64(base + i, fill, fill);
  }
  finish_run(P, e);
}

__global__ void k_advance(RunParams P) { finish_run(P, begin_run(P)); }

// ---- launchers ---------------------------------------------------------------

int current_device() {
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess ? dev : 0;
}

static int g_num_sms[kMaxDevices];

int device_sms() {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
  }
  if (g_num_sms[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    g_num_sms[dev] = n > 0 ? n : 1;
  }
  return g_num_sms[dev];
}

int fused_capacity(int enc) {
  int per_sm = 0;
  cudaError_t err =
      enc == ENC_LL8    ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                              &per_sm, k_fused<ENC_LL8>, kThreads, 0)
      : enc == ENC_SENT ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                              &per_sm, k_fused<ENC_SENT>, kThreads, 0)
                        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                              &per_sm, k_fused<ENC_LL128>, kThreads, 0);
  if (err != cudaSuccess || per_sm <= 0) return 0;
  return per_sm * device_sms();
}

int block_threads() { return kThreads; }

// A launch of kThreads-thread CTAs; dependent: with programmatic stream
// serialization (every kernel launched this way calls begin_run, which waits
// for the previous kernel in the stream, before it touches any data).
template <typename... KArgs, typename... Args>
static cudaError_t launch_k(void (*kernel)(KArgs...), int grid, size_t smem, cudaStream_t s,
                            bool dependent, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_stage(const RunParams& P, int grid, cudaStream_t s, bool dependent) {
  if (grid <= 0) return cudaSuccess;
  if (P.enc == ENC_LL8) return launch_k(k_stage<ENC_LL8>, grid, 0, s, dependent, P);
  if (P.enc == ENC_SENT) return launch_k(k_stage<ENC_SENT>, grid, 0, s, dependent, P);
  return launch_k(k_stage<ENC_LL128>, grid, 0, s, dependent, P);
}

cudaError_t launch_consume(const RunParams& P, int phase, int grid, cudaStream_t s,
                           bool dependent) {
  if (grid <= 0) grid = 1;
  if (P.enc == ENC_LL8) return launch_k(k_consume<ENC_LL8>, grid, 0, s, dependent, P, phase);
  if (P.enc == ENC_SENT) return launch_k(k_consume<ENC_SENT>, grid, 0, s, dependent, P, phase);
  return launch_k(k_consume<ENC_LL128>, grid, 0, s, dependent, P, phase);
}

cudaError_t launch_fused(const RunParams& P, int grid, cudaStream_t s, bool dependent) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 2 : 1;
  if (P.enc == ENC_LL8) return cudaLaunchKernelEx(&cfg, k_fused<ENC_LL8>, P);
  if (P.enc == ENC_SENT) return cudaLaunchKernelEx(&cfg, k_fused<ENC_SENT>, P);
  return cudaLaunchKernelEx(&cfg, k_fused<ENC_LL128>, P);
}

// The fixed cost of a one-launch run with no work in it: the CTAs do nothing
// but the dependent-launch handshake every run's prologue makes (wait for the
// previous kernel in the stream, then let the next dependent launch be
// placed).  No memory is touched.
__global__ void __launch_bounds__(kThreads) k_floor() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

cudaError_t launch_floor(int grid, cudaStream_t s, bool dependent, bool cooperative,
                         int threads) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads > 0 ? threads : kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = cooperative ? attr : attr + 1;
  cfg.numAttrs = (cooperative ? 1 : 0) + (dependent ? 1 : 0);
  return cudaLaunchKernelEx(&cfg, k_floor);
}

cudaError_t launch_fold(const RunParams& P, int grid, cudaStream_t s, bool dependent) {
  static size_t memo128[kMaxDevices], memo8[kMaxDevices], memo_sent[kMaxDevices];
  const size_t bytes = fold_smem_bytes(P.nranks);
  if (cudaError_t e = P.enc == ENC_LL8    ? raise_smem_limit(k_fold_ll8, bytes, memo8)
                      : P.enc == ENC_SENT ? raise_smem_limit(k_fold_sent, bytes, memo_sent)
                                          : raise_smem_limit(k_fold_ll128, bytes, memo128))
    return e;
  if (P.enc == ENC_LL8) return launch_k(k_fold_ll8, grid, bytes, s, dependent, P);
  if (P.enc == ENC_SENT) return launch_k(k_fold_sent, grid, bytes, s, dependent, P);
  return launch_k(k_fold_ll128, grid, bytes, s, dependent, P);
}

cudaError_t launch_copy(const RunParams& P, int phase, int grid, cudaStream_t s, bool dependent) {
  if (P.enc == ENC_LL8)
    return launch_k(k_copy_ll8, grid, copy_smem_bytes(), s, dependent, P, phase);
  if (P.enc == ENC_SENT)
    return launch_k(k_copy_sent, grid, copy_smem_bytes(), s, dependent, P, phase);
  return launch_k(k_copy_ll128, grid, copy_smem_bytes(), s, dependent, P, phase);
}

cudaError_t launch_stage_pipe(const RunParams& P, int grid, cudaStream_t s, bool dependent) {
  if (grid <= 0) return cudaSuccess;
  return launch_k(k_stage_ll128, grid, copy_smem_bytes(), s, dependent, P);
}

cudaError_t launch_withhold(const RunParams& P, cudaStream_t s) {
  if (P.wh_n <= 0) return cudaSuccess;
  const int grid = (int)((P.wh_n + kThreads - 1) / kThreads);
  if (P.enc == ENC_LL8)
    k_withhold<ENC_LL8><<<grid, kThreads, 0, s>>>(P);
  else if (P.enc == ENC_SENT)
    k_withhold<ENC_SENT><<<grid, kThreads, 0, s>>>(P);
  else
    k_withhold<ENC_LL128><<<grid, kThreads, 0, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_rearm(const RunParams& P, int grid, cudaStream_t s) {
  k_rearm<<<grid, kThreads, 0, s>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_advance(const RunParams& P, cudaStream_t s) {
  k_advance<<<1, 32, 0, s>>>(P);
  return cudaGetLastError();
}

}  // namespace coll
