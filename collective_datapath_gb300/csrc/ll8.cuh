// ll8.cuh -- LL8 datapath: 8-byte lines of 4 data bytes (two bf16) and a
// 4-byte flag equal to the epoch's low 32 bits.  Staging moves line pairs
// (8 input bytes -> one 16-byte store); consumers read pairs or groups of four
// lines.
//
// The line is the notification: Purlin §3.2 "Specializing for latency"
// packs payload and flag in one packet written by a single store; flash-comm
// §4.3 carries two copies of the sequence number beside 8 payload bytes in a
// 16-byte unit, which is exactly two LL8 lines.  Because data and flag share
// one single-copy-atomic 8-byte element, a consumer that sees the right flag
// also sees the right data, with no fence on either side.
#pragma once

#include "dev_common.cuh"

namespace coll {

struct LL8Group {
  uint64_t l0, l1, l2, l3;
};

__device__ __forceinline__ void ll8_load(const uint64_t* p, LL8Group& g) {
  ld_relaxed_v2u64(p, g.l0, g.l1);
  ld_relaxed_v2u64(p + 2, g.l2, g.l3);
}

__device__ __forceinline__ bool ll8_ready(const LL8Group& g, uint32_t flag) {
  return (uint32_t)(g.l0 >> 32) == flag && (uint32_t)(g.l1 >> 32) == flag &&
         (uint32_t)(g.l2 >> 32) == flag && (uint32_t)(g.l3 >> 32) == flag;
}

__device__ __forceinline__ void ll8_store(uint64_t* p, uint4 v, uint32_t flag) {
  const uint64_t f = (uint64_t)flag << 32;
  st_relaxed_v2u64(p, (uint64_t)v.x | f, (uint64_t)v.y | f);
  st_relaxed_v2u64(p + 2, (uint64_t)v.z | f, (uint64_t)v.w | f);
}

__device__ __forceinline__ void ll8_rearm(uint64_t* p) {
  st_relaxed_v2u64(p, 0ull, 0ull);
  st_relaxed_v2u64(p + 2, 0ull, 0ull);
}

// Poll `lines` (2 or 4) consecutive lines until every one carries `flag`
// (bounded); the caller then reloads them.  Returns false on timeout or
// abort (the error is latched).
static __device__ __noinline__ bool ll8_wait_lines(const RunParams& P, const uint64_t* p,
                                                   int lines, uint32_t flag, uint32_t rank,
                                                   int64_t line) {
  count_rejection(P.ws);
  Waiter w;
  for (;;) {
    if (w.expired(P.ws, P.timeout_ns)) {
      latch_error(P.ws, kStatusTimeout, rank, line);
      return false;
    }
    __nanosleep(64);
    bool ready = true;
    for (int j = 0; j < lines; j += 2) {
      uint64_t a, b;
      ld_relaxed_v2u64(p + j, a, b);
      ready = ready && (uint32_t)(a >> 32) == flag && (uint32_t)(b >> 32) == flag;
    }
    if (ready) return true;
  }
}

__device__ __forceinline__ uint64_t* image_lines(const RunParams& P, const Region& R,
                                                 uint64_t epoch, int rank) {
  return reinterpret_cast<uint64_t*>(P.ws + R.base + (epoch & R.slot_mask) * R.slot_bytes +
                                     (uint64_t)rank * R.rank_bytes);
}

// Fold of the payload words of two lines of every source (lo[p], hi[p]):
// 4 bf16 or 2 fp32, rank order, fp32 accumulation.
__device__ __forceinline__ void ll8_fold_pair(const uint64_t* lo, const uint64_t* hi, int n,
                                              int dtype, uint32_t& w0, uint32_t& w1) {
  if (dtype == kDtF32) {
    uint32_t w[kMaxRanks * 2], r[2];
#pragma unroll
    for (int p = 0; p < kMaxRanks; ++p) {
      w[2 * p] = (uint32_t)lo[p];
      w[2 * p + 1] = (uint32_t)hi[p];
    }
    fold_f32_words<2>(w, n, r);
    w0 = r[0];
    w1 = r[1];
    return;
  }
  float a0 = bf16_lo_to_f32((uint32_t)lo[0]), a1 = bf16_hi_to_f32((uint32_t)lo[0]);
  float a2 = bf16_lo_to_f32((uint32_t)hi[0]), a3 = bf16_hi_to_f32((uint32_t)hi[0]);
#pragma unroll
  for (int p = 1; p < kMaxRanks; ++p) {
    if (p < n) {
      a0 = __fadd_rn(a0, bf16_lo_to_f32((uint32_t)lo[p]));
      a1 = __fadd_rn(a1, bf16_hi_to_f32((uint32_t)lo[p]));
      a2 = __fadd_rn(a2, bf16_lo_to_f32((uint32_t)hi[p]));
      a3 = __fadd_rn(a3, bf16_hi_to_f32((uint32_t)hi[p]));
    }
  }
  w0 = pack_bf16x2(a0, a1);
  w1 = pack_bf16x2(a2, a3);
}

// Groups a thread keeps in flight per step (stage and copy).
constexpr int kGroupsInFlight = 4;

// Encode one staging tile (nlines is a multiple of 4 for LL8).
// Staging moves line pairs: a lane loads 8 input bytes (four bf16) and
// stores the two lines they make as one 16-byte store, so a warp's store
// covers 512 contiguous bytes (16 fully written sectors).
constexpr int kPairsInFlight = 8;

// The first input pair this thread stages from a tile (pair threadIdx.x):
// a one-launch run loads it while the epoch is still in flight and hands it
// to ll8_stage_tile as `first` (with have_first).
__device__ __forceinline__ uint2 ll8_stage_first(const RunParams& P, const StageItem& it) {
  return threadIdx.x < it.nlines / 2
             ? ld_stream_v2(P.in[it.rank] + it.in_elem + 4 * (size_t)threadIdx.x)
             : make_uint2(0, 0);
}

__device__ __forceinline__ void ll8_stage_tile(const RunParams& P, const StageItem& it,
                                               uint64_t epoch, bool have_first = false,
                                               uint2 first = make_uint2(0, 0)) {
  const uint16_t* in = P.in[it.rank] + it.in_elem;
  uint64_t* img = image_lines(P, P.P, epoch, it.rank) + it.dst_line;
  // Deferred re-arm: the same lines of the other slot were consumed by the
  // previous run, which has completed.
  const bool deferred = P.reset_mode == kResetDeferred;
  uint64_t* other = image_lines(P, P.P, epoch + 1, it.rank) + it.dst_line;
  const uint64_t f = (uint64_t)(uint32_t)epoch << 32;
  const uint32_t npairs = it.nlines / 2;
  for (uint32_t q0 = threadIdx.x; q0 < npairs; q0 += blockDim.x * kPairsInFlight) {
    uint2 v[kPairsInFlight];
#pragma unroll
    for (int j = 0; j < kPairsInFlight; ++j) {
      const uint32_t q = q0 + j * blockDim.x;
      if (q < npairs) v[j] = (j == 0 && have_first) ? first : ld_stream_v2(in + 4 * (size_t)q);
    }
    have_first = false;  // it held the first batch's pair only
#pragma unroll
    for (int j = 0; j < kPairsInFlight; ++j) {
      const uint32_t q = q0 + j * blockDim.x;
      if (q < npairs) {
        st_relaxed_v2u64(img + 2 * (size_t)q, (uint64_t)v[j].x | f, (uint64_t)v[j].y | f);
        if (deferred) st_relaxed_v2u64(other + 2 * (size_t)q, 0ull, 0ull);
      }
    }
  }
}

// Process one consume item: validate + unpack (+ fold) + write (+ re-arm).
// `R` is the source region (P for phase 1, AG for twoshot phase 2).  A fold
// loads the group of all n images before it checks them; a copy loads
// kGroupsInFlight groups before it checks them.
__device__ __forceinline__ void ll8_consume_item(const RunParams& P, const Region& R,
                                                 const Item& it, uint64_t epoch) {
  const uint32_t flag = (uint32_t)epoch;
  const int n = P.nranks;
  const uint32_t ngroups = it.nlines / kLL8GroupLines;
  const bool reduce = it.kind == IK_REDUCE;
  const bool publish = (it.flags & IF_PUBLISH) != 0;
  const bool sole = (it.flags & IF_RESET_SOLE) != 0 && P.reset_mode == kResetLastReader;
  const bool deferred = P.reset_mode == kResetDeferred;
  bool ok = true;
  if (reduce) {
    // Pairs of lines (16 bytes, 4 elements) per source per step: the N
    // sources' pairs are loaded before any is checked.
    const uint32_t npairs = it.nlines / 2;
    for (uint32_t q = threadIdx.x; q < npairs && ok; q += blockDim.x) {
      const uint64_t line = it.src_line + 2 * (uint64_t)q;
      uint64_t lo[kMaxRanks], hi[kMaxRanks];
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p)
        if (p < n) ld_relaxed_v2u64(image_lines(P, R, epoch, p) + line, lo[p], hi[p]);
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p)
        if (p < n && ((uint32_t)(lo[p] >> 32) != flag || (uint32_t)(hi[p] >> 32) != flag)) {
          const uint64_t* src = image_lines(P, R, epoch, p) + line;
          ok = ok && ll8_wait_lines(P, src, 2, flag, p, (int64_t)line);
          ld_relaxed_v2u64(src, lo[p], hi[p]);
        }
      if (!ok) break;
      uint32_t w0, w1;
      ll8_fold_pair(lo, hi, n, P.dtype, w0, w1);
      if (sole) {
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p)
          if (p < n) st_relaxed_v2u64(image_lines(P, R, epoch, p) + line, 0ull, 0ull);
      }
      if (publish) {
        const uint64_t f = (uint64_t)flag << 32;
        st_relaxed_v2u64(image_lines(P, P.AG, epoch, it.dst) + it.out_off + 2 * (uint64_t)q,
                         (uint64_t)w0 | f, (uint64_t)w1 | f);
        if (deferred)
          st_relaxed_v2u64(image_lines(P, P.AG, epoch + 1, it.dst) + it.out_off + 2 * (uint64_t)q,
                           0ull, 0ull);
      } else {
        st_v2u32(P.out[it.dst] + it.out_off + 4 * (uint64_t)q, w0, w1);
      }
    }
  } else {
    uint64_t* src0 = image_lines(P, R, epoch, it.src) + it.src_line;
    for (uint32_t g0 = threadIdx.x; g0 < ngroups && ok; g0 += blockDim.x * kGroupsInFlight) {
      LL8Group s[kGroupsInFlight];
#pragma unroll
      for (int j = 0; j < kGroupsInFlight; ++j) {
        const uint32_t g = g0 + j * blockDim.x;
        if (g < ngroups) ll8_load(src0 + 4 * (size_t)g, s[j]);
      }
#pragma unroll
      for (int j = 0; j < kGroupsInFlight; ++j) {
        const uint32_t g = g0 + j * blockDim.x;
        if (g < ngroups && !ll8_ready(s[j], flag)) {
          ok = ok && ll8_wait_lines(P, src0 + 4 * (size_t)g, 4, flag, it.src,
                                    (int64_t)(it.src_line + 4 * (uint64_t)g));
          ll8_load(src0 + 4 * (size_t)g, s[j]);
        }
      }
      if (!ok) break;
#pragma unroll
      for (int j = 0; j < kGroupsInFlight; ++j) {
        const uint32_t g = g0 + j * blockDim.x;
        if (g >= ngroups) break;
        const uint4 res =
            make_uint4((uint32_t)s[j].l0, (uint32_t)s[j].l1, (uint32_t)s[j].l2, (uint32_t)s[j].l3);
        if (sole) ll8_rearm(src0 + 4 * (size_t)g);
        if (publish) {
          ll8_store(image_lines(P, P.AG, epoch, it.dst) + it.out_off + 4 * (uint64_t)g, res,
                    flag);
          if (deferred)
            ll8_rearm(image_lines(P, P.AG, epoch + 1, it.dst) + it.out_off + 4 * (uint64_t)g);
        } else {
          st_v4(P.out[it.dst] + it.out_off + 8 * (uint64_t)g, res);
        }
      }
    }
  }
  if ((it.flags & IF_RESET_COUNTED) && P.reset_mode == kResetLastReader) {
    // The last of `readers` items over these lines re-arms them.
    __shared__ uint32_t last;
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      uint32_t old = atomicAdd(&P.counters[it.counter], 1u);
      last = (old == (uint32_t)it.readers - 1u);
      if (last) {
        P.counters[it.counter] = 0u;
        __threadfence();
      }
    }
    __syncthreads();
    if (last) {
      for (uint32_t g = threadIdx.x; g < ngroups; g += blockDim.x) {
        const uint64_t line = it.src_line + 4 * (uint64_t)g;
        if (reduce) {
          for (int p = 0; p < n; ++p) ll8_rearm(image_lines(P, R, epoch, p) + line);
        } else {
          ll8_rearm(image_lines(P, R, epoch, it.src) + line);
        }
      }
    }
  }
}

}  // namespace coll
