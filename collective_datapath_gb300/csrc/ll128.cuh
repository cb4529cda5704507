// ll128.cuh -- LL128 datapath: 128-byte lines holding 120 bytes of data (60
// bf16) and the epoch as an 8-byte sequence number in bytes 120..127
// (flash-comm §3.1 "Sequence-number readiness": accept a unit only when its
// number is the current call's; no re-arm is needed).
//
// A warp moves one "row" of four lines (512 bytes of lines, 480 bytes of
// payload) per step: lane L holds bytes [16L, 16L+16) of the row, i.e. chunk
// k = L & 7 of line i = L >> 3; chunk 7 of a line holds its last 8 data bytes
// and the sequence number.  Payload is 16-byte aligned per row (480 = 30 x 16)
// but not per line (120 is 8 mod 16), so rows are re-aligned between the line
// view and the payload view with warp shuffles of 8-byte granules.
//
// Two publication protocols:
//  * stream-ordered (stage and consume are separate kernels on one stream):
//    the kernel boundary orders every staged byte before every consumer
//    load, so a line is written with one 16-byte store per lane and read the
//    same way; the consumer still checks every line's number and rejects a
//    line that was not staged for this epoch.
//  * concurrent (producer and consumer CTAs of one cooperative launch):
//    data stores, __syncwarp, fence.acq_rel.gpu, then the number (a release
//    pattern); the consumer reads the number, fence.acq_rel.gpu, __syncwarp,
//    then the data (an acquire pattern).  A 128-byte line is not single-copy
//    atomic, so this ordering -- not the line size -- is what makes it safe.
#pragma once

#include "dev_common.cuh"

namespace coll {

constexpr int kRowElems = kLL128RowLines * kLL128Elems;  // 240
constexpr int kRowBytes = kLL128RowLines * kLL128LineBytes;  // 512

__device__ __forceinline__ char* image_bytes(const RunParams& P, const Region& R,
                                             uint64_t epoch, int rank) {
  return P.ws + R.base + (epoch & R.slot_mask) * R.slot_bytes + (uint64_t)rank * R.rank_bytes;
}

__device__ __forceinline__ uint4 shfl4(uint4 v, int src) {
  uint4 r;
  r.x = __shfl_sync(0xFFFFFFFFu, v.x, src);
  r.y = __shfl_sync(0xFFFFFFFFu, v.y, src);
  r.z = __shfl_sync(0xFFFFFFFFu, v.z, src);
  r.w = __shfl_sync(0xFFFFFFFFu, v.w, src);
  return r;
}

// Payload chunks (lane q < 30 holds payload bytes [16q, 16q+16) of the row)
// -> line chunks (lane L holds its 16 bytes of the row's lines).  For lane
// chunk k = 7 only .x/.y are data; .z/.w are left for the sequence number.
__device__ __forceinline__ uint4 payload_to_lines(uint4 pay, int lane) {
  const int i = lane >> 3, k = lane & 7;
  const int G = 15 * i + 2 * k;             // first 8-byte payload granule
  const int A = G >> 1;
  const int B = (k == 7) ? A : ((G + 1) >> 1);
  uint4 a = shfl4(pay, A);
  uint4 b = shfl4(pay, B);
  uint4 r;
  if ((G & 1) == 0) {
    r = a;
  } else {
    r.x = a.z; r.y = a.w; r.z = b.x; r.w = b.y;
  }
  return r;
}

// Line chunks -> payload chunks (inverse of payload_to_lines).
__device__ __forceinline__ uint4 lines_to_payload(uint4 ln, int lane) {
  const int q = lane < 30 ? lane : 29;
  const int G0 = 2 * q, G1 = 2 * q + 1;
  const int i0 = G0 / 15, g0 = G0 % 15, i1 = G1 / 15, g1 = G1 % 15;
  const int A = 8 * i0 + (g0 >> 1), B = 8 * i1 + (g1 >> 1);
  uint4 a = shfl4(ln, A);
  uint4 b = shfl4(ln, B);
  uint4 r;
  r.x = (g0 & 1) ? a.z : a.x;
  r.y = (g0 & 1) ? a.w : a.y;
  r.z = (g1 & 1) ? b.z : b.x;
  r.w = (g1 & 1) ? b.w : b.y;
  return r;
}

// Write one row of lines.  `ln` = this lane's line chunk (data), the lane
// with k = 7 adds the sequence number.  Lanes of lines >= nl write nothing.
template <bool kConc>
__device__ __forceinline__ void ll128_store_row(char* row, uint4 ln, int lane, int nl,
                                                uint64_t seq) {
  const int i = lane >> 3, k = lane & 7;
  const bool valid = i < nl;
  char* p = row + 16 * lane;
  if (!kConc) {
    if (valid) {
      if (k == 7) {
        ln.z = (uint32_t)seq;
        ln.w = (uint32_t)(seq >> 32);
      }
      st_v4(p, ln);
    }
    return;
  }
  if (valid) {
    if (k == 7)
      st_relaxed_u64(p, (uint64_t)ln.x | ((uint64_t)ln.y << 32));
    else
      st_relaxed_v2u64(p, (uint64_t)ln.x | ((uint64_t)ln.y << 32),
                       (uint64_t)ln.z | ((uint64_t)ln.w << 32));
  }
  __syncwarp();
  if (valid && k == 7) {
    fence_acq_rel_gpu();
    st_relaxed_u64(p + 8, seq);
  }
}

// Bounded wait for the sequence number at `p` (a lane with k = 7).
static __device__ __noinline__ bool ll128_wait_seq(const RunParams& P, const char* p,
                                            uint64_t seq, uint32_t rank, int64_t line) {
  count_rejection(P.ws);
  Waiter w;
  for (;;) {
    if (w.expired(P.ws, P.timeout_ns)) {
      latch_error(P.ws, kStatusTimeout, rank, line);
      return false;
    }
    __nanosleep(64);
    if (ld_relaxed_u64(p) == seq) return true;
  }
}

// Rows a warp keeps in flight per step (copy and stage: one load per row).
constexpr int kRowsInFlight = 4;

// Stage one tile: rows of 240 input elements -> rows of four lines.  A warp
// loads kRowsInFlight rows of input before it re-aligns and stores them.
template <bool kConc>
__device__ __forceinline__ void ll128_stage_tile(const RunParams& P, const StageItem& it,
                                                 uint64_t epoch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint16_t* in = P.in[it.rank] + it.in_elem;
  char* img = image_bytes(P, P.P, epoch, it.rank) + it.dst_line * kLL128LineBytes;
  const uint32_t nrows = (it.nlines + kLL128RowLines - 1) / kLL128RowLines;
  for (uint32_t r0 = warp; r0 < nrows; r0 += nwarps * kRowsInFlight) {
    uint4 pay[kRowsInFlight];
#pragma unroll
    for (int j = 0; j < kRowsInFlight; ++j) {
      const uint32_t r = r0 + j * nwarps;
      const int64_t left = (int64_t)it.nelems - (int64_t)r * kRowElems;
      pay[j] = make_uint4(0, 0, 0, 0);
      if (r < nrows && lane < 30 && 8 * lane < left)
        pay[j] = ld_stream_v4(in + (size_t)r * kRowElems + 8 * lane);
    }
#pragma unroll
    for (int j = 0; j < kRowsInFlight; ++j) {
      const uint32_t r = r0 + j * nwarps;
      if (r >= nrows) break;
      uint4 ln = payload_to_lines(pay[j], lane);
      const int nl = min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines));
      ll128_store_row<kConc>(img + (size_t)r * kRowBytes, ln, lane, nl, epoch);
    }
  }
}

__device__ __forceinline__ bool ll128_chunk_ready(const uint4& v, int lane, bool valid,
                                                  uint64_t seq) {
  return !(valid && (lane & 7) == 7) || ((((uint64_t)v.w) << 32) | v.z) == seq;
}

// Stream-ordered slow path: a chunk loaded optimistically did not carry the
// epoch.  The lane waits (bounded) for the number and fences; the caller
// reloads the chunk when every lane of the warp succeeded.  Warp-collective.
static __device__ __noinline__ bool ll128_wait_chunk(const RunParams& P, const char* row, int lane,
                                              bool ready, uint64_t seq, uint32_t rank,
                                              int64_t row_line) {
  bool ok = true;
  if (!ready) {
    ok = ll128_wait_seq(P, row + 16 * lane + 8, seq, rank, row_line + (lane >> 3));
    fence_acq_rel_gpu();
  }
  __syncwarp();
  return __all_sync(0xFFFFFFFFu, ok);
}

// Concurrent path: the lanes holding sequence numbers read them for `cnt`
// rows first (relaxed), wait for the missing ones, then one acquire fence;
// after __syncwarp every lane may load the data of those rows.
template <int CNT>
__device__ __forceinline__ bool ll128_acquire_rows(const RunParams& P, const char* const* rows,
                                                   const int* nls, int cnt, int lane,
                                                   uint64_t seq, const uint32_t* ranks,
                                                   const int64_t* row_lines) {
  bool ok = true;
  if ((lane & 7) == 7) {
    uint64_t v[CNT];
#pragma unroll
    for (int j = 0; j < CNT; ++j)
      if (j < cnt && (lane >> 3) < nls[j]) v[j] = ld_relaxed_u64(rows[j] + 16 * lane + 8);
#pragma unroll
    for (int j = 0; j < CNT; ++j)
      if (j < cnt && (lane >> 3) < nls[j] && v[j] != seq)
        ok = ok && ll128_wait_seq(P, rows[j] + 16 * lane + 8, seq, ranks[j],
                                  row_lines[j] + (lane >> 3));
    fence_acq_rel_gpu();
  }
  __syncwarp();
  return __all_sync(0xFFFFFFFFu, ok);
}

__device__ __forceinline__ uint4 ld_relaxed_v4(const char* p) {
  uint64_t a, b;
  ld_relaxed_v2u64(p, a, b);
  return make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
}

// Fold the 8 (k < 7) or 4 (k = 7) bf16, or 4 (2) fp32, of this lane's chunk
// over n images.
__device__ __forceinline__ uint4 ll128_fold_f32(const uint4* s, int n) {
  uint32_t w[kMaxRanks * 4], r[4];
#pragma unroll
  for (int p = 0; p < kMaxRanks; ++p) {
    w[4 * p] = s[p].x;
    w[4 * p + 1] = s[p].y;
    w[4 * p + 2] = s[p].z;
    w[4 * p + 3] = s[p].w;
  }
  fold_f32_words<4>(w, n, r);
  return make_uint4(r[0], r[1], r[2], r[3]);
}

__device__ __forceinline__ uint4 ll128_fold(const uint4* s, int n, int dtype) {
  if (dtype == kDtF32) return ll128_fold_f32(s, n);
  float a[8];
  a[0] = bf16_lo_to_f32(s[0].x); a[1] = bf16_hi_to_f32(s[0].x);
  a[2] = bf16_lo_to_f32(s[0].y); a[3] = bf16_hi_to_f32(s[0].y);
  a[4] = bf16_lo_to_f32(s[0].z); a[5] = bf16_hi_to_f32(s[0].z);
  a[6] = bf16_lo_to_f32(s[0].w); a[7] = bf16_hi_to_f32(s[0].w);
#pragma unroll
  for (int p = 1; p < kMaxRanks; ++p) {
    if (p < n) {
      a[0] = __fadd_rn(a[0], bf16_lo_to_f32(s[p].x));
      a[1] = __fadd_rn(a[1], bf16_hi_to_f32(s[p].x));
      a[2] = __fadd_rn(a[2], bf16_lo_to_f32(s[p].y));
      a[3] = __fadd_rn(a[3], bf16_hi_to_f32(s[p].y));
      a[4] = __fadd_rn(a[4], bf16_lo_to_f32(s[p].z));
      a[5] = __fadd_rn(a[5], bf16_hi_to_f32(s[p].z));
      a[6] = __fadd_rn(a[6], bf16_lo_to_f32(s[p].w));
      a[7] = __fadd_rn(a[7], bf16_hi_to_f32(s[p].w));
    }
  }
  return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                    pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
}

// Two steps of the bf16 fold in fewer instructions (no change in any result
// bit):
//  * add.rn.f32.bf16 takes the bf16 operand as it is (its widening to
//    binary32 is exact) and rounds the sum once, so it equals widening first
//    and __fadd_rn -- an exhaustive run on GB300 over every bf16 operand
//    against 65,536 binary32 operands each found no difference;
//  * cvt.rn.bf16x2.f32 rounds two binary32 sums to nearest-even at once;
//    the same kind of run over all 2^32 binary32 patterns matched
//    f32_to_bf16_rne on every non-NaN input.  For a NaN it returns 0x7FFF,
//    so NaN sums (rare: a NaN input, or opposite infinities) are rewritten
//    to the canonical 0x7FC0 of the fold's rounding rule.
__device__ __forceinline__ void add_bf16x2_f32(uint32_t w, float& lo, float& hi) {
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; add.rn.f32.bf16 %0, l, %0; "
      "add.rn.f32.bf16 %1, h, %1; }"
      : "+f"(lo), "+f"(hi)
      : "r"(w));
}
__device__ __forceinline__ uint32_t cvt_rn_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The fold of ll128_fold, taken one rank at a time: first() with rank 0's
// chunk, then add() with each later rank's chunk in rank order, then
// result().  Only the running sums are live, not every rank's chunk, which
// keeps register pressure low in the kernels that read ranks one by one.
template <bool kF32>
struct ChunkFold {
  float a[8];
  __device__ __forceinline__ void first(const uint4& v) {
    if (kF32) {
      a[0] = __uint_as_float(v.x); a[1] = __uint_as_float(v.y);
      a[2] = __uint_as_float(v.z); a[3] = __uint_as_float(v.w);
    } else {
      a[0] = bf16_lo_to_f32(v.x); a[1] = bf16_hi_to_f32(v.x);
      a[2] = bf16_lo_to_f32(v.y); a[3] = bf16_hi_to_f32(v.y);
      a[4] = bf16_lo_to_f32(v.z); a[5] = bf16_hi_to_f32(v.z);
      a[6] = bf16_lo_to_f32(v.w); a[7] = bf16_hi_to_f32(v.w);
    }
  }
  __device__ __forceinline__ void add(const uint4& v) {
    if (kF32) {
      a[0] = __fadd_rn(a[0], __uint_as_float(v.x)); a[1] = __fadd_rn(a[1], __uint_as_float(v.y));
      a[2] = __fadd_rn(a[2], __uint_as_float(v.z)); a[3] = __fadd_rn(a[3], __uint_as_float(v.w));
    } else {
      add_bf16x2_f32(v.x, a[0], a[1]);
      add_bf16x2_f32(v.y, a[2], a[3]);
      add_bf16x2_f32(v.z, a[4], a[5]);
      add_bf16x2_f32(v.w, a[6], a[7]);
    }
  }
  __device__ __forceinline__ uint4 result() const {
    if (kF32) return make_uint4(f32_bits(a[0]), f32_bits(a[1]), f32_bits(a[2]), f32_bits(a[3]));
    uint32_t r[4];
    bool nan = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r[i] = cvt_rn_bf16x2(a[2 * i], a[2 * i + 1]);
      nan = nan || a[2 * i] != a[2 * i] || a[2 * i + 1] != a[2 * i + 1];
    }
    if (nan) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (a[2 * i] != a[2 * i]) r[i] = (r[i] & 0xFFFF0000u) | 0x7FC0u;
        if (a[2 * i + 1] != a[2 * i + 1]) r[i] = (r[i] & 0x0000FFFFu) | 0x7FC00000u;
      }
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
  }
};

// Write the row's payload (line view `ln`) to a plain output buffer.
__device__ __forceinline__ void ll128_write_payload(uint16_t* out_row, uint4 ln, int lane,
                                                    int64_t left) {
  uint4 pay = lines_to_payload(ln, lane);
  if (lane < 30 && 8 * lane < left) st_v4(out_row + 8 * lane, pay);
}

// Process one consume item (see ll8_consume_item); `R` = source region.
// Fold: a warp loads the row of all n images before it validates them.
// Copy: a warp loads kRowsInFlight rows before it validates them.
template <bool kConc>
__device__ __forceinline__ void ll128_consume_item(const RunParams& P, const Region& R,
                                                   const Item& it, uint64_t epoch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int n = P.nranks;
  const bool publish = (it.flags & IF_PUBLISH) != 0;
  const uint32_t nrows = (it.nlines + kLL128RowLines - 1) / kLL128RowLines;
  const int li = lane >> 3;
  if (it.kind == IK_REDUCE) {
    for (uint32_t r = warp; r < nrows; r += nwarps) {
      const int nl = min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines));
      const bool valid = li < nl;
      const uint64_t row_line = it.src_line + (uint64_t)r * kLL128RowLines;
      const uint64_t roff = row_line * kLL128LineBytes;
      uint4 s[kMaxRanks];
      if (!kConc) {
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p)
          if (p < n) s[p] = valid ? ld_v4(image_bytes(P, R, epoch, p) + roff + 16 * lane)
                                  : make_uint4(0, 0, 0, 0);
        bool ready = true;
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p)
          if (p < n) ready = ready && ll128_chunk_ready(s[p], lane, valid, epoch);
        if (!__all_sync(0xFFFFFFFFu, ready)) {
#pragma unroll
          for (int p = 0; p < kMaxRanks; ++p) {
            if (p < n) {
              const bool rp = ll128_chunk_ready(s[p], lane, valid, epoch);
              if (!__all_sync(0xFFFFFFFFu, rp)) {
                const char* row = image_bytes(P, R, epoch, p) + roff;
                if (!ll128_wait_chunk(P, row, lane, rp, epoch, p, (int64_t)row_line)) return;
                if (valid) s[p] = ld_v4(row + 16 * lane);
              }
            }
          }
        }
      } else {
        const char* rows[kMaxRanks];
        int nls[kMaxRanks];
        uint32_t ranks[kMaxRanks];
        int64_t rls[kMaxRanks];
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p) {
          rows[p] = image_bytes(P, R, epoch, p < n ? p : 0) + roff;
          nls[p] = nl;
          ranks[p] = p;
          rls[p] = (int64_t)row_line;
        }
        if (!ll128_acquire_rows<kMaxRanks>(P, rows, nls, n, lane, epoch, ranks, rls)) return;
#pragma unroll
        for (int p = 0; p < kMaxRanks; ++p)
          if (p < n) s[p] = valid ? ld_relaxed_v4(rows[p] + 16 * lane) : make_uint4(0, 0, 0, 0);
      }
      const uint4 res = ll128_fold(s, n, P.dtype);
      if (publish) {
        char* dst = image_bytes(P, P.AG, epoch, it.dst) +
                    (it.out_off + (uint64_t)r * kLL128RowLines) * kLL128LineBytes;
        ll128_store_row<kConc>(dst, res, lane, nl, epoch);
      } else {
        const int64_t left = (int64_t)it.nelems - (int64_t)r * kRowElems;
        ll128_write_payload(P.out[it.dst] + it.out_off + (uint64_t)r * kRowElems, res, lane,
                            left);
      }
    }
    return;
  }
  // copy
  const char* src = image_bytes(P, R, epoch, it.src) + it.src_line * kLL128LineBytes;
  for (uint32_t r0 = warp; r0 < nrows; r0 += nwarps * kRowsInFlight) {
    uint4 v[kRowsInFlight];
    int nls[kRowsInFlight];
    if (!kConc) {
#pragma unroll
      for (int j = 0; j < kRowsInFlight; ++j) {
        const uint32_t r = r0 + j * nwarps;
        nls[j] = r < nrows ? min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines)) : 0;
        v[j] = li < nls[j] ? ld_v4(src + (size_t)r * kRowBytes + 16 * lane)
                           : make_uint4(0, 0, 0, 0);
      }
      bool ready = true;
#pragma unroll
      for (int j = 0; j < kRowsInFlight; ++j)
        ready = ready && ll128_chunk_ready(v[j], lane, li < nls[j], epoch);
      if (!__all_sync(0xFFFFFFFFu, ready)) {
#pragma unroll
        for (int j = 0; j < kRowsInFlight; ++j) {
          const uint32_t r = r0 + j * nwarps;
          const bool rj = ll128_chunk_ready(v[j], lane, li < nls[j], epoch);
          if (!__all_sync(0xFFFFFFFFu, rj)) {
            const char* row = src + (size_t)r * kRowBytes;
            if (!ll128_wait_chunk(P, row, lane, rj, epoch, it.src,
                                  (int64_t)(it.src_line + r * kLL128RowLines)))
              return;
            if (li < nls[j]) v[j] = ld_v4(row + 16 * lane);
          }
        }
      }
    } else {
      const char* rows[kRowsInFlight];
      uint32_t ranks[kRowsInFlight];
      int64_t rls[kRowsInFlight];
#pragma unroll
      for (int j = 0; j < kRowsInFlight; ++j) {
        const uint32_t r = r0 + j * nwarps;
        nls[j] = r < nrows ? min((int)kLL128RowLines, (int)(it.nlines - r * kLL128RowLines)) : 0;
        rows[j] = src + (size_t)(r < nrows ? r : 0) * kRowBytes;
        ranks[j] = it.src;
        rls[j] = (int64_t)(it.src_line + (uint64_t)r * kLL128RowLines);
      }
      if (!ll128_acquire_rows<kRowsInFlight>(P, rows, nls, kRowsInFlight, lane, epoch, ranks,
                                             rls))
        return;
#pragma unroll
      for (int j = 0; j < kRowsInFlight; ++j)
        v[j] = li < nls[j] ? ld_relaxed_v4(rows[j] + 16 * lane) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < kRowsInFlight; ++j) {
      const uint32_t r = r0 + j * nwarps;
      if (r >= nrows) break;
      if (publish) {
        char* dst = image_bytes(P, P.AG, epoch, it.dst) +
                    (it.out_off + (uint64_t)r * kLL128RowLines) * kLL128LineBytes;
        ll128_store_row<kConc>(dst, v[j], lane, nls[j], epoch);
      } else {
        const int64_t left = (int64_t)it.nelems - (int64_t)r * kRowElems;
        ll128_write_payload(P.out[it.dst] + it.out_off + (uint64_t)r * kRowElems, v[j], lane,
                            left);
      }
    }
  }
}

}  // namespace coll
