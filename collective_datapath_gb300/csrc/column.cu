// column.cu -- the composed one-launch collectives scheduled by columns.
//
// Purlin §3.2 ("Extending the execution to AllReduce", Figure 5, Algorithm 1)
// runs a twoshot all-reduce's stage, reduce and gather work at chunk
// granularity, each role signalling chunk completion to the next one.  Here
// a column (c, x) is chunk c of partition x (all-reduce, reduce-scatter), of
// destination x (all-to-all) or of source x (all-gather), and one CTA runs
// all of it in three phases:
//   stage   every rank p moves its piece of the column (its partition-x or
//           destination-x rows; the all-gather's one piece of source x) into
//           its staging image as LL128 lines carrying the run's number;
//   fold    (all-reduce, reduce-scatter) owner x validates the N images' lines
//           of the column, folds them in rank order (fp32, one rounding) and
//           publishes the result as its own lines, or writes its output;
//   gather  (all-reduce, all-to-all, all-gather) every destination validates
//           the column's lines it reads and unpacks them into its output.
// A CTA barrier between phases orders the CTA's line stores before the next
// phase's loads (the chunk counters of Algorithm 1, inside one CTA); every
// line's number is still checked.  A staged or published line is read back
// a few microseconds after it was written, by the same SM, and dropped from
// L2 once read, so staging stays out of HBM, and CTAs never wait for each
// other.  Every CTA takes its first column by its own index and later ones
// from one counter, in chunk-major order.  Columns are of three lengths
// (column_at): each CTA's first column is one of a staggered group (1/G ..
// G/G of a chunk), so the CTAs do not all stage at once; then full chunks;
// and the last half round of the CTAs' work in short columns, so they run
// out of work together.  A short run uses 16-line columns only, one per CTA.
// The all-to-all (V) reads its pieces from an exchange table, so each
// source's piece of a column has its own length.
//
// Bounded staging (Purlin §4.1, P.cp.ring > 0 chunk slots per rank image):
// CTA g owns slot g of every rank image and slot g / N of one owner's
// published image, and serves columns g, g + G, ... (G a multiple of N, so
// always partition g mod N).  Lines of column q carry epoch + q, and the run
// advances the epoch by the column count rounded up to odd (§4.2).
//
// Inside a phase each warp takes a contiguous range of the phase's rows
// (rows of piece k are numbered k * R + r, R rows of 4 lines per piece) and
// walks it with two cursors:
// the load cursor runs a ring of kRing rows ahead of the store cursor, and
// a cursor reloads its piece's fields only when it crosses into the next
// piece.
#include <cuda_runtime.h>

#include <algorithm>

#include "launch.h"
#include "ll128.cuh"
#include "pipe.cuh"

namespace coll {
namespace {

// One piece a phase moves: `nl` lines at `lines` in a rank or owner image,
// and `left` payload bytes (positive for the piece's rows) at `plain` in an
// input or output buffer.
struct ColPiece {
  char* lines;
  char* plain;
  int nl;
  int left;
};

__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Stage: input rows (480 payload bytes) -> LL128 rows (512 bytes).  Here a
// piece's `plain` is the input and `lines` the staged lines.
template <int kW, int kRing>
__device__ __forceinline__ void col_stage(const ColPiece* pc, int np, int R, uint32_t wbase,
                                          int lane, int warp, uint64_t seq, uint64_t pol) {
  const int T = np * R;
  const int lo = (T * warp) / kW, nj = (T * (warp + 1)) / kW - lo;
  if (nj <= 0) return;
  const int li = lane >> 3, kk = lane & 7;
  const int G = 15 * li + 2 * kk;  // first payload granule of this lane's line chunk
  // lanes 30 and 31 load no input (their load bound is never met)
  const int lb = lane < 30 ? 16 * lane : 1 << 30;
  int lk = lo / R, lr = lo - lk * R;
  const char* lsrc = pc[lk].plain + (size_t)lr * (2 * kRowElems);
  int lleft = pc[lk].left - lr * (2 * kRowElems);
  auto issue = [&](int j) {
    if (j < nj) {
      const bool valid = lb < lleft;
      cp_async16_hint(wbase + (j % kRing) * kRowBytes + 16 * lane,
                      lsrc + (valid ? 16 * lane : 0), valid, pol);
      lsrc += 2 * kRowElems;
      lleft -= 2 * kRowElems;
      if (++lr == R) {
        lr = 0;
        if (++lk < np) {
          lsrc = pc[lk].plain;
          lleft = pc[lk].left;
        }
      }
    }
    cp_async_commit();
  };
  int sk = lk, sr = lr;
  char* sdst = pc[sk].lines + (size_t)sr * kRowBytes;
  int snl = pc[sk].nl - kLL128RowLines * sr;
#pragma unroll 1
  for (int j = 0; j < kRing; ++j) issue(j);
  for (int j = 0; j < nj; ++j) {
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint32_t row = wbase + (j % kRing) * kRowBytes;
    // lanes 30, 31 hold no input: their slot bytes [480, 512) stay unread
    const uint2 a = lds_v2(row + 8 * G);
    const uint2 b = kk == 7 ? make_uint2(0, 0) : lds_v2(row + 8 * (G + 1));
    __syncwarp();
    issue(j + kRing);
    if (snl > 0)
      ll128_store_row<false>(sdst, make_uint4(a.x, a.y, b.x, b.y), lane,
                             min((int)kLL128RowLines, snl), seq);
    sdst += kRowBytes;
    snl -= kLL128RowLines;
    if (++sr == R) {
      sr = 0;
      if (++sk < np) {
        sdst = pc[sk].lines;
        snl = pc[sk].nl;
      }
    }
  }
  cp_async_wait<0>();
  __syncwarp();
}

// Gather: validated LL128 rows -> output rows.  A piece's `lines` is the
// source and `plain` the output; a timeout report names the piece index as
// the rank.
template <int kW, int kRing>
__device__ __forceinline__ bool col_gather(const RunParams& P, const ColPiece* pc, int np,
                                           int R, uint32_t wbase, int lane, int warp,
                                           uint64_t seq, uint64_t pol) {
  const int T = np * R;
  const int lo = (T * warp) / kW, nj = (T * (warp + 1)) / kW - lo;
  if (nj <= 0) return true;
  const int li = lane >> 3;
  const bool k7 = (lane & 7) == 7;
  // output chunk q = lane: its two payload granules in the row; lanes 30
  // and 31 hold none (their store bound is never met)
  const int q = lane < 30 ? lane : 29;
  const int lb = lane < 30 ? 16 * lane : 1 << 30;
  const uint32_t g0off = 128 * ((2 * q) / 15) + 8 * ((2 * q) % 15);
  const uint32_t g1off = 128 * ((2 * q + 1) / 15) + 8 * ((2 * q + 1) % 15);
  int lk = lo / R, lr = lo - lk * R;
  const char* lsrc = pc[lk].lines + (size_t)lr * kRowBytes;
  int lnl = pc[lk].nl - kLL128RowLines * lr;
  auto issue = [&](int j) {
    if (j < nj) {
      cp_async16(wbase + (j % kRing) * kRowBytes + 16 * lane, lsrc + 16 * lane, li < lnl);
      lsrc += kRowBytes;
      lnl -= kLL128RowLines;
      if (++lr == R) {
        lr = 0;
        if (++lk < np) {
          lsrc = pc[lk].lines;
          lnl = pc[lk].nl;
        }
      }
    }
    cp_async_commit();
  };
  int sk = lk, sr = lr;
  const char* ssrc = pc[sk].lines + (size_t)sr * kRowBytes;
  char* sdst = pc[sk].plain + (size_t)sr * (2 * kRowElems);
  int snl = pc[sk].nl - kLL128RowLines * sr;
  int sleft = pc[sk].left - sr * (2 * kRowElems);
#pragma unroll 1
  for (int j = 0; j < kRing; ++j) issue(j);
  bool ok = true;
  for (int j = 0; j < nj; ++j) {
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint32_t row = wbase + (j % kRing) * kRowBytes;
    const bool valid = li < snl;
    // every lane loads the upper half of its chunk; only the last chunk of a
    // line holds the number
    const uint64_t num = lds_u64(row + 16 * lane + 8);
    const bool ready = !(valid && k7) || num == seq;
    if (!__all_sync(0xFFFFFFFFu, ready)) {
      // the phase barrier ordered these lines' stores before this load, so
      // this only happens if the protocol is broken: wait, bounded
      ok = ll128_wait_chunk(P, ssrc, lane, ready, seq, (uint32_t)sk,
                            (int64_t)sr * kLL128RowLines);
      if (!ok) break;
      if (valid) sts_v4(row + 16 * lane, ld_v4(ssrc + 16 * lane));
      __syncwarp();
    }
    const uint2 a = lds_v2(row + g0off), b = lds_v2(row + g1off);
    __syncwarp();  // every lane read the slot before it is refilled
    issue(j + kRing);
    if (lb < sleft) st_v4_hint(sdst + 16 * lane, make_uint4(a.x, a.y, b.x, b.y), pol);
    ssrc += kRowBytes;
    sdst += 2 * kRowElems;
    snl -= kLL128RowLines;
    sleft -= 2 * kRowElems;
    if (++sr == R) {
      sr = 0;
      if (++sk < np) {
        ssrc = pc[sk].lines;
        sdst = pc[sk].plain;
        snl = pc[sk].nl;
        sleft = pc[sk].left;
      }
    }
  }
  cp_async_wait<0>();
  __syncwarp();
  return ok;
}

// Fold: the column's rows of every rank image (staged at line `src_line`),
// validated and folded in rank order; published as lines at `ag`
// (all-reduce) or written into owner x's output from element `out0`
// (reduce-scatter, `left` payload bytes).  Rows rr = warp, warp + kW, ...;
// kRing / kMaxRanks rows of all N images in flight per warp.
template <int kW, int kRing, bool kF32>
__device__ __forceinline__ bool col_fold(const RunParams& P, uint32_t wbase, int lane, int warp,
                                         int nl, uint64_t src_line, char* ag, uint16_t* out,
                                         int left, uint64_t e, uint64_t seq, bool discard) {
  constexpr int kStages = kRing / kMaxRanks;
  const int n = P.nranks;
  const int li = lane >> 3;
  const char* src0 = image_bytes(P, P.P, e, 0) + src_line * kLL128LineBytes + 16 * lane;
  const uint64_t rb = P.P.rank_bytes;
  const int nrows = (nl + kLL128RowLines - 1) / kLL128RowLines;
  const int nj = warp < nrows ? (nrows - warp + kW - 1) / kW : 0;
  const uint32_t seq_lo = (uint32_t)seq, seq_hi = (uint32_t)(seq >> 32);
  auto issue = [&](int j) {
    if (j < nj) {
      const int rr = warp + j * kW;
      const bool valid = li < nl - rr * kLL128RowLines;
      const uint32_t sl = wbase + (uint32_t)((j % kStages) * kMaxRanks * kRowBytes) + 16 * lane;
      const char* g = src0 + (size_t)rr * kRowBytes;
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p)
        if (p < n) cp_async16(sl + p * kRowBytes, g + p * rb, valid);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int j = 0; j < kStages; ++j) issue(j);
  bool ok = true;
  for (int j = 0; j < nj; ++j) {
    cp_async_wait<kStages - 1>();
    const uint32_t sl = wbase + (uint32_t)((j % kStages) * kMaxRanks * kRowBytes) + 16 * lane;
    const int rr = warp + j * kW;
    const int nl_row = min((int)kLL128RowLines, nl - rr * kLL128RowLines);
    const bool valid = li < nl_row;
    // each rank's chunk is checked and folded as it is read from shared
    // memory, in rank order
    ChunkFold<kF32> acc;
    uint32_t bad;
    {
      const uint4 v = lds_v4(sl);
      bad = (v.z ^ seq_lo) | (v.w ^ seq_hi);
      acc.first(v);
    }
#pragma unroll
    for (int p = 1; p < kMaxRanks; ++p)
      if (p < n) {
        const uint4 v = lds_v4(sl + p * kRowBytes);
        bad |= (v.z ^ seq_lo) | (v.w ^ seq_hi);
        acc.add(v);
      }
    const bool ready = !(valid && (lane & 7) == 7) || bad == 0;
    if (!__all_sync(0xFFFFFFFFu, ready)) {
      // the phase barrier ordered these lines' stores before this load, so
      // this only happens if the protocol is broken: wait (bounded) for
      // every rank's numbers on global memory, then fold the row again
      // from there
      const uint64_t row_line = src_line + (uint64_t)rr * kLL128RowLines;
      for (int p = 0; p < n && ok; ++p) {
        const bool rp = ll128_chunk_ready(lds_v4(sl + p * kRowBytes), lane, valid, seq);
        if (!__all_sync(0xFFFFFFFFu, rp))
          ok = ll128_wait_chunk(P, src0 - 16 * lane + p * rb + (size_t)rr * kRowBytes, lane, rp,
                                seq, p, (int64_t)row_line);
      }
      if (!ok) break;
      const char* grow = src0 + (size_t)rr * kRowBytes;
      acc.first(valid ? ld_v4(grow) : make_uint4(0, 0, 0, 0));
      for (int p = 1; p < n; ++p) acc.add(valid ? ld_v4(grow + p * rb) : make_uint4(0, 0, 0, 0));
    }
    issue(j + kStages);
    // the staged lines of this row have no other reader: drop them
    if (discard && lane < 4 * n && (lane & 3) < nl_row)
      discard_l2_line(src0 - 16 * lane + (lane >> 2) * rb + (size_t)rr * kRowBytes +
                      (size_t)(lane & 3) * kLL128LineBytes);
    const uint4 res = acc.result();
    if (out != nullptr) {
      const int lrow = left - rr * (2 * kRowElems);
      const uint4 pay = lines_to_payload(res, lane);
      if (lane < 30 && 16 * lane < lrow) st_v4(out + (size_t)rr * kRowElems + 8 * lane, pay);
    } else {
      ll128_store_row<false>(ag + (size_t)rr * kRowBytes, res, lane, nl_row, seq);
    }
  }
  cp_async_wait<0>();
  __syncwarp();
  return ok;
}

__device__ __forceinline__ int seg_lines(const RunParams& P, int k) {
  return (int)((P.seg_elems[k] + kLL128Elems - 1) / kLL128Elems);
}

// An all-to-all piece of chunk t0: `elems` units at `plain` (the input of
// the stage, or the output of the copy), whose lines start at `line` of
// `image`.  A source partition shorter than the column has fewer lines (or
// none) in the chunk.
__device__ __forceinline__ void exch_piece(ColPiece& pc, const uint16_t* plain, char* image,
                                           uint64_t line, uint64_t elems, uint32_t t0,
                                           uint32_t CL) {
  const int64_t lines = (int64_t)((elems + kLL128Elems - 1) / kLL128Elems) - (int64_t)t0;
  const int64_t bytes = 2 * ((int64_t)elems - (int64_t)t0 * kLL128Elems);
  pc.plain = const_cast<char*>(reinterpret_cast<const char*>(plain + (uint64_t)t0 * kLL128Elems));
  pc.lines = image + line * kLL128LineBytes;
  pc.nl = (int)max((int64_t)0, min((int64_t)CL, lines));
  pc.left = (int)max((int64_t)0, min((int64_t)CL * (2 * kLL128Elems), bytes));
}

// Rows of the g-th column of a staggered group (g = 0 .. G-1): 1/G, 2/G,
// .. of a chunk, at least one row.
__device__ __forceinline__ int stagger_rows(int g, int G, int chunk_rows) {
  return max(1, ((g + 1) * chunk_rows) / G);
}

// Column q of an unbounded run: its partition x, first line t0 and lines.
// The first `first_cols` columns (one per CTA at the start) come in groups
// of `stagger` columns of 1/G, 2/G, .. of a chunk, so that the CTAs end
// their first column at different times and their later phases do not all
// hit memory together; then chunks of chunk_lines, and after head_chunks of
// them, chunks of tail_lines.
struct ColumnAt {
  int x;
  uint32_t t0, len;
};
__device__ __forceinline__ ColumnAt column_at(const ComposedParams& Q, int q, int n) {
  ColumnAt a;
  if (q < (int)Q.first_cols) {
    const int j = q / n, G = (int)Q.stagger, cr = (int)Q.chunk_lines / kLL128RowLines;
    const int grp = j / G, g = j - grp * G;
    int rows = 0;
    for (int i = 0; i < G; ++i) rows += stagger_rows(i, G, cr);
    rows *= grp;
    for (int i = 0; i < g; ++i) rows += stagger_rows(i, G, cr);
    a.x = q - j * n;
    a.t0 = (uint32_t)rows * kLL128RowLines;
    a.len = (uint32_t)stagger_rows(g, G, cr) * kLL128RowLines;
    return a;
  }
  q -= (int)Q.first_cols;
  const int c = q / n;
  a.x = q - c * n;
  if (c < (int)Q.head_chunks) {
    a.t0 = Q.first_lines + (uint32_t)c * Q.chunk_lines;
    a.len = Q.chunk_lines;
  } else {
    a.t0 = Q.first_lines + Q.head_chunks * Q.chunk_lines + (uint32_t)(c - (int)Q.head_chunks) * Q.tail_lines;
    a.len = Q.tail_lines;
  }
  return a;
}

template <int kW, int kRing, int kMinBlocks, bool kF32>
__global__ void __launch_bounds__(kW * 32, kMinBlocks) k_column_ll128(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  __shared__ ColPiece s_piece[2][kMaxRanks];  // [0] stage pieces, [1] gather pieces
  __shared__ int s_col[2];
  __shared__ int s_ok;
  const uint64_t e = begin_run_per_thread(P);
  const ComposedParams& Q = P.cp;
  WsHeader* h = header(P.ws);
  const int n = P.nranks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = (int)(e & 1);
  const int ncols = (int)Q.first_cols + (int)Q.nchunks * n;
  const bool bounded = Q.ring != 0;
  const uint32_t CL = Q.chunk_lines;
  const uint32_t wbase =
      (uint32_t)__cvta_generic_to_shared(smem) + (uint32_t)(warp * kRing * kRowBytes);
  const bool folds = Q.mode == 0 || Q.mode == 1, gathers = Q.mode != 1;
  const uint64_t pol = l2_evict_first_policy();  // inputs and outputs are touched once
  if (threadIdx.x == 0) {
    // every CTA's first column is its own index; later ones come from the
    // run's counter, past the grid (bounded staging: every grid-th column)
    s_col[0] = (int)blockIdx.x;
    s_ok = 1;
  }
  __syncthreads();
  for (int it = 0;; ++it) {
    const int q = s_col[it & 1];
    if (q >= ncols) break;
    if (threadIdx.x == 0)
      s_col[(it + 1) & 1] = aborted(P.ws) ? ncols
                            : bounded     ? q + (int)gridDim.x
                                          : (int)gridDim.x + (int)atomicAdd(&h->task_next[slot], 1u);
    ColumnAt at;
    if (bounded) {
      at.x = q % n;
      at.t0 = (uint32_t)(q / n) * CL;
      at.len = CL;
    } else {
      at = column_at(Q, q, n);
    }
    const int x = at.x;
    const uint32_t t0 = at.t0, cl = at.len;
    const int R = (int)cl / kLL128RowLines;  // rows per piece
    const uint64_t seq = bounded ? e + (uint64_t)q : e;
    // the column's line in every rank image, and in owner x's published image
    const uint64_t pline = bounded ? (uint64_t)blockIdx.x * CL : P.seg_line0[x] + t0;
    const uint64_t agline = bounded ? (uint64_t)(blockIdx.x / n) * CL : (uint64_t)t0;
    const int nl = max(0, min((int)cl, seg_lines(P, x) - (int)t0));
    const int64_t lx = 2 * ((int64_t)P.seg_elems[x] - (int64_t)t0 * kLL128Elems);
    const int left = (int)(lx < (int64_t)cl * (2 * kLL128Elems) ? lx
                                                                : (int64_t)cl * (2 * kLL128Elems));
    if (nl == 0) {
      // partition x is shorter than the longest one (V sizes): nothing to
      // move in this chunk.  The barrier publishes the next column.
      __syncthreads();
      continue;
    }
    // stage: rank p's piece of column x (all-gather: source x's one piece;
    // all-to-all: source p's partition x, whose length is its own)
    const int nstage = Q.mode == 3 ? 1 : n;
    if ((int)threadIdx.x < nstage) {
      const int p = Q.mode == 3 ? x : (int)threadIdx.x;
      ColPiece& pc = s_piece[0][threadIdx.x];
      if (Q.mode == 2) {
        const ExchPiece v = Q.exch[p * n + x];
        exch_piece(pc, P.in[p] + v.in0, image_bytes(P, P.P, e, p), bounded ? pline : v.line0 + t0,
                   v.elems, t0, cl);
      } else {
        pc.plain = const_cast<char*>(reinterpret_cast<const char*>(
            P.in[p] + (Q.mode == 3 ? 0 : P.seg_in0[x]) + (uint64_t)t0 * kLL128Elems));
        pc.lines = image_bytes(P, P.P, e, p) + pline * kLL128LineBytes;
        pc.nl = nl;
        pc.left = left;
      }
    }
    __syncthreads();
    col_stage<kW, kRing>(s_piece[0], nstage, R, wbase, lane, warp, seq, pol);
    __syncthreads();
    char* ag = image_bytes(P, P.AG, e, x) + agline * kLL128LineBytes;
    if (folds) {
      // the element type is the kernel's template parameter, so no row
      // carries the other type's fold
      uint16_t* out = P.out[x] + (uint64_t)t0 * kLL128Elems;
      const bool dsc = Q.discard != 0;
      if (!col_fold<kW, kRing, kF32>(P, wbase, lane, warp, nl, pline, ag,
                                     Q.mode == 1 ? out : nullptr, left, e, seq, dsc))
        s_ok = 0;
      __syncthreads();
      if (!s_ok) break;
    }
    if (gathers) {
      // piece d: all-reduce, all-gather: the column's lines into partition x
      // of destination d's output; all-to-all: source d's staged piece into
      // block d of destination x's output
      if ((int)threadIdx.x < n) {
        const int d = (int)threadIdx.x;
        ColPiece& pc = s_piece[1][d];
        if (Q.mode == 0) {
          pc.lines = ag;
          pc.plain = reinterpret_cast<char*>(P.out[d] + P.seg_in0[x] + (uint64_t)t0 * kLL128Elems);
        } else if (Q.mode == 2) {
          const ExchPiece v = Q.exch[d * n + x];
          exch_piece(pc, P.out[x] + v.out0, image_bytes(P, P.P, e, d),
                     bounded ? pline : v.line0 + t0, v.elems, t0, cl);
        } else {
          pc.lines = image_bytes(P, P.P, e, x) + pline * kLL128LineBytes;
          pc.plain = reinterpret_cast<char*>(P.out[d] + P.seg_in0[x] + (uint64_t)t0 * kLL128Elems);
        }
        if (Q.mode != 2) {
          pc.nl = nl;
          pc.left = left;
        }
      }
      __syncthreads();
      if (!col_gather<kW, kRing>(P, s_piece[1], n, R, wbase, lane, warp, seq, pol)) s_ok = 0;
      __syncthreads();
      if (!s_ok) break;
      if (Q.discard) {
        // every reader of these lines is done (the barrier above): drop them
        // before they are written back.  All-to-all: the N sources' staged
        // pieces; otherwise the one piece every destination read.
        // Each piece's own line count: past it lie other columns' lines.
        const int npieces = Q.mode == 2 ? n : 1;
        for (int k = 0; k < npieces; ++k) {
          const char* src = s_piece[1][k].lines;
          const int pnl = s_piece[1][k].nl;
          for (int j = threadIdx.x; j < pnl; j += blockDim.x)
            discard_l2_line(src + (size_t)j * kLL128LineBytes);
        }
      }
    }
  }
  finish_run(P, e);
}

// Launch shapes: warps per CTA, rows in flight per warp, CTAs per SM.
struct ColVariant {
  int warps, ring;
};
constexpr ColVariant kColVariants[3] = {{8, 16}, {8, 24}, {4, 16}};

template <int W, int R, int B>
int capacity_of() {
  static size_t memo[kMaxDevices], memo32[kMaxDevices];
  const int bytes = (int)((size_t)W * R * kRowBytes);
  if (raise_smem_limit(k_column_ll128<W, R, B, false>, (size_t)bytes, memo) != cudaSuccess ||
      raise_smem_limit(k_column_ll128<W, R, B, true>, (size_t)bytes, memo32) != cudaSuccess)
    return 0;
  int per_sm = 0, per_sm32 = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_column_ll128<W, R, B, false>,
                                                    W * 32, bytes) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm32, k_column_ll128<W, R, B, true>,
                                                    W * 32, bytes) != cudaSuccess)
    return 0;
  return std::min(per_sm, per_sm32) * device_sms();
}

}  // namespace

int column_threads(int variant) {
  const int v = variant >= 0 && variant <= 2 ? variant : 0;
  return kColVariants[v].warps * 32;
}

int column_capacity(int variant) {
  if (variant == 1) return capacity_of<8, 24, 2>();
  if (variant == 2) return capacity_of<4, 16, 6>();
  return capacity_of<8, 16, 3>();
}

cudaError_t launch_column(const RunParams& P, int grid, cudaStream_t s, bool dependent) {
  const int v = P.cp.variant >= 0 && P.cp.variant <= 2 ? P.cp.variant : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kColVariants[v].warps * 32);
  cfg.dynamicSmemBytes = (size_t)kColVariants[v].warps * kColVariants[v].ring * kRowBytes;
  cfg.stream = s;
  // co-resident CTAs: the grid's last CTA counts every CTA in before it
  // advances the epoch
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 2 : 1;
  const bool f32 = P.dtype == kDtF32;
  if (v == 1)
    return f32 ? cudaLaunchKernelEx(&cfg, k_column_ll128<8, 24, 2, true>, P)
               : cudaLaunchKernelEx(&cfg, k_column_ll128<8, 24, 2, false>, P);
  if (v == 2)
    return f32 ? cudaLaunchKernelEx(&cfg, k_column_ll128<4, 16, 6, true>, P)
               : cudaLaunchKernelEx(&cfg, k_column_ll128<4, 16, 6, false>, P);
  return f32 ? cudaLaunchKernelEx(&cfg, k_column_ll128<8, 16, 3, true>, P)
             : cudaLaunchKernelEx(&cfg, k_column_ll128<8, 16, 3, false>, P);
}

}  // namespace coll
