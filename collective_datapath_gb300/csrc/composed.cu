// composed.cu -- the twoshot all-reduce as one persistent cooperative launch.
//
// Purlin §3.2 ("Extending the execution to AllReduce", Figure 5, Algorithm 1)
// runs the reduce-scatter and the all-gather of a twoshot all-reduce as
// concurrent stage, reduce and gather work at chunk granularity, with chunk
// completion signalled to the next role.  Here every partition is cut into
// chunks of `chunk_lines` LL128 lines and the run is a queue of tasks:
//   stage  S(c, p): rank p's input -> its staged lines of chunk c (all N
//                   partitions);
//   fold   F(c, r): chunk c of partition r from all N staged images ->
//                   folded in rank order, published as lines of owner r;
//   gather G(c, d): chunk c of every owner's published partition -> rank d's
//                   output.
// Queue step t holds S(t, *), then F(t - lag, *), then G(t - lag - lag2, *).  CTAs
// take tasks in queue order from one counter, so a task only ever waits for
// tasks that are earlier in the queue and already taken by co-resident CTAs:
// the earliest unfinished task waits for nothing, so the launch always
// progresses.  The lag keeps a chunk's staged and published lines in L2
// between producer and reader (the working set is about `lag` steps of
// chunks, a few tens of MB at most), and a staged line's only reader drops
// it from L2 once folded, so staging does not reach HBM.
//
// Readiness: a producer task stores its lines (data and the epoch as the
// LL128 sequence number), then __syncthreads, one fence.acq_rel.gpu and the
// task's flag = epoch (release); a consumer task waits for the flags of the
// N tasks it reads (acquire fence, __syncthreads), loads the lines and still
// checks every line's number.  Flags hold epochs, so they never need a
// reset.  The gather count of a chunk carries the epoch in its high bits; the
// N-th gather of a chunk drops the published lines of that chunk from L2.
#include <cuda_runtime.h>

#include "launch.h"
#include "ll128.cuh"
#include "pipe.cuh"

namespace coll {

// Launch shapes: kW warps per CTA, kCRing rows in flight per warp (stage,
// gather; the fold keeps kCRing / 8 rows of all N images), kMinBlocks CTAs
// per SM.
//   variant 0: 8 warps, 16 rows, 3 CTAs per SM (64 KB of shared memory each)
//   variant 1: 8 warps, 24 rows, 2 CTAs per SM (96 KB each)
//   variant 2: 4 warps, 16 rows, 6 CTAs per SM (32 KB each)
struct CVariant {
  int warps, ring;
};
constexpr CVariant kCVariants[3] = {{8, 16}, {8, 24}, {4, 16}};

size_t composed_smem_bytes(int variant) {
  const CVariant v = kCVariants[variant];
  return (size_t)v.warps * v.ring * kRowBytes;
}

__device__ __forceinline__ void discard_l2_line(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ int seg_lines_of(const RunParams& P, int k) {
  return (int)((P.seg_elems[k] + kLL128Elems - 1) / kLL128Elems);
}

// Lines of segment k inside the chunk starting at line t0 (0 past its end).
__device__ __forceinline__ int chunk_lines_of(const RunParams& P, int k, uint32_t t0) {
  return max(0, min((int)P.cp.chunk_lines, seg_lines_of(P, k) - (int)t0));
}

// Threads 0..n-1 wait (bounded) for flags[thread] == e, each then fences
// (acquire); the caller's __syncthreads hands the ordering to the CTA.
__device__ __forceinline__ bool acquire_flags(const RunParams& P, const uint64_t* flags, int n,
                                              uint64_t e) {
  bool ok = true;
  if ((int)threadIdx.x < n) {
    const uint64_t* f = flags + threadIdx.x;
    if (ld_relaxed_u64(f) != e) {
      Waiter w;
      while (ld_relaxed_u64(f) != e) {
        if (w.expired(P.ws, P.timeout_ns)) {
          latch_error(P.ws, kStatusTimeout, threadIdx.x, -3);
          ok = false;
          break;
        }
        __nanosleep(64);
      }
    }
    fence_acq_rel_gpu();
  }
  return ok;
}

// After every data store of the CTA: one release of the task's flag, unless
// the task failed.
__device__ __forceinline__ void release_flag(uint64_t* flag, uint64_t e, const int& s_ok) {
  __syncthreads();
  if (threadIdx.x == 0 && s_ok) {
    fence_acq_rel_gpu();
    st_relaxed_u64(flag, e);
  }
}

// Per-task descriptors of the N pieces a stage or gather task moves (one
// per partition), filled by threads 0..n-1 before the task's first barrier.
// Rows of the task are numbered i = piece * R + row, R = chunk_lines / 4 a
// power of two; rows past a short piece are skipped.
struct Piece {
  const char* src;  // first source byte of the piece in this chunk
  char* dst;        // first destination byte
  int nl;           // lines of the piece in this chunk
  int left;         // payload elements of the piece from the chunk start
};

__device__ __forceinline__ void fill_stage_piece(const RunParams& P, Piece* pc, int c, int p,
                                                 uint64_t e, uint32_t W) {
  const int k = threadIdx.x;
  const uint32_t t0 = (uint32_t)c * P.cp.chunk_lines;
  pc[k].src = reinterpret_cast<const char*>(P.in[p] + P.seg_in0[k] + (uint64_t)t0 * kLL128Elems);
  // cycling staging: chunk slot c mod W holds the N partitions' lines of the
  // chunk, partition-major; otherwise each partition's lines sit in place
  const uint64_t line = W ? ((uint64_t)(c % W) * P.nranks + k) * P.cp.chunk_lines
                         : P.seg_line0[k] + t0;
  pc[k].dst = image_bytes(P, P.P, e, p) + line * kLL128LineBytes;
  pc[k].nl = chunk_lines_of(P, k, t0);
  const int64_t lk = (int64_t)P.seg_elems[k] - (int64_t)t0 * kLL128Elems;
  pc[k].left = (int)(lk < (int64_t)P.cp.chunk_lines * kLL128Elems ? lk
                                                                  : (int64_t)P.cp.chunk_lines * kLL128Elems);
}

__device__ __forceinline__ void fill_gather_piece(const RunParams& P, Piece* pc, int c, int d,
                                                  uint64_t e, uint32_t W) {
  const int r = threadIdx.x;
  const uint32_t t0 = (uint32_t)c * P.cp.chunk_lines;
  const uint64_t line = W ? (uint64_t)(c % W) * P.cp.chunk_lines : t0;
  pc[r].src = image_bytes(P, P.AG, e, r) + line * kLL128LineBytes;
  pc[r].dst = reinterpret_cast<char*>(P.out[d] + P.seg_in0[r] + (uint64_t)t0 * kLL128Elems);
  pc[r].nl = chunk_lines_of(P, r, t0);
  const int64_t lr = (int64_t)P.seg_elems[r] - (int64_t)t0 * kLL128Elems;
  pc[r].left = (int)(lr < (int64_t)P.cp.chunk_lines * kLL128Elems ? lr
                                                                  : (int64_t)P.cp.chunk_lines * kLL128Elems);
}

// All-to-all: destination d copies segment d of every source r.
__device__ __forceinline__ void fill_a2a_piece(const RunParams& P, Piece* pc, int c, int d,
                                               uint64_t e, uint32_t W) {
  const int r = threadIdx.x;
  const uint32_t t0 = (uint32_t)c * P.cp.chunk_lines;
  const uint64_t line = W ? ((uint64_t)(c % W) * P.nranks + d) * P.cp.chunk_lines
                         : P.seg_line0[d] + t0;
  pc[r].src = image_bytes(P, P.P, e, r) + line * kLL128LineBytes;
  pc[r].dst = reinterpret_cast<char*>(P.out[d] + P.seg_in0[r] + (uint64_t)t0 * kLL128Elems);
  pc[r].nl = chunk_lines_of(P, d, t0);
  const int64_t ld = (int64_t)P.seg_elems[d] - (int64_t)t0 * kLL128Elems;
  pc[r].left = (int)(ld < (int64_t)P.cp.chunk_lines * kLL128Elems
                         ? ld
                         : (int64_t)P.cp.chunk_lines * kLL128Elems);
}

// All-gather (mode 3): rank p stages chunk c of its one packed segment;
// the seg_* fields hold each source's segment and its output offset.
__device__ __forceinline__ void fill_ag_stage_piece(const RunParams& P, Piece* pc, int c, int p,
                                                    uint64_t e) {
  const uint32_t t0 = (uint32_t)c * P.cp.chunk_lines;
  pc[0].src = reinterpret_cast<const char*>(P.in[p] + (uint64_t)t0 * kLL128Elems);
  pc[0].dst = image_bytes(P, P.P, e, p) + (P.seg_line0[p] + t0) * kLL128LineBytes;
  pc[0].nl = chunk_lines_of(P, p, t0);
  const int64_t lk = (int64_t)P.seg_elems[p] - (int64_t)t0 * kLL128Elems;
  pc[0].left = (int)(lk < (int64_t)P.cp.chunk_lines * kLL128Elems
                         ? lk
                         : (int64_t)P.cp.chunk_lines * kLL128Elems);
}

// All-gather copy: destination d copies chunk c of every source r's staged
// segment into partition r of its output.
__device__ __forceinline__ void fill_ag_copy_piece(const RunParams& P, Piece* pc, int c, int d,
                                                   uint64_t e) {
  const int r = threadIdx.x;
  const uint32_t t0 = (uint32_t)c * P.cp.chunk_lines;
  pc[r].src = image_bytes(P, P.P, e, r) + (P.seg_line0[r] + t0) * kLL128LineBytes;
  pc[r].dst = reinterpret_cast<char*>(P.out[d] + P.seg_in0[r] + (uint64_t)t0 * kLL128Elems);
  pc[r].nl = chunk_lines_of(P, r, t0);
  const int64_t lr = (int64_t)P.seg_elems[r] - (int64_t)t0 * kLL128Elems;
  pc[r].left = (int)(lr < (int64_t)P.cp.chunk_lines * kLL128Elems
                         ? lr
                         : (int64_t)P.cp.chunk_lines * kLL128Elems);
}

template <int kCWarps, int kCRing>
__device__ __forceinline__ void stage_task(const Piece* pc, uint32_t wbase, int lane, int warp,
                                           int n, int rsh, uint64_t e) {
  const int li = lane >> 3, kk = lane & 7;
  const int G = 15 * li + 2 * kk;  // first payload granule of this lane's line chunk
  const int rmask = (1 << rsh) - 1;
  const int nrows = n << rsh;
  const int nj = warp < nrows ? (nrows - warp + kCWarps - 1) / kCWarps : 0;
  const uint64_t pol = l2_evict_first_policy();  // inputs are read once
  auto issue = [&](int j) {
    if (j < nj) {
      const int i = warp + j * kCWarps, k = i >> rsh, r = i & rmask;
      const int left = pc[k].left - r * kRowElems;
      const bool valid = 4 * r < pc[k].nl && lane < 30 && 8 * lane < left;
      cp_async16_hint(wbase + (j % kCRing) * kRowBytes + 16 * lane,
                      pc[k].src + (size_t)r * (2 * kRowElems) + (valid ? 16 * lane : 0), valid,
                      pol);
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int j = 0; j < kCRing; ++j) issue(j);
  for (int j = 0; j < nj; ++j) {
    cp_async_wait<kCRing - 1>();
    __syncwarp();
    const uint32_t row = wbase + (j % kCRing) * kRowBytes;
    // lanes 30, 31 hold no input: their slot bytes [480, 512) stay unread
    const uint2 a = lds_v2(row + 8 * G);
    const uint2 b = kk == 7 ? make_uint2(0, 0) : lds_v2(row + 8 * (G + 1));
    __syncwarp();
    issue(j + kCRing);
    const int i = warp + j * kCWarps, k = i >> rsh, r = i & rmask;
    const int nl_row = pc[k].nl - 4 * r;
    if (nl_row > 0)
      ll128_store_row<false>(pc[k].dst + (size_t)r * kRowBytes, make_uint4(a.x, a.y, b.x, b.y),
                             lane, min((int)kLL128RowLines, nl_row), e);
  }
  cp_async_wait<0>();
  __syncwarp();
}

// Fold the `nl` lines of partition r that start at line t0 of the segment
// (staged at line src_line of every rank image) over the N images, in rank
// order; publish the result as lines at `ag` (all-reduce) or write it into
// rank r's output (reduce-scatter).
template <int kCWarps, int kCRing>
__device__ __forceinline__ bool fold_rows(const RunParams& P, uint32_t wbase, int lane, int warp,
                                          int r, uint32_t t0, int nl, uint64_t src_line,
                                          char* ag, uint64_t e, uint64_t seq, bool to_out) {
  constexpr int kCFoldStages = kCRing / kMaxRanks;  // rows of all N images per warp
  const int n = P.nranks;
  const int li = lane >> 3;
  // rank p's rows of this piece start at src0 + p * rank_bytes
  const char* src0 = image_bytes(P, P.P, e, 0) + src_line * kLL128LineBytes;
  const uint64_t rb = P.P.rank_bytes;
  const int nrows = (nl + kLL128RowLines - 1) / kLL128RowLines;
  const int nj = warp < nrows ? (nrows - warp + kCWarps - 1) / kCWarps : 0;
  auto issue = [&](int j) {
    if (j < nj) {
      const int rr = warp + j * kCWarps;
      const bool valid = li < nl - rr * kLL128RowLines;
      const uint32_t sl = wbase + (uint32_t)((j % kCFoldStages) * kMaxRanks * kRowBytes) + 16 * lane;
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p)
        if (p < n)
          cp_async16(sl + p * kRowBytes, src0 + p * rb + (size_t)rr * kRowBytes + 16 * lane, valid);
    }
    cp_async_commit();
  };
#pragma unroll
  for (int j = 0; j < kCFoldStages; ++j) issue(j);
  bool ok = true;
  for (int j = 0; j < nj; ++j) {
    cp_async_wait<kCFoldStages - 1>();
    const uint32_t sl = wbase + (uint32_t)((j % kCFoldStages) * kMaxRanks * kRowBytes) + 16 * lane;
    const int rr = warp + j * kCWarps;
    const int nl_row = min((int)kLL128RowLines, nl - rr * kLL128RowLines);
    const bool valid = li < nl_row;
    uint4 s[kMaxRanks];
#pragma unroll
    for (int p = 0; p < kMaxRanks; ++p)
      if (p < n) s[p] = lds_v4(sl + p * kRowBytes);
    bool ready = true;
#pragma unroll
    for (int p = 0; p < kMaxRanks; ++p)
      if (p < n) ready = ready && ll128_chunk_ready(s[p], lane, valid, seq);
    if (!__all_sync(0xFFFFFFFFu, ready)) {
      // the producer's flag was set, so this only happens if the protocol
      // is broken: wait for the numbers on global memory, bounded
      const uint64_t row_line = src_line + (uint64_t)rr * kLL128RowLines;
#pragma unroll
      for (int p = 0; p < kMaxRanks; ++p) {
        if (p < n && ok) {
          const bool rp = ll128_chunk_ready(s[p], lane, valid, seq);
          if (!__all_sync(0xFFFFFFFFu, rp)) {
            const char* grow = src0 + p * rb + (size_t)rr * kRowBytes;
            ok = ll128_wait_chunk(P, grow, lane, rp, seq, p, (int64_t)row_line);
            if (ok && valid) s[p] = ld_v4(grow + 16 * lane);
          }
        }
      }
      if (!ok) break;
    }
    issue(j + kCFoldStages);
    // the staged lines of this row have no other reader: drop them
    if (P.cp.discard && lane < 4 * n && (lane & 3) < nl_row) {
      discard_l2_line(src0 + (lane >> 2) * rb + (size_t)rr * kRowBytes +
                      (size_t)(lane & 3) * kLL128LineBytes);
    }
    const uint4 res = ll128_fold(s, n, P.dtype);
    if (to_out) {
      const uint64_t line = (uint64_t)t0 + (uint64_t)rr * kLL128RowLines;
      ll128_write_payload(P.out[r] + line * kLL128Elems, res, lane,
                          (int64_t)P.seg_elems[r] - (int64_t)line * kLL128Elems);
    } else {
      ll128_store_row<false>(ag + (size_t)rr * kRowBytes, res, lane, nl_row, seq);
    }
  }
  cp_async_wait<0>();
  __syncwarp();
  return ok;
}

// Fold chunk c of partition r over the N staged images; publish it as lines
// of owner r (all-reduce) or write it into rank r's output (reduce-scatter).
template <int kCWarps, int kCRing>
__device__ __forceinline__ bool fold_task(const RunParams& P, uint32_t wbase, int lane, int warp,
                                          int c, int r, uint64_t e, uint64_t seq, bool to_out,
                                          uint32_t W) {
  const uint32_t t0 = (uint32_t)c * P.cp.chunk_lines;
  const uint64_t src_line =
      W ? ((uint64_t)(c % W) * P.nranks + r) * P.cp.chunk_lines : P.seg_line0[r] + t0;
  char* ag = image_bytes(P, P.AG, e, r) +
             (W ? (uint64_t)(c % W) * P.cp.chunk_lines : (uint64_t)t0) * kLL128LineBytes;
  return fold_rows<kCWarps, kCRing>(P, wbase, lane, warp, r, t0, chunk_lines_of(P, r, t0),
                                    src_line, ag, e, seq, to_out);
}

template <int kCWarps, int kCRing>
__device__ __forceinline__ bool gather_task(const RunParams& P, const Piece* pc, uint32_t wbase,
                                            int lane, int warp, int rsh, uint64_t e) {
  const int n = P.nranks;
  const int li = lane >> 3;
  // output chunk q = lane: its two payload granules in the row
  const int q = lane < 30 ? lane : 29;
  const uint32_t g0off = 128 * ((2 * q) / 15) + 8 * ((2 * q) % 15);
  const uint32_t g1off = 128 * ((2 * q + 1) / 15) + 8 * ((2 * q + 1) % 15);
  const int rmask = (1 << rsh) - 1;
  const int nrows = n << rsh;
  const int nj = warp < nrows ? (nrows - warp + kCWarps - 1) / kCWarps : 0;
  const uint64_t pol = l2_evict_first_policy();  // outputs are written once
  auto issue = [&](int j) {
    if (j < nj) {
      const int i = warp + j * kCWarps, r = i >> rsh, rr = i & rmask;
      cp_async16(wbase + (j % kCRing) * kRowBytes + 16 * lane,
                 pc[r].src + (size_t)rr * kRowBytes + 16 * lane, li < pc[r].nl - 4 * rr);
    }
    cp_async_commit();
  };
#pragma unroll 1
  for (int j = 0; j < kCRing; ++j) issue(j);
  bool ok = true;
  for (int j = 0; j < nj; ++j) {
    cp_async_wait<kCRing - 1>();
    __syncwarp();
    const uint32_t row = wbase + (j % kCRing) * kRowBytes;
    const int i = warp + j * kCWarps, r = i >> rsh, rr = i & rmask;
    const int nl_row = pc[r].nl - 4 * rr;
    const bool valid = li < nl_row;
    const bool ready = !(valid && (lane & 7) == 7) || lds_u64(row + 16 * lane + 8) == e;
    if (!__all_sync(0xFFFFFFFFu, ready)) {
      const char* grow = pc[r].src + (size_t)rr * kRowBytes;
      ok = ll128_wait_chunk(P, grow, lane, ready, e, r, (int64_t)rr * kLL128RowLines);
      if (!ok) break;
      if (valid) sts_v4(row + 16 * lane, ld_v4(grow + 16 * lane));
      __syncwarp();
    }
    const uint2 a = lds_v2(row + g0off), b = lds_v2(row + g1off);
    __syncwarp();  // every lane read the slot before it is refilled
    issue(j + kCRing);
    const int left = pc[r].left - rr * kRowElems;
    if (nl_row > 0 && lane < 30 && 8 * lane < left)
      st_v4_hint(pc[r].dst + (size_t)rr * (2 * kRowElems) + 16 * lane,
                 make_uint4(a.x, a.y, b.x, b.y), pol);
  }
  cp_async_wait<0>();
  __syncwarp();
  return ok;
}

// Counts one finished gather of chunk c in this epoch; true for the N-th.
// Called by one thread after its CTA's reads of the chunk completed.
__device__ __forceinline__ bool last_gather(const RunParams& P, int c, uint64_t e, bool release) {
  unsigned long long* cnt = reinterpret_cast<unsigned long long*>(P.cp.gather_cnt + c);
  // cycling staging: the count frees the published slot, so the CTA's reads
  // of the chunk must come before it
  if (release) fence_acq_rel_gpu();
  unsigned long long old = ld_relaxed_u64(cnt), want;
  for (;;) {
    want = (old >> 8) == e ? old + 1 : ((e << 8) | 1ull);
    const unsigned long long seen = atomicCAS(cnt, old, want);
    if (seen == old) break;
    old = seen;
  }
  return (int)(want & 0xFFull) == P.nranks;
}

// Thread 0 waits (bounded) until all N gathers of chunk c finished in this
// epoch, then fences (acquire); the caller's __syncthreads hands the order
// to the CTA.  Cycling staging: the fold that reuses the chunk's published
// slot waits for this.
__device__ __forceinline__ bool acquire_gathers(const RunParams& P, int c, uint64_t e) {
  bool ok = true;
  if (threadIdx.x == 0) {
    const uint64_t want = (e << 8) | (uint64_t)P.nranks;
    const uint64_t* cnt = P.cp.gather_cnt + c;
    if (ld_relaxed_u64(cnt) != want) {
      Waiter w;
      while (ld_relaxed_u64(cnt) != want) {
        if (w.expired(P.ws, P.timeout_ns)) {
          latch_error(P.ws, kStatusTimeout, 0xFFFFFFFFu, -5);
          ok = false;
          break;
        }
        __nanosleep(64);
      }
    }
    fence_acq_rel_gpu();
  }
  return ok;
}

// kCycle: the staging images cycle through P.cp.ring chunk slots (a
// separate instantiation, so the default launch carries none of it)
template <int kCWarps, int kCRing, int kMinBlocks, bool kCycle>
__global__ void __launch_bounds__(kCWarps * 32, kMinBlocks) k_composed_ll128(RunParams P) {
  extern __shared__ __align__(128) char smem[];
  __shared__ Piece s_piece[kMaxRanks];
  __shared__ int s_task[2];
  __shared__ int s_ok;
  const uint64_t e = begin_run(P);
  const ComposedParams& Q = P.cp;
  WsHeader* h = header(P.ws);
  const int n = P.nranks;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int slot = (int)(e & 1);
  // all-reduce: stage, fold + publish, gather; reduce-scatter: stage, fold
  // into the outputs; all-to-all: stage, copy into the outputs
  const int kinds = Q.mode == 0 ? 3 : 2;
  const int per_step = kinds * n;
  const int ntasks = ((int)Q.nchunks + Q.lag + (kinds == 3 ? Q.lag2 : 0)) * per_step;
  const int rsh = __ffs((int)Q.chunk_lines / kLL128RowLines) - 1;  // rows per chunk = 2^rsh
  const uint32_t wbase =
      (uint32_t)__cvta_generic_to_shared(smem) + (uint32_t)(warp * kCRing * kRowBytes);
  if (threadIdx.x == 0) {
    s_task[0] = (int)atomicAdd(&h->task_next[slot], 1u);
    s_ok = 1;
  }
  __syncthreads();
  // Barriers per task: two.  The first publishes the task's descriptors or
  // its acquired flags; the second ends the task's reads and writes (and
  // publishes the next task index and s_ok, written before it).
  for (int it = 0;; ++it) {
    const int t = s_task[it & 1];
    if (t >= ntasks) break;
    // take the next task now; it is needed only after this one
    if (threadIdx.x == 0)
      s_task[(it + 1) & 1] = aborted(P.ws) ? ntasks : (int)atomicAdd(&h->task_next[slot], 1u);
    const int step = t / per_step, rem = t % per_step;
    const int kind = rem / n, x = rem % n;
    const int c = step - (kind == 0 ? 0 : (kind == 1 ? Q.lag : Q.lag + Q.lag2));
    if (c < 0 || c >= (int)Q.nchunks) {
      __syncthreads();
      continue;
    }
    // cycling staging: chunk c's lines carry e + c, and its chunk slot was
    // last used by chunk c - W, whose readers must be done with it
    const uint32_t W = kCycle ? Q.ring : 0u;
    const uint64_t seq = W ? e + (uint64_t)c : e;
    const bool reuse = W && c >= (int)W;
    if (kind == 0) {
      if (Q.mode == 3) {
        if (threadIdx.x == 0) fill_ag_stage_piece(P, s_piece, c, x, e);
      } else if ((int)threadIdx.x < n) {
        fill_stage_piece(P, s_piece, c, x, e, W);
      }
      if (reuse && !acquire_flags(P, Q.flag_fold + (size_t)(c - (int)W) * n, n, e))
        s_ok = 0;
      __syncthreads();
      if (!s_ok) break;
      stage_task<kCWarps, kCRing>(s_piece, wbase, lane, warp, Q.mode == 3 ? 1 : n, rsh, seq);
      release_flag(Q.flag_stage + (size_t)c * n + x, e, s_ok);
    } else if (kind == 1 && (Q.mode == 0 || Q.mode == 1)) {
      if (!acquire_flags(P, Q.flag_stage + (size_t)c * n, n, e)) s_ok = 0;
      if (reuse && Q.mode == 0 && !acquire_gathers(P, c - (int)W, e)) s_ok = 0;
      __syncthreads();
      if (!s_ok) break;
      if (!fold_task<kCWarps, kCRing>(P, wbase, lane, warp, c, x, e, seq, Q.mode == 1, W))
        s_ok = 0;
      release_flag(Q.flag_fold + (size_t)c * n + x, e, s_ok);
    } else if (kind == 1 && Q.mode == 3) {
      // all-gather: chunk c of every source's segment into rank x's output;
      // the N-th copy of a chunk drops its staged lines from L2
      if ((int)threadIdx.x < n) fill_ag_copy_piece(P, s_piece, c, x, e);
      if (!acquire_flags(P, Q.flag_stage + (size_t)c * n, n, e)) s_ok = 0;
      __syncthreads();
      if (!s_ok) break;
      if (!gather_task<kCWarps, kCRing>(P, s_piece, wbase, lane, warp, rsh, seq)) s_ok = 0;
      __syncthreads();
      if (warp == 0 && s_ok && Q.discard == 1) {
        // warp 0 alone, as for the all-reduce's gathers
        const bool last =
            __shfl_sync(0xFFFFFFFFu, lane == 0 ? (int)last_gather(P, c, e, false) : 0, 0);
        if (last)
          for (int r = 0; r < n; ++r) {
            const int nl = s_piece[r].nl;
            for (int j = lane; j < nl; j += 32)
              discard_l2_line(s_piece[r].src + (size_t)j * kLL128LineBytes);
          }
      }
    } else if (kind == 1) {
      // all-to-all: segment x of every source's chunk c into rank x's output;
      // each staged line has this one reader, which drops it once copied
      if ((int)threadIdx.x < n) fill_a2a_piece(P, s_piece, c, x, e, W);
      if (!acquire_flags(P, Q.flag_stage + (size_t)c * n, n, e)) s_ok = 0;
      __syncthreads();
      if (!s_ok) break;
      if (!gather_task<kCWarps, kCRing>(P, s_piece, wbase, lane, warp, rsh, seq)) s_ok = 0;
      __syncthreads();
      if (s_ok && Q.discard)
        for (int r = 0; r < n; ++r) {
          const int nl = s_piece[r].nl;
          for (int j = threadIdx.x; j < nl; j += blockDim.x)
            discard_l2_line(s_piece[r].src + (size_t)j * kLL128LineBytes);
        }
      // cycling staging: the copy's completion (a stage reusing the chunk
      // slot waits for it); either barrier keeps s_piece until every thread
      // is done with it
      if (W)
        release_flag(Q.flag_fold + (size_t)c * n + x, e, s_ok);
      else
        __syncthreads();
    } else {
      if ((int)threadIdx.x < n) fill_gather_piece(P, s_piece, c, x, e, W);
      if (!acquire_flags(P, Q.flag_fold + (size_t)c * n, n, e)) s_ok = 0;
      __syncthreads();
      if (!s_ok) break;
      if (!gather_task<kCWarps, kCRing>(P, s_piece, wbase, lane, warp, rsh, seq)) s_ok = 0;
      __syncthreads();
      if (warp == 0 && s_ok && (Q.discard == 1 || W)) {
        // warp 0 alone: it also fills the next task's descriptors, so it
        // is done with these before anyone reads the next ones
        // with cycling staging the count frees the published slot for the fold
        // of chunk c + W, so a discard after it could drop that fold's lines:
        // published lines are then left in place to be overwritten
        const bool last = __shfl_sync(0xFFFFFFFFu, lane == 0 ? (int)last_gather(P, c, e, W != 0) : 0, 0);
        if (last && Q.discard == 1 && !W)
          for (int r = 0; r < n; ++r) {
            const int nl = s_piece[r].nl;
            for (int j = lane; j < nl; j += 32)
              discard_l2_line(s_piece[r].src + (size_t)j * kLL128LineBytes);
          }
      }
    }
    if (!s_ok) break;
  }
  finish_run(P, e);
}

template <int W, int R, int B, bool C>
static int capacity_of() {
  static size_t memo[kMaxDevices];
  const int bytes = (int)((size_t)W * R * kRowBytes);
  if (raise_smem_limit(k_composed_ll128<W, R, B, C>, (size_t)bytes, memo) != cudaSuccess) return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_composed_ll128<W, R, B, C>, W * 32,
                                                    bytes) != cudaSuccess)
    return 0;
  return per_sm * device_sms();
}

int composed_capacity(int variant, bool cycle) {
  if (cycle) {
    if (variant == 1) return capacity_of<8, 24, 2, true>();
    if (variant == 2) return capacity_of<4, 16, 6, true>();
    return capacity_of<8, 16, 3, true>();
  }
  if (variant == 1) return capacity_of<8, 24, 2, false>();
  if (variant == 2) return capacity_of<4, 16, 6, false>();
  return capacity_of<8, 16, 3, false>();
}

cudaError_t launch_composed(const RunParams& P, int grid, cudaStream_t s) {
  const int v = P.cp.variant;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCVariants[v].warps * 32);
  cfg.dynamicSmemBytes = composed_smem_bytes(v);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (P.cp.ring > 0) {
    if (v == 1) return cudaLaunchKernelEx(&cfg, k_composed_ll128<8, 24, 2, true>, P);
    if (v == 2) return cudaLaunchKernelEx(&cfg, k_composed_ll128<4, 16, 6, true>, P);
    return cudaLaunchKernelEx(&cfg, k_composed_ll128<8, 16, 3, true>, P);
  }
  if (v == 1) return cudaLaunchKernelEx(&cfg, k_composed_ll128<8, 24, 2, false>, P);
  if (v == 2) return cudaLaunchKernelEx(&cfg, k_composed_ll128<4, 16, 6, false>, P);
  return cudaLaunchKernelEx(&cfg, k_composed_ll128<8, 16, 3, false>, P);
}

}  // namespace coll
