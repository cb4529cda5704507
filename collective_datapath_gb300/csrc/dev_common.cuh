// dev_common.cuh -- device helpers of the datapath kernels: memory accesses
// with explicit PTX memory-model semantics, bounded waits, bf16 conversion,
// error latching.  sm_103a only.
#pragma once

#include <cstdint>

#include "plan.h"

namespace coll {

// coll_status_t values used on the device (see coll.h).
constexpr uint32_t kStatusTimeout = 6;
// COLL_RESET_* values used on the device (see coll.h).
constexpr int kResetLastReader = 0, kResetKernel = 1, kResetNone = 2, kResetDeferred = 3;

// ---- global memory accesses ------------------------------------------------
// Readiness lines are written and polled with .relaxed.gpu accesses: they are
// morally strong at GPU scope (no data race in the PTX memory model) and
// bypass the non-coherent L1.  A vector access is a set of element accesses;
// each 8-byte element is single-copy atomic, which is what makes an LL8 line
// (4 bytes of data + its 4-byte flag in one element) self-validating.

__device__ __forceinline__ void ld_relaxed_v2u64(const void* p, uint64_t& a,
                                                 uint64_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];"
               : "=l"(a), "=l"(b)
               : "l"(p)
               : "memory");
}

__device__ __forceinline__ void st_relaxed_v2u64(void* p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a),
               "l"(b)
               : "memory");
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const void* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(void* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(void* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Acquire/release fences at GPU scope: a relaxed load followed by this fence
// is an acquire pattern; this fence followed by a relaxed store is a release
// pattern (PTX memory consistency model).
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Read-only input data: non-coherent path, no L1 allocation (streamed once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// Plain 16-byte accesses for data no other CTA of the same launch touches.
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_v2u32(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b)
               : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- bf16 <-> fp32 -----------------------------------------------------------
// Widening is exact: a bf16 pattern is the high half of a binary32 pattern.
__device__ __forceinline__ float bf16_lo_to_f32(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi_to_f32(uint32_t w) {
  return __uint_as_float(w & 0xFFFF0000u);
}

// binary32 -> bf16 with IEEE roundTiesToEven on the 16 dropped bits, written
// as the usual integer formulation: add 0x7FFF plus the lowest kept bit, then
// truncate (a carry into the exponent yields the next magnitude or Inf).
// Subnormals are kept; any NaN becomes the quiet NaN 0x7FC0.
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return f32_to_bf16_rne(lo) | (f32_to_bf16_rne(hi) << 16);
}

// Element types (values match COLL_BF16 / COLL_F32 of coll.h).  A 32-bit
// word holds two bf16 or one fp32.
constexpr int kDtBF16 = 0, kDtF32 = 1;

// An fp32 result as written: any NaN becomes the canonical quiet NaN.
__device__ __forceinline__ uint32_t f32_bits(float a) {
  return a != a ? 0x7FC00000u : __float_as_uint(a);
}

// Fold of K 32-bit words of every source as fp32, in rank order, binary32
// round-to-nearest-even, no narrowing.  w[p * K + k] = word k of source p.
template <int K>
__device__ __forceinline__ void fold_f32_words(const uint32_t* w, int n, uint32_t* out) {
  float a[K];
#pragma unroll
  for (int k = 0; k < K; ++k) a[k] = __uint_as_float(w[k]);
#pragma unroll
  for (int p = 1; p < kMaxRanks; ++p)
    if (p < n) {
#pragma unroll
      for (int k = 0; k < K; ++k) a[k] = __fadd_rn(a[k], __uint_as_float(w[p * K + k]));
    }
#pragma unroll
  for (int k = 0; k < K; ++k) out[k] = f32_bits(a[k]);
}

// ---- status -----------------------------------------------------------------

__device__ __forceinline__ WsHeader* header(char* ws) {
  return reinterpret_cast<WsHeader*>(ws);
}

// Latch the first device error (later ones are dropped) and raise `abort`
// so that every other wait of the run gives up promptly.
static __device__ __noinline__ void latch_error(char* ws, uint32_t code, uint32_t rank,
                                         int64_t line) {
  WsHeader* h = header(ws);
  if (atomicCAS(&h->status_code, 0u, code) == 0u) {
    h->status_rank = rank;
    h->status_line = line;
  }
  __threadfence();
  st_relaxed_u32(&h->abort, 1u);
}

__device__ __forceinline__ bool aborted(char* ws) {
  return ld_relaxed_u32(&header(ws)->abort) != 0u;
}

// Bounded wait bookkeeping: the first failed check starts the clock; the
// wait gives up when the bound passes, or -- checked only once the wait is
// older than 20 us, to keep the common short poll to one load -- when
// another wait of the run failed.
struct Waiter {
  uint64_t t0 = 0;
  __device__ __forceinline__ bool expired(char* ws, uint64_t timeout_ns) {
    uint64_t now = globaltimer_ns();
    if (t0 == 0) {
      t0 = now;
      return false;
    }
    const uint64_t waited = now - t0;
    return waited > timeout_ns || (waited > 20000 && aborted(ws));
  }
};

// One atomic per warp for the stale lines its active lanes observed.
__device__ __forceinline__ void count_rejection(char* ws) {
  const unsigned mask = __activemask();
  const int leader = __ffs(mask) - 1;
  if ((int)(threadIdx.x & 31) == leader)
    atomicAdd(reinterpret_cast<unsigned long long*>(&header(ws)->rejections),
              (unsigned long long)__popc(mask));
}

// Epoch protocol of a launch.  Thread 0 of each CTA reads the device epoch
// and hands it to the CTA in shared memory: a read by every warp of every CTA
// at the same moment queues on one L2 line, on the critical path of a short
// run.  In the launch that ends a run each CTA then adds one to `arrived`
// once all its threads hold the value (the barrier's predicate consumes it).
// The last CTA of the grid advances the epoch once every CTA has arrived, so
// the next run uses the other staging slot; no CTA waits at the end of its
// own work.  run_arrive (the first use of the epoch) lets a dependent launch
// place its CTAs and counts this CTA in; a kernel that issues loads of its
// own while the epoch is in flight calls it after its own read.
__device__ __forceinline__ void run_arrive(const RunParams& P, uint64_t e) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (P.advance_epoch) {
    const int z = __syncthreads_or((int)(e >> 63));  // 0: the epoch never gets there
    if (threadIdx.x == 0)
      asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(&header(P.ws)->arrived),
                   "r"(1u + (uint32_t)z)
                   : "memory");
  }
}

__device__ __forceinline__ uint64_t begin_run(const RunParams& P) {
  __shared__ uint64_t s_run_epoch;
  // Under programmatic stream serialization the CTAs may start before the
  // previous kernel in the stream has completed: wait for it (and for its
  // writes) before reading anything; without that launch attribute the wait
  // returns at once.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) s_run_epoch = ld_relaxed_u64(&header(P.ws)->epoch);
  __syncthreads();
  const uint64_t e = s_run_epoch;
  run_arrive(P, e);
  return e;
}

// begin_run with every thread reading the epoch itself (one L2 request per
// warp).  The column-scheduled composed kernel keeps this form: its DRAM
// counters were measured with it.  The shared-memory form above took an
// 8 x 1 MiB composed all-reduce from 9.69 to 9.30 us on the same GPU, but
// that kernel has not been profiled with it.
__device__ __forceinline__ uint64_t begin_run_per_thread(const RunParams& P) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint64_t e = ld_relaxed_u64(&header(P.ws)->epoch);
  run_arrive(P, e);
  return e;
}

// The arrival count as the grid's last CTA sees it early (before its last
// phase of work), so that finish_run usually need not read it again; other
// CTAs, and launches that do not end a run, get 0.
__device__ __forceinline__ uint32_t early_arrivals(const RunParams& P) {
  if (!P.advance_epoch || threadIdx.x != 0 || blockIdx.x != gridDim.x - 1) return 0;
  return ld_relaxed_u32(&header(P.ws)->arrived);
}

// `seen`: an arrival count this CTA read earlier (early_arrivals), or 0.
__device__ __forceinline__ void finish_run(const RunParams& P, uint64_t epoch,
                                           uint32_t seen = 0) {
  if (!P.advance_epoch || threadIdx.x != 0) return;
  const uint32_t total = gridDim.x * gridDim.y * gridDim.z;
  if (blockIdx.x != gridDim.x - 1) return;
  WsHeader* h = header(P.ws);
  // Every CTA has started (and read the epoch) long before the last CTA
  // finishes; the 10 s bound only guards against a broken launch.  This wait
  // ignores `abort`: the epoch must not move before every CTA has read it.
  const uint64_t t0 = globaltimer_ns();
  while (seen < total && ld_relaxed_u32(&h->arrived) < total) {
    if (globaltimer_ns() - t0 > 10000000000ull) {
      latch_error(P.ws, kStatusTimeout, 0xFFFFFFFFu, -2);
      break;
    }
    __nanosleep(100);
  }
  st_relaxed_u32(&h->arrived, 0u);
  // the next run's counters
  st_relaxed_u32(&h->started[(epoch + 1) & 1], 0u);
  st_relaxed_u32(&h->task_next[(epoch + 1) & 1], 0u);
  st_relaxed_u64(&h->epoch, epoch + (uint64_t)P.advance_epoch);
}

}  // namespace coll
