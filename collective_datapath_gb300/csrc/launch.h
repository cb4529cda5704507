// launch.h -- host-side launchers of the datapath kernels (kernels.cu).
#pragma once

#include <cuda_runtime.h>

#include "plan.h"

namespace coll {

// Device ordinals a process can drive; per-device host caches are this long.
constexpr int kMaxDevices = 64;
// The device current on the calling host thread (0 if it cannot be read).
int current_device();
// SM count of the current device (cached per device).
int device_sms();
// Raise a kernel's dynamic shared-memory limit on the current device to at
// least `bytes`; `memo` (kMaxDevices entries, zero-initialised, owned by the
// caller) remembers what each device was given, so the driver call is made
// once per kernel and device.  The attribute belongs to the device that is
// current at the call, so one process driving several GPUs sets it on each.
template <typename K>
cudaError_t raise_smem_limit(K* kernel, size_t bytes, size_t* memo) {
  const int d = current_device();
  if (d >= 0 && d < kMaxDevices && memo[d] >= bytes) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && d >= 0 && d < kMaxDevices) memo[d] = bytes;
  return e;
}
int block_threads();
// Co-resident CTAs of the fused kernel on this device (0 if unknown).
int fused_capacity(int enc);

// dependent (here and below): programmatic stream serialization, as for
// launch_fused.
cudaError_t launch_stage(const RunParams& P, int grid, cudaStream_t s, bool dependent);
cudaError_t launch_consume(const RunParams& P, int phase, int grid, cudaStream_t s,
                           bool dependent);
// dependent: programmatic stream serialization (the kernel's CTAs may be
// placed before the previous kernel in the stream completes; begin_run waits
// for it before touching any data).
cudaError_t launch_fused(const RunParams& P, int grid, cudaStream_t s, bool dependent);
// An empty kernel in launch_fused's configuration (the fixed launch cost),
// or with `threads` per CTA (0 = launch_fused's block).
cudaError_t launch_floor(int grid, cudaStream_t s, bool dependent, bool cooperative = true,
                         int threads = 0);
// LL128 phase-1 folds through the shared-memory pipeline (all items IK_REDUCE).
cudaError_t launch_fold(const RunParams& P, int grid, cudaStream_t s, bool dependent);
// LL128 copy phases (all items IK_COPY, plain outputs) and LL128 staging
// through cp.async shared-memory rings.
cudaError_t launch_copy(const RunParams& P, int phase, int grid, cudaStream_t s, bool dependent);
cudaError_t launch_stage_pipe(const RunParams& P, int grid, cudaStream_t s, bool dependent);
cudaError_t launch_withhold(const RunParams& P, cudaStream_t s);
// Composed twoshot all-reduce: co-resident CTAs of the persistent kernel, and
// the launch (P.cp filled in).
int composed_capacity(int variant, bool cycle);
cudaError_t launch_composed(const RunParams& P, int grid, cudaStream_t s);
// The same collectives scheduled by columns (P.cp.schedule == 0).
int column_capacity(int variant);
int column_threads(int variant);
cudaError_t launch_column(const RunParams& P, int grid, cudaStream_t s, bool dependent);
// MoE dispatch: routing + gather-stage of one source (P.stage_rank) or all,
// then the destination scan + validated copy (ends the run).
cudaError_t launch_moe_stage_all(const RunParams& P, cudaStream_t s);
cudaError_t launch_moe_consume(const RunParams& P, cudaStream_t s);
cudaError_t launch_moe_routing(const RunParams& P, cudaStream_t s);
cudaError_t launch_moe_composed(const RunParams& P, cudaStream_t s);
// One-sided copy with an explicit pipeline (atom.cu): engine 0 = TMA bulk
// ring, 1 = cp.async ring; `stages` in 1..kAtomMaxStages of `stage_bytes`.
constexpr int kAtomMaxStages = 8;
constexpr int kAtomMaxSmem = 192 * 1024;
cudaError_t launch_atom_copy(void* dst, const void* src, uint64_t bytes, int engine, int ctas,
                             int stages, uint32_t stage_bytes, int32_t* status,
                             cudaStream_t st);
cudaError_t launch_rearm(const RunParams& P, int grid, cudaStream_t s);
cudaError_t launch_advance(const RunParams& P, cudaStream_t s);

}  // namespace coll
