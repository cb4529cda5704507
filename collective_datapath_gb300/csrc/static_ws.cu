// static_ws.cu -- an all-reduce entry point that allocates nothing.
//
// Every other entry point works in a workspace the caller allocates and binds.
// Some callers cannot allocate device memory at the moment they need a
// collective: code running where cudaMalloc is forbidden or unsafe (inside a
// stream capture that must not allocate, inside an allocator's own callback,
// or in a process whose device memory is fully reserved by another runtime).
// For them coll_allreduce_static runs the oneshot LL8 all-reduce (the same
// stage / validate / rank-order fold as the fused path) in a fixed scratch
// array that lives in this file, so no call allocates or frees anything.
//
// The scratch is a file-scope __device__ array: every GPU that loads this
// library holds it (kStaticBytes) until the process exits.  Host code must
// not use the array's name as a device address; set-up obtains the address
// with cudaGetSymbolAddress once per device, with that device current.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstddef>
#include <mutex>

#include "../../include/coll.h"
#include "launch.h"
#include "ll8.cuh"

namespace coll {
namespace {

constexpr size_t kStaticHeaderBytes = 4096;
// nranks * count may not exceed this many bf16 elements (2 MiB of input).
constexpr size_t kStaticMaxElems = size_t(1) << 20;
// Header + two LL8 slots (8 bytes of lines per 2 elements, so 4 bytes per
// element per slot) of every rank's image: 8 MiB + 4 KiB.
constexpr size_t kStaticBytes = kStaticHeaderBytes + 2 * kStaticMaxElems * 4;
constexpr int kStaticThreads = 256;
constexpr uint32_t kStaticTileLines = 4 * kStaticThreads;  // one LL8 group per thread

static __device__ __align__(256) char g_static_scratch[kStaticBytes];

// CTA (d, b) of the cooperative grid serves emulated rank d: it stages tiles
// b, b + B, ... of rank d's input, then folds the same tiles of every rank
// into rank d's output.  Waits are bounded; lines of earlier calls carry
// older epochs and are never accepted.
__global__ void __launch_bounds__(kStaticThreads)
    k_allreduce_static(RunParams P, uint32_t rank_lines) {
  const uint64_t e = begin_run(P);
  const int B = P.ctas_per_rank;
  const int d = blockIdx.x / B, b = blockIdx.x % B;
  for (uint32_t t0 = b * kStaticTileLines; t0 < rank_lines; t0 += B * kStaticTileLines) {
    StageItem it{};
    it.rank = (uint16_t)d;
    it.nlines = min(kStaticTileLines, rank_lines - t0);
    it.nelems = it.nlines * kLL8Elems;
    it.dst_line = t0;
    it.in_elem = (uint64_t)t0 * kLL8Elems;
    ll8_stage_tile(P, it, e);
  }
  for (uint32_t t0 = b * kStaticTileLines; t0 < rank_lines; t0 += B * kStaticTileLines) {
    if (aborted(P.ws)) break;
    Item it{};
    it.kind = IK_REDUCE;
    it.dst = (uint8_t)d;
    it.nlines = min(kStaticTileLines, rank_lines - t0);
    it.nelems = it.nlines * kLL8Elems;
    it.src_line = t0;
    it.out_off = (uint64_t)t0 * kLL8Elems;
    ll8_consume_item(P, P.P, it, e);
  }
  finish_run(P, e);
}

struct DeviceScratch {
  char* ptr = nullptr;
  int sms = 0;
};

std::mutex g_setup_mutex;
DeviceScratch g_devices[kMaxDevices];

// Set-up, once per device with that device current: the device address of
// the scratch array, a cleared header, and the first epoch (1).
coll_status_t static_setup(int dev, DeviceScratch** out) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceScratch& ds = g_devices[dev];
  if (ds.ptr == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) return COLL_ERR_CUDA;
    if (cudaMemset(ptr, 0, kStaticHeaderBytes) != cudaSuccess) return COLL_ERR_CUDA;
    const uint64_t first_epoch = 1;
    if (cudaMemcpy(ptr, &first_epoch, sizeof first_epoch, cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return COLL_ERR_CUDA;
    if (cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return COLL_ERR_CUDA;
    ds.ptr = static_cast<char*>(ptr);
  }
  *out = &ds;
  return COLL_OK;
}

}  // namespace
}  // namespace coll

using namespace coll;

extern "C" coll_status_t coll_allreduce_static(int nranks, size_t count,
                                               const void* const* dev_ins,
                                               void* const* dev_outs, coll_stream_t stream) {
  if (nranks < 1 || nranks > kMaxRanks || dev_ins == nullptr || dev_outs == nullptr)
    return COLL_ERR_INVALID;
  if (count % 8 != 0) return COLL_ERR_ALIGN;
  if ((size_t)nranks * count > kStaticMaxElems) return COLL_ERR_NOMEM;
  for (int r = 0; r < nranks; ++r) {
    if (count > 0 && (dev_ins[r] == nullptr || dev_outs[r] == nullptr)) return COLL_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(dev_ins[r]) & 15u) ||
        (reinterpret_cast<uintptr_t>(dev_outs[r]) & 15u))
      return COLL_ERR_ALIGN;
  }
  if (count == 0) return COLL_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return COLL_ERR_CUDA;
  DeviceScratch* ds = nullptr;
  if (coll_status_t st = static_setup(dev, &ds)) return st;

  const uint32_t rank_lines = (uint32_t)(count / kLL8Elems);
  const int tiles = (int)((rank_lines + kStaticTileLines - 1) / kStaticTileLines);
  const int B = std::max(1, std::min(tiles, ds->sms / nranks));
  RunParams P{};
  P.ws = ds->ptr;
  for (int r = 0; r < nranks; ++r) {
    P.in[r] = static_cast<const uint16_t*>(dev_ins[r]);
    P.out[r] = static_cast<uint16_t*>(dev_outs[r]);
  }
  P.nranks = nranks;
  P.enc = ENC_LL8;
  P.dtype = kDtBF16;
  P.reset_mode = kResetNone;
  P.ctas_per_rank = B;
  P.timeout_ns = 200000000ull;
  P.P.base = kStaticHeaderBytes;
  P.P.rank_bytes = (uint64_t)rank_lines * kLL8LineBytes;
  P.P.slot_bytes = P.P.rank_bytes * (uint64_t)nranks;
  P.P.slot_mask = 1;
  P.stage_rank = -1;
  P.advance_epoch = 1;

  // A device-side timeout latches the status words and raises `abort` in
  // the shared header, and an abort left standing would make every later
  // call skip its fold.  So every call starts by clearing those words, in
  // stream order ahead of its own launch; the status of an earlier call that
  // timed out is dropped with them.
  constexpr size_t kErrBegin = offsetof(WsHeader, status_code);
  constexpr size_t kErrEnd = offsetof(WsHeader, abort) + sizeof(uint32_t);
  static_assert(kErrEnd - kErrBegin == 20, "status code, rank, line and abort are contiguous");
  if (cudaMemsetAsync(ds->ptr + kErrBegin, 0, kErrEnd - kErrBegin,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return COLL_ERR_CUDA;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nranks * B);
  cfg.blockDim = dim3(kStaticThreads);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_allreduce_static, P, rank_lines) == cudaSuccess
             ? COLL_OK
             : COLL_ERR_CUDA;
}
