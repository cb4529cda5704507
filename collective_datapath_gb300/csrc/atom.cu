// atom.cu -- the one-sided copy primitive with an explicit pipeline depth.
//
// Purlin (Separating Orchestration from the Datapath of Collectives) §3.3
// sizes a datapath by the bytes it keeps in flight: C transfer CTAs, each with
// S pipeline stages of B_stage bytes, give a capacity Q_cap = C * S * B_stage
// (Eq. (3)); by Little's law the copy reaches the link's bandwidth only once
// Q_cap covers bandwidth x latency.  Its copy ablation (§5.2, Figure 9)
// holds C and the message fixed and raises S from 1 to 8.  On one GB300 the
// two ends of the copy are both in this GPU's HBM, so the "link" is HBM
// itself; pull and push coincide (the same CTAs read and write the same
// memory) and the two arms here are instead the two load engines of the SM:
//
//   ATOM_BULK: a ring of S shared-memory stages driven with untiled TMA
//     copies.  One producer thread issues a bulk load of B_stage bytes into
//     a stage (completion counted on the stage's "full" mbarrier); two store
//     threads, each owning alternate stages, issue the bulk store of a full
//     stage and release it on its "empty" mbarrier once the store has read
//     it out.
//     Up to S loads are in flight and two stores can be queued at once.
//   ATOM_LSU: all 256 threads keep S stages of cp.async 16-byte granules in
//     flight (thread t owns granules t, t + 256, ... of every stage, so the
//     ring is thread-private and needs no barrier), then store each granule
//     from registers.
//
// Chunk c of the message (B_stage bytes, the last one shorter) goes to CTA
// c mod C; every wait on an mbarrier is bounded and reports a timeout in the
// caller's status word.
#include <cuda_runtime.h>

#include "../../include/coll.h"
#include "launch.h"
#include "pipe.cuh"
#include "tma.cuh"

namespace coll {

constexpr int kAtomThreads = 256;
constexpr uint64_t kAtomWaitNs = 1000000000ull;  // per stage: far above any HBM latency
constexpr int kAtomStoreWarps = 2;                // bulk engine: threads issuing stores

struct AtomArgs {
  char* dst;
  const char* src;
  uint64_t bytes;
  uint32_t stage_bytes;
  int32_t* status;  // may be null
};

__device__ __forceinline__ uint32_t atom_chunk_len(const AtomArgs& a, uint64_t c) {
  const uint64_t off = c * a.stage_bytes;
  const uint64_t left = a.bytes - off;
  return left < a.stage_bytes ? (uint32_t)left : a.stage_bytes;
}

template <int S>
__global__ void __launch_bounds__(kAtomThreads) k_atom_bulk(AtomArgs a) {
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t full[S], empty[S];
  const int warp = threadIdx.x >> 5;
  const uint32_t sbuf = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t sfull = (uint32_t)__cvta_generic_to_shared(full);
  const uint32_t sempty = (uint32_t)__cvta_generic_to_shared(empty);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) {
      mbar_init(sfull + 8 * s, 1);
      mbar_init(sempty + 8 * s, 1);
    }
    fence_mbarrier_init();
  }
  __syncthreads();  // every thread is still here: the barriers are set up
  if ((threadIdx.x & 31) != 0 || warp > kAtomStoreWarps) return;
  const uint64_t nchunks = (a.bytes + a.stage_bytes - 1) / a.stage_bytes;
  const uint64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nj = first < nchunks ? (int64_t)((nchunks - first + stride - 1) / stride) : 0;
  if (warp == 0) {
    // producer: chunk j goes to slot j mod S once the store of chunk j - S
    // has read that slot out (phase (j / S - 1) of its empty barrier)
    int64_t j = 0;
    uint32_t slot = 0, round = 0;  // j = round * S + slot
    for (; j < nj; ++j) {
      if (round > 0 &&
          !mbar_wait_bounded(sempty + 8 * slot, (round - 1) & 1, kAtomWaitNs)) {
        if (a.status) atomicExch(a.status, (int32_t)kStatusTimeout);
        break;
      }
      const uint64_t c = first + (uint64_t)j * stride;
      const uint32_t len = atom_chunk_len(a, c);
      mbar_expect_tx(sfull + 8 * slot, len);
      tma_load_1d(sbuf + slot * a.stage_bytes, a.src + c * a.stage_bytes, len, sfull + 8 * slot);
      if (++slot == S) {
        slot = 0;
        ++round;
      }
    }
    // every load issued must have landed before the CTA may retire (bounded)
    for (int64_t k = j > S ? j - S : 0; k < j; ++k)
      mbar_wait_bounded(sfull + 8 * (uint32_t)(k % S), (uint32_t)((k / S) & 1), kAtomWaitNs);
  } else {
    // store thread w owns the slots s with s mod kAtomStoreWarps = w - 1 and
    // takes their chunks in order, so it has seen every earlier phase of a
    // slot's full barrier before it waits on the next one (a parity wait
    // can only tell apart adjacent phases); two stores can be queued while
    // each slot is released as soon as it is read out
    uint32_t slot = 0, round = 0;  // j = round * S + slot
    for (int64_t j = 0; j < nj; ++j) {
      if ((int)(slot % kAtomStoreWarps) == warp - 1) {
        if (!mbar_wait_bounded(sfull + 8 * slot, round & 1, kAtomWaitNs)) {
          if (a.status) atomicExch(a.status, (int32_t)kStatusTimeout);
          break;
        }
        const uint64_t c = first + (uint64_t)j * stride;
        tma_store_1d(a.dst + c * a.stage_bytes, sbuf + slot * a.stage_bytes,
                     atom_chunk_len(a, c));
        bulk_commit();
        bulk_wait_read<0>();
        mbar_arrive(sempty + 8 * slot);
      }
      if (++slot == S) {
        slot = 0;
        ++round;
      }
    }
    bulk_wait<0>();
  }
}

template <int S>
__global__ void __launch_bounds__(kAtomThreads) k_atom_lsu(AtomArgs a) {
  extern __shared__ __align__(128) char smem[];
  const uint32_t sbuf = (uint32_t)__cvta_generic_to_shared(smem);
  const uint64_t nchunks = (a.bytes + a.stage_bytes - 1) / a.stage_bytes;
  const uint64_t first = blockIdx.x, stride = gridDim.x;
  const int64_t nj = first < nchunks ? (int64_t)((nchunks - first + stride - 1) / stride) : 0;
  const uint32_t granules = a.stage_bytes / 16;
  const uint32_t t = threadIdx.x;
  // chunk j of this CTA sits in stage j mod S; `slot` follows it without a
  // 64-bit division
  auto issue = [&](int64_t j, uint32_t slot) {
    if (j < nj) {
      const uint64_t c = first + (uint64_t)j * stride;
      const uint32_t len = atom_chunk_len(a, c);
      const uint32_t base = sbuf + slot * a.stage_bytes;
      for (uint32_t g = t; g < granules; g += kAtomThreads) {
        const bool valid = 16 * g < len;
        cp_async16(base + 16 * g, valid ? a.src + c * a.stage_bytes + 16 * g : a.src, valid);
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int j = 0; j < S; ++j) issue(j, (uint32_t)j);
  uint32_t slot = 0;
  for (int64_t j = 0; j < nj; ++j) {
    cp_async_wait<S - 1>();
    const uint64_t c = first + (uint64_t)j * stride;
    const uint32_t len = atom_chunk_len(a, c);
    const uint32_t base = sbuf + slot * a.stage_bytes;
    for (uint32_t g = t; g < granules && 16 * g < len; g += kAtomThreads)
      st_v4(a.dst + c * a.stage_bytes + 16 * g, lds_v4(base + 16 * g));
    issue(j + S, slot);  // the granules just stored were this thread's own
    if (++slot == S) slot = 0;
  }
  cp_async_wait<0>();
}

template <int S>
static cudaError_t launch_atom_s(const AtomArgs& a, int engine, int ctas, cudaStream_t st) {
  const size_t smem = (size_t)S * a.stage_bytes;
  static size_t memo[2][kMaxDevices];
  auto* fn = engine == 0 ? k_atom_bulk<S> : k_atom_lsu<S>;
  if (cudaError_t err = raise_smem_limit(fn, (size_t)kAtomMaxSmem, memo[engine])) return err;
  fn<<<ctas, kAtomThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_atom_copy(void* dst, const void* src, uint64_t bytes, int engine, int ctas,
                             int stages, uint32_t stage_bytes, int32_t* status,
                             cudaStream_t st) {
  const AtomArgs a{(char*)dst, (const char*)src, bytes, stage_bytes, status};
  switch (stages) {
    case 1: return launch_atom_s<1>(a, engine, ctas, st);
    case 2: return launch_atom_s<2>(a, engine, ctas, st);
    case 3: return launch_atom_s<3>(a, engine, ctas, st);
    case 4: return launch_atom_s<4>(a, engine, ctas, st);
    case 5: return launch_atom_s<5>(a, engine, ctas, st);
    case 6: return launch_atom_s<6>(a, engine, ctas, st);
    case 7: return launch_atom_s<7>(a, engine, ctas, st);
    case 8: return launch_atom_s<8>(a, engine, ctas, st);
    default: return cudaErrorInvalidValue;
  }
}

// Copy ceiling probe: `passes` full copies of src -> dst in one launch with
// grid-stride 16-byte accesses (loads cached in L2 only), so that buffers
// that fit L2 measure the SM <-> L2 copy throughput with no launch gaps
// between passes.
__global__ void __launch_bounds__(256) k_copy_passes(uint4* dst, const uint4* src, uint64_t n16,
                                                     int passes) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (int p = 0; p < passes; ++p)
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n16; i += stride) {
      uint4 v;
      asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                   : "l"(src + i));
      asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(dst + i), "r"(v.x),
                   "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
}

}  // namespace coll

using namespace coll;

extern "C" coll_status_t coll_copy_passes(void* dev_dst, const void* dev_src, size_t bytes,
                                          int passes, int ctas, coll_stream_t stream) {
  if (passes < 1 || passes > 65535 || ctas < 0 || ctas > 65535) return COLL_ERR_INVALID;
  if (bytes % 16 != 0) return COLL_ERR_ALIGN;
  if (bytes == 0) return COLL_OK;
  if (dev_dst == nullptr || dev_src == nullptr) return COLL_ERR_INVALID;
  const uintptr_t d = reinterpret_cast<uintptr_t>(dev_dst);
  const uintptr_t s = reinterpret_cast<uintptr_t>(dev_src);
  if ((d | s) & 15u) return COLL_ERR_ALIGN;
  if (d < s + bytes && s < d + bytes) return COLL_ERR_INVALID;  // overlapping ranges
  if (ctas == 0) ctas = 8 * device_sms();
  k_copy_passes<<<ctas, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(dev_dst), static_cast<const uint4*>(dev_src), bytes / 16, passes);
  return cudaGetLastError() == cudaSuccess ? COLL_OK : COLL_ERR_CUDA;
}

extern "C" coll_status_t coll_atom_copy(void* dev_dst, const void* dev_src, size_t bytes,
                                        int engine, int ctas, int stages, int stage_bytes,
                                        int32_t* dev_status, coll_stream_t stream) {
  if (engine != COLL_ATOM_BULK && engine != COLL_ATOM_LSU) return COLL_ERR_INVALID;
  if (stages < 1 || stages > kAtomMaxStages || stage_bytes < 16 ||
      (size_t)stages * (size_t)stage_bytes > (size_t)kAtomMaxSmem || ctas < 0 || ctas > 65535)
    return COLL_ERR_INVALID;
  if (stage_bytes % 16 != 0 || bytes % 16 != 0) return COLL_ERR_ALIGN;
  if (bytes == 0) return COLL_OK;
  if (dev_dst == nullptr || dev_src == nullptr) return COLL_ERR_INVALID;
  const uintptr_t d = reinterpret_cast<uintptr_t>(dev_dst);
  const uintptr_t s = reinterpret_cast<uintptr_t>(dev_src);
  if ((d | s) & 15u) return COLL_ERR_ALIGN;
  if (d < s + bytes && s < d + bytes) return COLL_ERR_INVALID;  // overlapping ranges
  if (ctas == 0) ctas = device_sms();
  const cudaError_t err =
      launch_atom_copy(dev_dst, dev_src, bytes, engine, ctas, stages, (uint32_t)stage_bytes,
                       dev_status, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? COLL_OK : COLL_ERR_CUDA;
}
