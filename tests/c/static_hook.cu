// static_hook.cu -- test-only build of the allocation-free all-reduce.
//
// The library's coll_allreduce_static keeps its scratch (and the status and
// abort words of its header) in a file-scope device array that no other
// translation unit can name.  To test that a call recovers from an abort
// that an earlier call left latched, the test compiles that same source
// file into a separate library together with the two functions below, which
// read and plant header words of this build's own array.  The product
// library carries no such hook.
#include "../../collective_datapath_gb300/csrc/static_ws.cu"

namespace {

int hook_header(coll::DeviceScratch** ds) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= coll::kMaxDevices) return -1;
  return coll::static_setup(dev, ds) == COLL_OK ? 0 : -1;
}

}  // namespace

// Latch a device error as a timed-out wait would: status {code, rank, line}
// and abort = 1.  Synchronous; returns 0 on success.
extern "C" int static_hook_latch(uint32_t code, uint32_t rank, int64_t line) {
  coll::DeviceScratch* ds = nullptr;
  if (hook_header(&ds) != 0) return -1;
  coll::WsHeader h;
  if (cudaMemcpy(&h, ds->ptr, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  h.status_code = code;
  h.status_rank = rank;
  h.status_line = line;
  h.abort = 1u;
  return cudaMemcpy(ds->ptr, &h, sizeof h, cudaMemcpyHostToDevice) == cudaSuccess ? 0 : -1;
}

// Read the header's epoch, status code and abort word.  Synchronous.
extern "C" int static_hook_read(uint64_t* epoch, uint32_t* code, uint32_t* abort_word) {
  coll::DeviceScratch* ds = nullptr;
  if (hook_header(&ds) != 0) return -1;
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  coll::WsHeader h;
  if (cudaMemcpy(&h, ds->ptr, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
  *epoch = h.epoch;
  *code = h.status_code;
  *abort_word = h.abort;
  return 0;
}
