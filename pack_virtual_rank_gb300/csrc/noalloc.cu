// noalloc.cu -- an allreduce entry point that allocates nothing.
//
// Some callers cannot allocate device memory at the moment they need an allreduce:
// code running inside a custom allocator or memory-pool hook (allocating would recurse
// into the allocator it is serving), a serving process that reserved all of HBM for
// its caches at start-up and must keep its footprint fixed, or a latency-critical path
// that cannot afford the device-wide synchronisation cudaMalloc and cudaFree may
// perform. relay_allreduce_noalloc serves them: the caller passes only the actives'
// input and output buffers, and the relay slots of the helpers and the receive
// staging of the actives come from one file-scope device array of
// RELAY_NOALLOC_SCRATCH_BYTES (64 MiB). Every GPU that loads this library holds that
// array until the process exits.
//
// The page has no counterpart to this entry point; it is an addition of this library.
#include <cuda_runtime.h>

#include "program.h"

namespace relay {
namespace {

constexpr size_t kNoAllocBytes = RELAY_NOALLOC_SCRATCH_BYTES;

// Shared by every call on a device. It keeps whatever the previous call left in it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// The device address of g_noalloc_scratch on device `dev`. In host code the array's name
// is only a host-side stand-in, so the address is looked up with cudaGetSymbolAddress,
// once per device, while that device is current (the caller's current device).
void* noalloc_base(int dev, cudaError_t* err) {
  static void* cached[kMaxDevices] = {nullptr};
  if (dev < 0) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  if (dev < kMaxDevices && cached[dev] != nullptr) {
    *err = cudaSuccess;
    return cached[dev];
  }
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (*err != cudaSuccess) return nullptr;
  if (dev < kMaxDevices) cached[dev] = p;
  return p;
}

size_t round_up_256(size_t bytes) { return (bytes + 255) / 256 * 256; }

}  // namespace
}  // namespace relay

extern "C" relay_status_t relay_allreduce_noalloc(void* const* send, void* const* recv,
                                                  size_t count, relay_dtype_t dtype, int A,
                                                  int R, float scale, const relay_opts_t* opts,
                                                  cudaStream_t stream) {
  using namespace relay;
  relay_plan_t p;
  relay_status_t st = relay_plan(RELAY_ALLREDUCE, count, dtype, A, R, opts, &p);
  if (st != RELAY_OK) return st;
  void* scratch[RELAY_MAX_RANKS] = {nullptr};
  if (p.count > 0) {
    // every scratch element a pass reads was written by an earlier pass of the same
    // call, so nothing has to be cleared between calls
    const size_t active = round_up_256((size_t)p.active_scratch_elems * p.esize);
    const size_t helper = round_up_256((size_t)p.helper_elems * p.esize);
    const size_t need = (size_t)A * active + (size_t)p.H * helper;
    if (need > kNoAllocBytes)
      return report_error(RELAY_ERR_INVALID_ARGUMENT,
                          "relay_allreduce_noalloc: this allreduce needs " + std::to_string(need) +
                              " bytes of scratch; the built-in array holds " +
                              std::to_string(kNoAllocBytes));
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    char* base = e == cudaSuccess ? static_cast<char*>(noalloc_base(dev, &e)) : nullptr;
    if (base == nullptr)
      return report_error(RELAY_ERR_CUDA, std::string("relay_allreduce_noalloc: ") +
                                              cudaGetErrorString(e));
    size_t off = 0;
    for (int r = 0; r < R; ++r) {
      const size_t b = r < A ? active : helper;
      if (b > 0) scratch[r] = base + off;
      off += b;
    }
  }
  return relay_allreduce(send, recv, scratch, count, dtype, A, R, scale, opts, stream);
}
