// noalloc.cu -- the single-pass 2D quantize for callers that cannot allocate
// device memory.
//
// nvfp4_quantize_2d_single_pass needs a small workspace (the grid barrier's
// 64-byte header: a generation, arrival counts and maxima) that the caller
// normally allocates.  Some callers cannot do that: a plain C host
// that embeds this library without any device memory manager, code on a
// latency-critical path that must not take an allocator's lock or risk a
// synchronizing cudaMalloc / cudaFree, or a process that sized all of its
// device memory up front.  This entry point instead uses scratch that lives
// in this file, in a static device array the CUDA runtime places on every
// GPU that loads the library (and keeps there until the process exits).
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "nvfp4.h"

namespace {

// The scratch: the kernel's 64-byte barrier header (any number of CTAs).
constexpr size_t kScratchBytes = 256;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceScratch {
  bool ready = false;
  void* ptr = nullptr;  // device address of g_noalloc_scratch on that device
};
DeviceScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

// Once per device, with that device current: the device address of the
// array.  In host code the symbol itself is only a host-side stand-in, never
// a device address.  The address is that of the device's primary context at
// the time of the first call; it is not looked up again, so a
// cudaDeviceReset() of that device leaves it stale (documented in nvfp4.h).
nvfp4_status scratch_for_current_device(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  DeviceScratch& d = g_scratch[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return NVFP4_ERR_CUDA;
    d.ptr = p;
    d.ready = true;
  }
  *ptr = d.ptr;
  return NVFP4_OK;
}

}  // namespace

namespace nvfp4 {
nvfp4_status validate_single_pass(int mode, const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                                  unsigned flags, const float* noop);
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_quantize_2d_single_pass_noalloc(const void* x, int dtype, int64_t M, int64_t N,
                                                             const nvfp4_output* out, unsigned flags,
                                                             const float* noop, void* stream) {
  nvfp4_status st = nvfp4::validate_single_pass(nvfp4::kCast2D, x, dtype, M, N, out, flags, noop);
  if (st != NVFP4_OK) return st;
  void* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != NVFP4_OK) return st;
  // The array keeps whatever the previous call left; the barrier header
  // (generation, arrival counts, maxima) must start at zero, so clear it on the
  // stream before the kernel (a memset, no allocation).
  if (cudaMemsetAsync(scratch, 0, nvfp4::kSinglePassHeaderBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return nvfp4_quantize_2d_single_pass(x, dtype, M, N, out, flags, noop, scratch, stream);
}
