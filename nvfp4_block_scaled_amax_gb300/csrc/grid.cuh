// grid.cuh -- the grid-wide barrier and maximum of the single-pass kernels
// (all CTAs co-resident: cooperative launch), in the caller's workspace
// header.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add_gpu(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_relaxed_max_gpu(unsigned* p, unsigned v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier and maximum.  Generation-counted, so the workspace needs
// no clearing between calls: call g (its generation read at kernel start)
// uses the pair arrive[g & 1] / maxbits[g & 1].  The last warp of each CTA
// to finish phase A (a shared-memory count) publishes the CTA's maximum with
// a relaxed atomic max, then arrives with a release add (which orders the
// max before it); thread 0 of each CTA polls the count (acquire, bounded)
// and then reads the maximum.  CTA 0 clears the other pair, which the next
// call uses, and advances the generation, which the next call (ordered after
// this kernel) reads.
__device__ __forceinline__ void grid_arrive(SinglePassWorkspace* ws, unsigned gen, float warp_max) {
  red_relaxed_max_gpu(&ws->maxbits[gen & 1u], __float_as_uint(warp_max));
  red_release_add_gpu(&ws->arrive[gen & 1u], 1u);
}
// The same with a second maximum (maxbits2).
__device__ __forceinline__ void grid_arrive2(SinglePassWorkspace* ws, unsigned gen, float max1, float max2) {
  red_relaxed_max_gpu(&ws->maxbits[gen & 1u], __float_as_uint(max1));
  red_relaxed_max_gpu(&ws->maxbits2[gen & 1u], __float_as_uint(max2));
  red_release_add_gpu(&ws->arrive[gen & 1u], 1u);
}
// Thread 0 only; false when the wait ran out.
__device__ __forceinline__ bool grid_wait_max(SinglePassWorkspace* ws, unsigned gen, unsigned expected,
                                              unsigned* status, float* out, float* out2 = nullptr) {
  const long long t0 = clock64();
  while (ld_acquire_gpu(&ws->arrive[gen & 1u]) < expected) {
    if (clock64() - t0 > kWaitLimitCycles) {
      atomicOr(status, kStatusGridTimeout);
      return false;
    }
  }
  *out = __uint_as_float(ld_relaxed_gpu(&ws->maxbits[gen & 1u]));
  if (out2 != nullptr) *out2 = __uint_as_float(ld_relaxed_gpu(&ws->maxbits2[gen & 1u]));
  if (blockIdx.x == 0) {  // unused by this call; the next one counts there
    ws->arrive[(gen + 1u) & 1u] = 0u;
    ws->maxbits[(gen + 1u) & 1u] = 0u;
    ws->maxbits2[(gen + 1u) & 1u] = 0u;
    st_release_gpu(&ws->gen, gen + 1u);
  }
  return true;
}


}  // namespace nvfp4
