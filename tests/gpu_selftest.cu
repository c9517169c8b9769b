// gpu_selftest.cu -- test-only kernels that run the library's device helpers
// (hardware E2M1 / E4M3 / BF16 conversions, the stochastic-rounding E2M1
// encoder, the division by 6, the bounded
// mbarrier wait) on arbitrary inputs, so the tests can compare them with the
// oracle exhaustively.  Built by the GPU tests; never part of libnvfp4.
#include "common.cuh"

using namespace nvfp4;

namespace {

__global__ void e2m1_kernel(const float* in, uint8_t* out, int64_t n8) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (int64_t)gridDim.x * blockDim.x) {
    const float* v = in + 8 * i;
    const uint32_t w = e2m1x8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
    for (int k = 0; k < 8; ++k) out[8 * i + k] = (w >> (4 * k)) & 0xFu;
  }
}

__global__ void e2m1_sr_kernel(const float* in, const uint8_t* rb, uint8_t* out, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (uint8_t)e2m1_sr(in[i], sr_offset(rb[i]));
}

__global__ void e4m3_kernel(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (uint8_t)e4m3_rn_satfinite(in[i]);
}

__global__ void bf16_kernel(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = (uint16_t)(__float_as_uint(round_bf16(in[i])) >> 16);
}

// Every positive finite FP32 bit pattern in [lo, hi): counts where the
// FMA-corrected quotient differs from the IEEE division, keeps one example.
__global__ void div6_kernel(uint32_t lo, uint32_t hi, unsigned long long* bad, uint32_t* example) {
  for (uint64_t b = (uint64_t)lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < hi;
       b += (uint64_t)gridDim.x * blockDim.x) {
    const float x = __uint_as_float((uint32_t)b);
    if (__float_as_uint(div6_rn(x)) != __float_as_uint(__fdiv_rn(x, 6.0f))) {
      atomicAdd(bad, 1ull);
      *example = (uint32_t)b;
    }
  }
}

// An mbarrier that nothing ever arrives on: the bounded wait must give up,
// set the status bit and let the kernel return.
__global__ void wait_timeout_kernel(unsigned* status, long long limit, int* result) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0, status, limit);
  if (threadIdx.x == 0) *result = ok ? 1 : 0;
}

}  // namespace

extern "C" {

int selftest_e2m1(const float* in, uint8_t* out, int64_t n) {
  e2m1_kernel<<<1024, 256>>>(in, out, n / 8);
  return (int)cudaDeviceSynchronize();
}

int selftest_e2m1_sr(const float* in, const uint8_t* rb, uint8_t* out, int64_t n) {
  e2m1_sr_kernel<<<1024, 256>>>(in, rb, out, n);
  return (int)cudaDeviceSynchronize();
}

int selftest_e4m3(const float* in, uint8_t* out, int64_t n) {
  e4m3_kernel<<<1024, 256>>>(in, out, n);
  return (int)cudaDeviceSynchronize();
}

int selftest_bf16(const float* in, uint16_t* out, int64_t n) {
  bf16_kernel<<<1024, 256>>>(in, out, n);
  return (int)cudaDeviceSynchronize();
}

int selftest_div6(uint32_t lo, uint32_t hi, unsigned long long* bad, uint32_t* example) {
  div6_kernel<<<4096, 256>>>(lo, hi, bad, example);
  return (int)cudaDeviceSynchronize();
}

int selftest_wait_timeout(unsigned* status, long long limit, int* result) {
  wait_timeout_kernel<<<1, 32>>>(status, limit, result);
  return (int)cudaDeviceSynchronize();
}

}  // extern "C"
