// amax.cu -- per-tensor amax for NVFP4: zero both direction buffers, then a
// vectorised max|x| reduction that applies one atomic max per thread block
// to both buffers ("Write both NVFP4 amax buffers", Description and
// Changes), and the random-Hadamard variant that reduces max|x| and
// max|RHT(x)| in the same read (the Hadamard-amax kernel of that page's
// "GPU work per quantize call" table).
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {
namespace {

constexpr int kAmaxThreads = 256;

__global__ void amax_zero_kernel(float* a, float* b, const float* noop) {
  grid_launch_dependents();
  if (noop != nullptr && *noop == 1.0f) return;
  if (a != nullptr) *a = 0.0f;
  if (b != nullptr) *b = 0.0f;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Block-wide max of non-negative floats; the result is valid in thread 0.
__device__ __forceinline__ float block_max(float m, float* red) {
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = (lane < (int)(blockDim.x >> 5)) ? red[lane] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  }
  return m;
}

// One atomic max per block into each buffer.  Non-negative floats order like
// their bit patterns read as signed integers.
__device__ __forceinline__ void publish_max(float m, float* a, float* b) {
  grid_dependency_wait();  // the zeroing kernel has completed
  atomicMax(reinterpret_cast<int*>(a), __float_as_int(m));
  if (b != nullptr) atomicMax(reinterpret_cast<int*>(b), __float_as_int(m));
}

// max|x| over n elements; x is 16-byte aligned.  nvec 16-byte vectors are
// read by the grid-stride loop in batches of kUnroll independent loads per
// thread (the last batch predicated, so no load waits behind another); one
// resident wave of CTAs keeps ~128 KB of reads in flight per SM.  The last
// n - nvec*epv elements are read by block 0.
constexpr int kUnroll = 8;

template <bool kBF16>
__global__ void __launch_bounds__(kAmaxThreads, 4) amax_reduce_kernel(const void* __restrict__ x, int64_t n,
                                                                      float* a, float* b, const float* noop) {
  __shared__ float red[kAmaxThreads / 32];
  grid_launch_dependents();
  if (noop != nullptr && *noop == 1.0f) return;
  constexpr int kEpv = kBF16 ? 8 : 4;
  const uint4* xv = static_cast<const uint4*>(x);
  const int64_t nvec = n / kEpv;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  float m = 0.0f;
  if constexpr (kBF16) {
    uint32_t acc0 = 0, acc1 = 0;
    auto fold = [&](const uint4& v) {
      uint32_t t0, t1;
      asm("max.bf16x2 %0, %1, %2;" : "=r"(t0) : "r"(v.x & 0x7FFF7FFFu), "r"(v.y & 0x7FFF7FFFu));
      asm("max.bf16x2 %0, %1, %2;" : "=r"(t1) : "r"(v.z & 0x7FFF7FFFu), "r"(v.w & 0x7FFF7FFFu));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(acc0) : "r"(t0));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(acc1) : "r"(t1));
    };
    for (; i < nvec; i += kUnroll * stride) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        v[u] = (i + u * stride < nvec) ? ld_stream(xv + i + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) fold(v[u]);
    }
    uint32_t acc;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(acc) : "r"(acc0), "r"(acc1));
    m = bf16x2_hmax_to_f32(acc);
    if (blockIdx.x == 0) {
      const uint16_t* xs = static_cast<const uint16_t*>(x);
      for (int64_t j = nvec * kEpv + threadIdx.x; j < n; j += blockDim.x)
        m = fmaxf(m, fabsf(__uint_as_float((uint32_t)xs[j] << 16)));
    }
  } else {
    float m0 = 0.0f, m1 = 0.0f;
    auto fold = [&](const uint4& v) {
      m0 = fmaxf(m0, fmaxf(fabsf(__uint_as_float(v.x)), fabsf(__uint_as_float(v.y))));
      m1 = fmaxf(m1, fmaxf(fabsf(__uint_as_float(v.z)), fabsf(__uint_as_float(v.w))));
    };
    for (; i < nvec; i += kUnroll * stride) {
      uint4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        v[u] = (i + u * stride < nvec) ? ld_stream(xv + i + u * stride) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) fold(v[u]);
    }
    m = fmaxf(m0, m1);
    if (blockIdx.x == 0) {
      const float* xs = static_cast<const float*>(x);
      for (int64_t j = nvec * kEpv + threadIdx.x; j < n; j += blockDim.x) m = fmaxf(m, fabsf(xs[j]));
    }
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) publish_max(m, a, b);
}

constexpr int kRhtAmaxThreads = 256;

// One work item = 16 rows x 8 columns (one 16-byte vector per row): row
// max|x| over the 128 values and, per column, max|(1/4) H16 diag(sign) v|.
// Consecutive threads take consecutive 8-column chunks (512 contiguous
// bytes per row and warp).  Two columns go through the transform together as
// FP32x2 pairs; each output is rounded to BF16 (as the cast rounds it) and
// the maxima are kept as packed BF16 pairs.
__global__ void __launch_bounds__(kRhtAmaxThreads, 2) rht_amax_kernel(const uint16_t* __restrict__ x, int64_t M,
                                                                   int64_t N, uint32_t sign_mask, float* a_row,
                                                                   float* a_col, const float* noop) {
  __shared__ float red[kRhtAmaxThreads / 32];
  grid_launch_dependents();
  if (noop != nullptr && *noop == 1.0f) return;
  float sgn[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) sgn[i] = ((sign_mask >> i) & 1u) ? -0.25f : 0.25f;
  const int64_t chunks = N / 8;
  const int64_t items = (M / 16) * chunks;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t racc = 0, cacc = 0;
  for (int64_t it = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; it < items; it += stride) {
    const int64_t band = it / chunks, chunk = it - band * chunks;
    const uint4* base = reinterpret_cast<const uint4*>(x + (band * 16) * N + chunk * 8);
    const int64_t rs = N / 8;  // row stride in 16-byte vectors
    uint4 v[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) v[r] = ld_stream(base + r * rs);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      uint32_t t0, t1;
      asm("max.bf16x2 %0, %1, %2;" : "=r"(t0) : "r"(v[r].x & 0x7FFF7FFFu), "r"(v[r].y & 0x7FFF7FFFu));
      asm("max.bf16x2 %0, %1, %2;" : "=r"(t1) : "r"(v[r].z & 0x7FFF7FFFu), "r"(v[r].w & 0x7FFF7FFFu));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(racc) : "r"(t0));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(racc) : "r"(t1));
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // columns 2q and 2q + 1 as FP32x2 pairs
      uint64_t u[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const uint32_t w = (q == 0) ? v[r].x : (q == 1) ? v[r].y : (q == 2) ? v[r].z : v[r].w;
        u[r] = bf16x2_scaled(w, sgn[r]);
      }
      fwht16_x2(u);
#pragma unroll
      for (int o = 0; o < 16; ++o) {
        uint32_t h = pair_to_bf16x2(u[o]) & 0x7FFF7FFFu;
        asm("max.bf16x2 %0, %0, %1;" : "+r"(cacc) : "r"(h));
      }
    }
  }
  float rm = block_max(bf16x2_hmax_to_f32(racc), red);
  __syncthreads();
  float cm = block_max(bf16x2_hmax_to_f32(cacc), red);
  if (threadIdx.x == 0) {
    grid_dependency_wait();
    if (a_row != nullptr) atomicMax(reinterpret_cast<int*>(a_row), __float_as_int(rm));
    atomicMax(reinterpret_cast<int*>(a_col), __float_as_int(cm));
  }
}

}  // namespace

cudaError_t launch_amax(const void* x, bool bf16, int64_t n, float* amax_a, float* amax_b, const float* noop,
                        const LaunchCtx& ctx) {
  amax_zero_kernel<<<1, 1, 0, ctx.stream>>>(amax_a, amax_b, noop);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int epv = bf16 ? 8 : 4;
  const int64_t nvec = n / epv;
  const void* fn = bf16 ? (const void*)amax_reduce_kernel<true> : (const void*)amax_reduce_kernel<false>;
  // One resident wave of CTAs; each walks the tensor with a grid stride.
  static std::atomic<int> occ[2] = {0, 0};  // CTAs per SM, same on every GB300
  int per_sm = occ[bf16].load();
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kAmaxThreads, 0);
    if (e != cudaSuccess) return e;
    occ[bf16].store(per_sm);
  }
  int64_t want = (nvec + kAmaxThreads * kUnroll - 1) / (kAmaxThreads * kUnroll);
  int64_t cap = (int64_t)ctx.num_sms * (per_sm > 0 ? per_sm : 1);
  int grid = (int)(want < 1 ? 1 : (want > cap ? cap : want));
  void* args[] = {(void*)&x, (void*)&n, (void*)&amax_a, (void*)&amax_b, (void*)&noop};
  return launch_pdl(fn, dim3(grid), dim3(kAmaxThreads), 0, ctx.stream, args);
}

cudaError_t launch_rht_amax(const uint16_t* x, int64_t M, int64_t N, uint32_t sign_mask, float* amax_row,
                            float* amax_col, const float* noop, const LaunchCtx& ctx) {
  amax_zero_kernel<<<1, 1, 0, ctx.stream>>>(amax_row, amax_col, noop);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t items = (M / 16) * (N / 8);
  static std::atomic<int> occ{0};
  int per_sm = occ.load();
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rht_amax_kernel, kRhtAmaxThreads, 0);
    if (e != cudaSuccess) return e;
    occ.store(per_sm);
  }
  int64_t want = (items + kRhtAmaxThreads - 1) / kRhtAmaxThreads;
  int64_t cap = (int64_t)ctx.num_sms * (per_sm > 0 ? per_sm : 1);
  int grid = (int)(want < 1 ? 1 : (want > cap ? cap : want));
  void* args[] = {(void*)&x, (void*)&M, (void*)&N, (void*)&sign_mask, (void*)&amax_row, (void*)&amax_col,
                  (void*)&noop};
  return launch_pdl((const void*)rht_amax_kernel, dim3(grid), dim3(kRhtAmaxThreads), 0, ctx.stream, args);
}

}  // namespace nvfp4
