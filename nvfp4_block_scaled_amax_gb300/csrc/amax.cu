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

// max|x| over n elements; x is 16-byte aligned.  One persistent CTA per SM
// streams 32 KB chunks of x (chunk b + k G for CTA b of G) through a ring of
// kAmaxStages shared-memory stages with bulk copies, several chunks in flight
// per SM; each chunk is folded by the CTA's threads (16-byte reads,
// consecutive threads on consecutive vectors), then refilled.  The last
// (n * element size) mod 16 bytes are read by block 0.
constexpr int kAmaxThreads = 512, kAmaxStages = 4;
constexpr uint32_t kAmaxChunk = 32768;
constexpr size_t kAmaxSmem = (size_t)kAmaxStages * kAmaxChunk + 128;

template <bool kBF16>
__global__ void __launch_bounds__(kAmaxThreads, 1) amax_reduce_kernel(const uint8_t* __restrict__ x, int64_t n,
                                                                      float* a, float* b, const float* noop,
                                                                      unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kAmaxStages];
  __shared__ float red[kAmaxThreads / 32];
  __shared__ int failed;
  grid_launch_dependents();
  if (noop != nullptr && *noop == 1.0f) return;
  constexpr int kEb = kBF16 ? 2 : 4;
  const uint32_t stages = (smem_u32(smem_raw) + 127u) & ~127u;
  const int tid = threadIdx.x, G = gridDim.x, bid = blockIdx.x;
  const int64_t main_bytes = (n * kEb) & ~(int64_t)15;
  const int64_t nchunks = (main_bytes + kAmaxChunk - 1) / kAmaxChunk;
  const int my = bid < nchunks ? (int)((nchunks - 1 - bid) / G + 1) : 0;
  auto chunk_bytes = [&](int k) {
    const int64_t left = main_bytes - (bid + (int64_t)k * G) * (int64_t)kAmaxChunk;
    return (uint32_t)(left < (int64_t)kAmaxChunk ? left : (int64_t)kAmaxChunk);
  };
  auto issue = [&](int k) {
    const int s = k % kAmaxStages;
    const uint32_t sz = chunk_bytes(k);
    mbar_arrive_expect_tx(&full[s], sz);
    bulk_load(stages + (uint32_t)s * kAmaxChunk, x + (bid + (int64_t)k * G) * (int64_t)kAmaxChunk, sz, &full[s]);
  };
  if (tid == 0) {
    for (int s = 0; s < kAmaxStages; ++s) mbar_init(&full[s], 1);
    failed = 0;
    fence_mbar_init();
    for (int k = 0; k < kAmaxStages && k < my; ++k) issue(k);
  }
  __syncthreads();
  uint32_t acc0 = 0, acc1 = 0;  // BF16: packed maxima of |x|
  float m0 = 0.0f, m1 = 0.0f;   // FP32
  int k = 0;
  for (; k < my; ++k) {
    const int s = k % kAmaxStages;
    const bool ok = mbar_wait_bounded(&full[s], (uint32_t)((k / kAmaxStages) & 1), status);
    if (__syncthreads_or(!ok)) break;
    const uint32_t sz = chunk_bytes(k), base = stages + (uint32_t)s * kAmaxChunk;
#pragma unroll
    for (int q = 0; q < (int)(kAmaxChunk / 16 / kAmaxThreads); ++q) {
      const uint32_t off = (uint32_t)(q * kAmaxThreads + tid) * 16u;
      if (off < sz) {
        uint4 v;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "r"(base + off));
        if constexpr (kBF16) {
          uint32_t t0, t1;
          asm("max.bf16x2 %0, %1, %2;" : "=r"(t0) : "r"(v.x & 0x7FFF7FFFu), "r"(v.y & 0x7FFF7FFFu));
          asm("max.bf16x2 %0, %1, %2;" : "=r"(t1) : "r"(v.z & 0x7FFF7FFFu), "r"(v.w & 0x7FFF7FFFu));
          asm("max.bf16x2 %0, %0, %1;" : "+r"(acc0) : "r"(t0));
          asm("max.bf16x2 %0, %0, %1;" : "+r"(acc1) : "r"(t1));
        } else {
          m0 = fmaxf(m0, fmaxf(fabsf(__uint_as_float(v.x)), fabsf(__uint_as_float(v.y))));
          m1 = fmaxf(m1, fmaxf(fabsf(__uint_as_float(v.z)), fabsf(__uint_as_float(v.w))));
        }
      }
    }
    __syncthreads();  // stage s read by every thread
    if (tid == 0 && k + kAmaxStages < my) issue(k + kAmaxStages);
  }
  if (k < my) {
    // A wait ran out (status recorded): let the copies still in flight land,
    // bounded, before the shared memory is released; publish nothing.
    if (tid == 0) {
      const int issued = k + kAmaxStages < my ? k + kAmaxStages : my;
      for (int jj = k; jj < issued; ++jj)
        mbar_wait_bounded(&full[jj % kAmaxStages], (uint32_t)((jj / kAmaxStages) & 1), status);
    }
    return;
  }
  float m;
  if constexpr (kBF16) {
    uint32_t acc;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(acc) : "r"(acc0), "r"(acc1));
    m = bf16x2_hmax_to_f32(acc);
    if (bid == 0) {
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(x);
      for (int64_t j = main_bytes / kEb + tid; j < n; j += kAmaxThreads)
        m = fmaxf(m, fabsf(__uint_as_float((uint32_t)xs[j] << 16)));
    }
  } else {
    m = fmaxf(m0, m1);
    if (bid == 0) {
      const float* xs = reinterpret_cast<const float*>(x);
      for (int64_t j = main_bytes / kEb + tid; j < n; j += kAmaxThreads) m = fmaxf(m, fabsf(xs[j]));
    }
  }
  m = block_max(m, red);
  if (tid == 0) publish_max(m, a, b);
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
  const void* fn = bf16 ? (const void*)amax_reduce_kernel<true> : (const void*)amax_reduce_kernel<false>;
  static std::atomic<uint64_t> attr_set[2] = {0, 0};  // per kernel, bit per device
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set[bf16].load() & bit)) {
    if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAmaxSmem)) != cudaSuccess)
      return e;
    attr_set[bf16].fetch_or(bit);
  }
  // one persistent CTA per SM (fewer if x has fewer 32 KB chunks)
  const int64_t chunks = ((n * (bf16 ? 2 : 4)) / 16 * 16 + kAmaxChunk - 1) / kAmaxChunk;
  const int grid = (int)(chunks < 1 ? 1 : (chunks > ctx.num_sms ? ctx.num_sms : chunks));
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  unsigned* status = ctx.status;
  void* args[] = {(void*)&xb, (void*)&n, (void*)&amax_a, (void*)&amax_b, (void*)&noop, (void*)&status};
  return launch_pdl(fn, dim3(grid), dim3(kAmaxThreads), kAmaxSmem, ctx.stream, args);
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
