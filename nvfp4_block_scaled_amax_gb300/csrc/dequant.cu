// dequant.cu -- NVFP4 dequantize of one direction, and the standalone
// compact -> cuBLAS 128x4 scale permutation.
//
// Dequantize ("Implement row-scaled NVFP4 fprop recipe", Important Files
// Changed: dequantize_nvfp4.cuh selects tensor_amax[y] for row-scaled data):
//   out[y][j] = (E2M1(q) * float(s)) * (a / 2688), FP32, then BF16 (RNE).
// One thread per 16-element block: 8 bytes of codes and one scale byte in,
// 32 (BF16) or 64 (FP32) bytes out.
#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

// E2M1 code -> value: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 from the
// exponent (bits 1..2) and mantissa (bit 0) fields; bit 3 is the sign.
__device__ __forceinline__ float e2m1_decode(uint32_t q) {
  const uint32_t m = q & 7u;
  uint32_t bits;
  if (m == 0)
    bits = 0;
  else if (m == 1)
    bits = 0x3F000000u;  // 0.5
  else
    bits = ((126u + (m >> 1)) << 23) | ((m & 1u) << 22);
  return __uint_as_float(bits | ((q & 8u) << 28));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// A warp walks the rows (one row at a time, rows spread over the grid's
// warps): each step covers 16 blocks of the row as 32 half blocks, lane l
// taking half (l & 1) of block (l >> 1) -- 4 code bytes in, 8 outputs out.
// The warp's code loads are then 128 contiguous bytes and, for BF16 output,
// its stores 512 contiguous bytes (whole 32-byte sectors).  Four steps are
// loaded before any is decoded, to keep enough loads in flight.
constexpr int kDeqSteps = 4;

template <bool kOutBF16>
__global__ void __launch_bounds__(kThreads) dequant_kernel(const uint8_t* __restrict__ data,
                                                           const uint8_t* __restrict__ scale,
                                                           const float* __restrict__ amax, int64_t rows,
                                                           int64_t cols, int swizzled, int row_scaled, void* out) {
  __shared__ float lut[16];
  if (threadIdx.x < 16) lut[threadIdx.x] = e2m1_decode(threadIdx.x);
  __syncthreads();
  const int64_t C = cols / 16;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int half = lane & 1;
  for (int64_t y = warp0; y < rows; y += nwarps) {
    const float kf = __fdiv_rn(row_scaled ? amax[y] : amax[0], 2688.0f);
    const uint8_t* drow = data + y * (cols / 2);
    for (int64_t k0 = 0; k0 < C; k0 += 16 * kDeqSteps) {
      uint32_t q[kDeqSteps], sc[kDeqSteps];
#pragma unroll
      for (int u = 0; u < kDeqSteps; ++u) {
        const int64_t k = k0 + 16 * u + (lane >> 1);
        if (k < C) {
          q[u] = *reinterpret_cast<const uint32_t*>(drow + 8 * k + 4 * half);
          sc[u] = scale[swizzled ? swizzled_scale_offset(y, k, C) : y * C + k];
        }
      }
#pragma unroll
      for (int u = 0; u < kDeqSteps; ++u) {
        const int64_t k = k0 + 16 * u + (lane >> 1);
        if (k >= C) break;
        const float sv = e4m3_decode(sc[u]);
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = __fmul_rn(__fmul_rn(lut[(q[u] >> (4 * i)) & 0xFu], sv), kf);
        const int64_t e0 = y * cols + 16 * k + 8 * half;  // first output element
        if constexpr (kOutBF16) {
          st_cs_v4(static_cast<uint8_t*>(out) + e0 * 2, pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                   pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
        } else {
          uint8_t* dst = static_cast<uint8_t*>(out) + e0 * 4;
          st_cs_v4(dst, __float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]), __float_as_uint(o[3]));
          st_cs_v4(dst + 16, __float_as_uint(o[4]), __float_as_uint(o[5]), __float_as_uint(o[6]),
                   __float_as_uint(o[7]));
        }
      }
    }
  }
}

// One thread per group of four scales (r, 4g .. 4g+3): one aligned 32-bit
// load from the compact matrix, one 32-bit store into the 128x4 layout.
__global__ void __launch_bounds__(kThreads) swizzle_kernel(const uint8_t* __restrict__ compact, uint8_t* swizzled,
                                                           int64_t rows, int64_t C) {
  const int64_t groups = rows * (C / 4);
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < groups; i += (int64_t)gridDim.x * kThreads) {
    const int64_t r = i / (C / 4), g = i - r * (C / 4);
    const uint32_t v = *reinterpret_cast<const uint32_t*>(compact + r * C + 4 * g);
    *reinterpret_cast<uint32_t*>(swizzled + swizzled_scale_offset(r, 4 * g, C)) = v;
  }
}

int grid_for(int64_t work, int num_sms) {
  const int64_t want = (work + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)num_sms * 8;
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_dequantize(const uint8_t* data, const uint8_t* scale, const float* amax, int64_t rows,
                              int64_t cols, bool swizzled, bool row_scaled, void* out, bool out_bf16,
                              const LaunchCtx& ctx) {
  const int64_t nblk = rows * (cols / 16);
  if (nblk == 0) return cudaSuccess;
  const int grid = grid_for(rows * 32, ctx.num_sms);  // a warp per row at a time
  if (out_bf16)
    dequant_kernel<true><<<grid, kThreads, 0, ctx.stream>>>(data, scale, amax, rows, cols, swizzled, row_scaled,
                                                            out);
  else
    dequant_kernel<false><<<grid, kThreads, 0, ctx.stream>>>(data, scale, amax, rows, cols, swizzled,
                                                             row_scaled, out);
  return cudaGetLastError();
}

cudaError_t launch_swizzle(const uint8_t* compact, uint8_t* swizzled, int64_t rows, int64_t scale_cols,
                           const LaunchCtx& ctx) {
  const int64_t groups = rows * (scale_cols / 4);
  if (groups == 0) return cudaSuccess;
  swizzle_kernel<<<grid_for(groups, ctx.num_sms), kThreads, 0, ctx.stream>>>(compact, swizzled, rows, scale_cols);
  return cudaGetLastError();
}

}  // namespace nvfp4
