// row_scaled.cu -- per-token (row-scaled) NVFP4: one FP32 amax per row,
// block scales relative to that row's global scale ("Implement row-scaled
// NVFP4 fprop recipe", Greptile summary).  The per-row amax and the cast are
// fused: a warp owns a row; when the row fits in the warp's registers
// (N <= 32 * 16 * kBPL elements) it is read from HBM exactly once, otherwise
// the warp makes an amax pass and re-reads the row (from L1/L2) to cast it.
#include "common.cuh"
#include "kernels.h"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;  // 8 warps = 8 rows in flight per CTA

__device__ __forceinline__ uint4 ld_row(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <bool kBF16>
struct RowCfg {
  static constexpr int kV = kBF16 ? 2 : 4;    // 16-byte vectors per 16-element block
  static constexpr int kBPL = kBF16 ? 8 : 4;  // blocks per lane per segment
};

template <bool kBF16>
__device__ __forceinline__ float vec_elem(const uint4* v, int i) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(v);
  if constexpr (kBF16)
    return (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
  else
    return __uint_as_float(w[i]);
}

template <bool kBF16>
__device__ __forceinline__ float block_absmax(const uint4* v) {
  if constexpr (kBF16) {  // packed BF16 pairs
    const uint32_t acc = tile::xsa(tile::xsa(tile::xsa(v[0].x, v[0].y), tile::xsa(v[0].z, v[0].w)),
                                   tile::xsa(tile::xsa(v[1].x, v[1].y), tile::xsa(v[1].z, v[1].w))) &
                         0x7FFF7FFFu;
    return fmaxf(bf16_lo(acc), bf16_hi(acc));
  } else {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(vec_elem<kBF16>(v, i)));
    return m;
  }
}

template <bool kBF16>
__device__ __forceinline__ void cast_block(const uint4* v, float bmax, float g, int64_t y, int64_t k, int64_t N,
                                           uint8_t* data, uint8_t* scale, bool swizzled) {
  const uint32_t s = e4m3_rn_satfinite(__fmul_rn(div6_rn(bmax), g));
  const float r = encode_factor(s, g);
  uint32_t lo, hi;
  if constexpr (kBF16) {  // packed FP32x2 products straight from the BF16 words
    const uint32_t* w = reinterpret_cast<const uint32_t*>(v);
    lo = tile::encode8(bf16_lo(w[0]), bf16_hi(w[0]), bf16_lo(w[1]), bf16_hi(w[1]), bf16_lo(w[2]), bf16_hi(w[2]),
                       bf16_lo(w[3]), bf16_hi(w[3]), r);
    hi = tile::encode8(bf16_lo(w[4]), bf16_hi(w[4]), bf16_lo(w[5]), bf16_hi(w[5]), bf16_lo(w[6]), bf16_hi(w[6]),
                       bf16_lo(w[7]), bf16_hi(w[7]), r);
  } else {
    float e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) e[i] = __fmul_rn(vec_elem<kBF16>(v, i), r);
    lo = e2m1x8(e[0], e[1], e[2], e[3], e[4], e[5], e[6], e[7]);
    hi = e2m1x8(e[8], e[9], e[10], e[11], e[12], e[13], e[14], e[15]);
  }
  st_cs_v2(data + y * (N / 2) + 8 * k, lo, hi);
  const int64_t C = N / 16;
  st_cs_u8(scale + (swizzled ? swizzled_scale_offset(y, k, C) : y * C + k), s);
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 2) row_scaled_kernel(const void* __restrict__ x, int64_t M, int64_t N,
                                                              uint8_t* data, uint8_t* scale, float* amax,
                                                              int skip_amax, int swizzled, const float* noop) {
  using RC = RowCfg<kBF16>;
  if (noop != nullptr && *noop == 1.0f) return;
  const int lane = threadIdx.x & 31;
  const int64_t warp_g = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int64_t nblk = N / 16;
  constexpr int kSeg = 32 * RC::kBPL;  // blocks per segment
  const int64_t nseg = (nblk + kSeg - 1) / kSeg;
  const int64_t row_vecs = nblk * RC::kV;

  for (int64_t y = warp_g; y < M; y += nwarps) {
    const uint4* xr = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(x) + y * N * (kBF16 ? 2 : 4));
    if (nseg <= 1) {
      // Whole row in registers: one HBM read.
      uint4 v[RC::kBPL][RC::kV];
#pragma unroll
      for (int j = 0; j < RC::kBPL; ++j) {
        const int64_t k = (int64_t)j * 32 + lane;
#pragma unroll
        for (int q = 0; q < RC::kV; ++q)
          v[j][q] = (k < nblk) ? ld_row(xr + k * RC::kV + q) : make_uint4(0, 0, 0, 0);
      }
      float m = 0.0f;
#pragma unroll
      for (int j = 0; j < RC::kBPL; ++j) m = fmaxf(m, block_absmax<kBF16>(v[j]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      if (skip_amax)
        m = amax[y];
      else if (lane == 0)
        amax[y] = m;
      const float g = global_encode_scale(m);
#pragma unroll
      for (int j = 0; j < RC::kBPL; ++j) {
        const int64_t k = (int64_t)j * 32 + lane;
        if (k < nblk) cast_block<kBF16>(v[j], block_absmax<kBF16>(v[j]), g, y, k, N, data, scale, swizzled);
      }
    } else {
      // Long row: amax pass, then a second read that casts.
      float m = 0.0f;
      if (skip_amax) {
        m = amax[y];
      } else {
        for (int64_t k = lane; k < nblk; k += 32) {
          uint4 v[RC::kV];
#pragma unroll
          for (int q = 0; q < RC::kV; ++q) v[q] = ld_row(xr + k * RC::kV + q);
          m = fmaxf(m, block_absmax<kBF16>(v));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (lane == 0) amax[y] = m;
      }
      const float g = global_encode_scale(m);
      for (int64_t k = lane; k < nblk; k += 32) {
        uint4 v[RC::kV];
#pragma unroll
        for (int q = 0; q < RC::kV; ++q) v[q] = ld_row(xr + k * RC::kV + q);
        cast_block<kBF16>(v, block_absmax<kBF16>(v), g, y, k, N, data, scale, swizzled);
      }
    }
    (void)row_vecs;
  }
}

}  // namespace

cudaError_t launch_row_scaled(const void* x, bool bf16, int64_t M, int64_t N, uint8_t* data, uint8_t* scale,
                              float* amax, bool skip_amax, bool swizzled, const float* noop,
                              const LaunchCtx& ctx) {
  if (M == 0) return cudaSuccess;
  const int64_t want = (M + 7) / 8;
  const int64_t cap = (int64_t)ctx.num_sms * 2;
  const int grid = (int)(want < cap ? want : cap);
  if (bf16)
    row_scaled_kernel<true><<<grid, kThreads, 0, ctx.stream>>>(x, M, N, data, scale, amax, skip_amax, swizzled,
                                                               noop);
  else
    row_scaled_kernel<false><<<grid, kThreads, 0, ctx.stream>>>(x, M, N, data, scale, amax, skip_amax,
                                                                swizzled, noop);
  return cudaGetLastError();
}

}  // namespace nvfp4
