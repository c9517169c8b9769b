// hadamard.cuh -- the random Hadamard transform of column blocks on the
// tensor cores, and the column-wise cast of its results ("Write both NVFP4
// amax buffers", review reply: with RHT the column amax is max|RHT(x)|; the
// transform of each 16-element column block is H16 diag(sign) / 4).
//
// For each 16-row block kk of a staged 128x128 BF16 tile, D_kk (128 x 16,
// FP32, tensor memory) = A_kk * B with A_kk[m][k] = x[16 kk + k][m] read
// straight from the TMA tile (MN-major, 128-byte swizzle: the two 64-column
// boxes are the M halves, 8-row groups 1024 bytes apart) and
// B[k][n] = sign_k H16[n][k] / 4 (exact in BF16), so that D_kk[m][n] is
// output n of the transform of column m's block.  Every product is exact and
// the sums are FP32 (their order is the tensor core's; codes may then differ
// from a left-to-right sum at rounding ties only).  Tile column m is
// tensor-memory lane m, so the warp with w % 4 == q reads columns 32q..32q+31.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace tile {

// B as 8x8 core matrices (K-major, no swizzle): element (k, n) at
// (n / 8) * gstride + (k / 8) * 128 + (n % 8) * 16 + (k % 8) * 2.
__device__ __forceinline__ void fill_hadamard_operand(uint8_t* hmat, int gstride, uint32_t sign_mask) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    const int k = i >> 4, n = i & 15;
    const bool neg = (((sign_mask >> k) & 1u) != 0) != ((__popc(n & k) & 1) != 0);
    const uint16_t v = neg ? 0xBE80u : 0x3E80u;  // -0.25 / +0.25 in BF16
    *reinterpret_cast<uint16_t*>(hmat + (n >> 3) * gstride + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2) = v;
  }
}

// One thread: the eight block transforms of the tile staged at `stage` into
// tensor-memory columns tmem .. tmem + 127, then one arrival on `bar` when
// they are complete.
__device__ __forceinline__ void rht_issue_mma(uint32_t stage, uint32_t hmat, int gstride, uint32_t tmem,
                                              uint64_t* bar) {
  constexpr uint32_t kIdesc = umma_idesc_bf16(128, 16, true);
  const uint64_t bdesc = umma_smem_desc(hmat, 128, (uint32_t)gstride, 0);
  tcgen05_after_sync();
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    umma_bf16(tmem + 16 * kk, umma_smem_desc(stage + kk * 16 * 128, kBoxBytes, 1024, 2), bdesc, kIdesc, 0);
  umma_commit(bar);
}

// max|BF16(t)| over the transformed blocks of this lane's tile column (the
// warp's lane quarter q), as a float.
__device__ __forceinline__ float rht_col_max(uint32_t tmem, int q) {
  uint32_t acc = 0;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t v[16];
    tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 16 * kk, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t h;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(__uint_as_float(v[2 * i + 1])), "f"(__uint_as_float(v[2 * i])));
      acc = xsa(acc, h);
    }
  }
  acc &= 0x7FFF7FFFu;
  return fmaxf(bf16_lo(acc), bf16_hi(acc));
}

// The column-wise cast of the transformed blocks of this lane's tile column
// m = 32 q + lane: rounds each output to BF16, takes each block's maximum,
// scale and codes, writes each 64 rows of the column as one 32-byte run and
// stages the eight block scales: compact staging byte kk * kScPitchCol + m,
// or (kSwz) the 128x4 layout's byte order (row m of atom kk / 4, byte kk % 4).
// Returns an XOR of every code word (depends on every value read).
template <bool kSwz>
__device__ __forceinline__ uint32_t rht_col_epilogue(uint32_t tmem, int q, const float* rtab_col, uint8_t* sc_col,
                                                     const CastArgs& a, int64_t r0, int64_t c0, float g_col) {
  const int lane = threadIdx.x & 31;
  const int m = 32 * q + lane;  // tile column
  uint32_t tok = 0;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t code[8];  // rows 64 half .. +64 of column m, eight per word
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int kk = 4 * half + j;
      uint32_t v[16];
      tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 16 * kk, v);
      uint32_t hb[8], acc = 0;  // BF16 pairs: rows 2i (low) and 2i + 1
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hb[i]) : "f"(__uint_as_float(v[2 * i + 1])), "f"(__uint_as_float(v[2 * i])));
        acc = xsa(acc, hb[i]);
      }
      acc &= 0x7FFF7FFFu;
      const uint32_t s = block_scale(fmaxf(bf16_lo(acc), bf16_hi(acc)), g_col);
      const float r = rtab_col[s];
      code[2 * j] = encode8(bf16_lo(hb[0]), bf16_hi(hb[0]), bf16_lo(hb[1]), bf16_hi(hb[1]), bf16_lo(hb[2]),
                            bf16_hi(hb[2]), bf16_lo(hb[3]), bf16_hi(hb[3]), r);
      code[2 * j + 1] = encode8(bf16_lo(hb[4]), bf16_hi(hb[4]), bf16_lo(hb[5]), bf16_hi(hb[5]), bf16_lo(hb[6]),
                                bf16_hi(hb[6]), bf16_lo(hb[7]), bf16_hi(hb[7]), r);
      tok ^= code[2 * j] ^ code[2 * j + 1];
      if constexpr (kSwz)
        sc_col[(kk >> 2) * 512 + (m & 31) * 16 + (m >> 5) * 4 + (kk & 3)] = (uint8_t)s;
      else
        sc_col[kk * kScPitchCol + m] = (uint8_t)s;
    }
    const int64_t x = c0 + m, rg = r0 + 64 * half;
    // M % 16 == 0: block kk is inside x when its first row is.
    if (x < a.N && rg < a.M) {
      uint8_t* dst = a.data_col + x * (a.M / 2) + rg / 2;
      if (rg + 64 <= a.M && (reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
        st_cs_v8(dst, code);  // the whole 32-byte sector at once
      } else if (rg + 64 <= a.M && ((a.M / 2) & 15) == 0) {
        st_cs_v4(dst, code[0], code[1], code[2], code[3]);
        st_cs_v4(dst + 16, code[4], code[5], code[6], code[7]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (rg + 16 * j < a.M) st_cs_v2(dst + 8 * j, code[2 * j], code[2 * j + 1]);
      }
    }
  }
  return tok;
}

}  // namespace tile
}  // namespace nvfp4
