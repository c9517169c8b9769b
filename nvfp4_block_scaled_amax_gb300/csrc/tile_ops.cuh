// tile_ops.cuh -- the per-tile arithmetic shared by the NVFP4 cast kernels:
// a 128x128 tile of x staged by TMA in shared memory (128-byte swizzle) is
// cast by 8 warps, each thread owning an 8x8 sub-block.
//
//   * a 1x16 row block is the sub-blocks of lanes l and l^1; a 16x1 column
//     block those of lanes l and l^8; a 16x16 tile lanes l, l^1, l^8, l^9;
//     block maxima are combined with one or two shuffles;
//   * row-wise codes: one 32-bit word (8 codes) per row of the sub-block;
//   * column-wise codes: one word per column of the sub-block, computed from
//     the same registers (1D, with the column block's scale) or, in 2D, the
//     8x8 nibble transpose of the row-wise words (same scale per tile);
//   * the tile's scales are staged in shared memory (see staged_scale) and
//     stored as 16-byte lines of the cuBLAS 128x4 layout ("Fuse NVFP4 scale
//     swizzling on SM120 and SM121", Changes: aligned groups of four scales
//     written together) or 8-byte runs of the compact layout.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {
namespace tile {

constexpr int kTile = 128;            // tile rows = tile columns (elements)
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 128 bytes

template <typename T>
struct TileCfg;
template <>
struct TileCfg<uint16_t> {
  static constexpr int kBoxCols = 64, kBoxes = 2, kStages = 3, kMinBlocks = 2;
};
template <>
struct TileCfg<float> {
  static constexpr int kBoxCols = 32, kBoxes = 4, kStages = 3, kMinBlocks = 1;
};

template <typename T>
__host__ __device__ constexpr int tile_bytes() {
  return TileCfg<T>::kBoxes * kBoxBytes;
}
// Staged scales of one tile, one region per direction.  Index r is the tile
// row of that direction's output (an x row for the row-wise scales, an x
// column for the column-wise ones), c its scale column (0..7).
//   * 1D: scale (r, c) at c * pitch + r.  A thread stages the eight scales of
//     its sub-block's rows (row-wise) or columns (column-wise) for one scale
//     column with one 8-byte store; the pitches (row-wise 160, column-wise
//     192 bytes) put the eight-byte stores of a warp in distinct banks.
//   * 2D: one byte per 16x16 tile, at (r / 16) * 8 + c in both directions:
//     tile (ty, tx) at ty * 8 + tx row-wise and at tx * 8 + ty column-wise,
//     so that four consecutive scale columns of a row are one 32-bit word.
constexpr int kScPitchRow = 160, kScPitchCol = 192;
constexpr int kScRegion = 8 * kScPitchCol;  // bytes per direction

template <int MODE, bool kColDir>
__device__ __forceinline__ uint32_t staged_scale(const uint8_t* s, int r, int c) {
  if constexpr (MODE == kCast2D)
    return s[(r >> 4) * 8 + c];
  else
    return s[c * (kColDir ? kScPitchCol : kScPitchRow) + r];
}

// stages | 2 encode-factor tables | 2 x 2 staged scale regions | barriers | flag
template <typename T>
__host__ __device__ constexpr size_t smem_bytes() {
  return 1024 + (size_t)TileCfg<T>::kStages * tile_bytes<T>() + 2 * 128 * 4 + 4 * kScRegion +
         8 * TileCfg<T>::kStages + 16;
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in box `box` of a
// stage: the TMA 128-byte swizzle XORs the chunk index with row % 8.
__device__ __forceinline__ uint32_t swz(int box, int row, int chunk) {
  return (uint32_t)(box * kBoxBytes + row * 128 + (((chunk ^ row) & 7) << 4));
}

// E4M3 scale code of a block with maximum b under global scale g.
__device__ __forceinline__ uint32_t block_scale(float b, float g) {
  return e4m3_rn_satfinite(__fmul_rn(div6_rn(b), g));
}
// block_scale of two block maxima at once (packed FP32x2 arithmetic, one
// E4M3 pair conversion): s(b0) | s(b1) << 8.  The same steps as div6_rn
// (quotient, exact residual, correction; tiny maxima take the division).
__device__ __forceinline__ uint32_t block_scale2(float b0, float b1, float g) {
  float v0, v1;
  if (fminf(b0, b1) < 1.0e-30f) {
    v0 = __fmul_rn(div6_rn(b0), g);
    v1 = __fmul_rn(div6_rn(b1), g);
  } else {
    uint64_t b, q, e, c, m6, gg;
    asm("mov.b64 %0, {%1, %2};" : "=l"(b) : "f"(b0), "f"(b1));
    asm("mov.b64 %0, {%1, %1};" : "=l"(c) : "f"(1.0f / 6.0f));
    asm("mov.b64 %0, {%1, %1};" : "=l"(m6) : "f"(-6.0f));
    asm("mov.b64 %0, {%1, %1};" : "=l"(gg) : "f"(g));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(b), "l"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(e) : "l"(q), "l"(m6), "l"(b));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(e), "l"(c), "l"(q));
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(q) : "l"(q), "l"(gg));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v0), "=f"(v1) : "l"(q));
  }
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(v1), "f"(v0));
  return h;
}

// Two products in one packed FP32x2 multiply (each an IEEE product rounded
// to nearest), then the E2M1 codes of eight values.
__device__ __forceinline__ uint64_t mul2(float a, float b, uint64_t rr) {
  uint64_t p, v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(a), "f"(b));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(v), "l"(rr));
  return p;
}
__device__ __forceinline__ uint64_t splat2(float r) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %1};" : "=l"(v) : "f"(r));
  return v;
}
__device__ __forceinline__ uint32_t e2m1x8_pairs(uint64_t p0, uint64_t p1, uint64_t p2, uint64_t p3) {
  uint32_t out;
  asm("{\n"
      ".reg .b8 q0, q1, q2, q3;\n"
      ".reg .f32 a0, a1, a2, a3, a4, a5, a6, a7;\n"
      "mov.b64 {a0, a1}, %1;\n"
      "mov.b64 {a2, a3}, %2;\n"
      "mov.b64 {a4, a5}, %3;\n"
      "mov.b64 {a6, a7}, %4;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q0, a1, a0;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q1, a3, a2;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q2, a5, a4;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q3, a7, a6;\n"
      "mov.b32 %0, {q0, q1, q2, q3};\n"
      "}"
      : "=r"(out)
      : "l"(p0), "l"(p1), "l"(p2), "l"(p3));
  return out;
}
// Codes of v[0..7] * r, v[0] in the low nibble.
__device__ __forceinline__ uint32_t encode8(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                            float v7, float r) {
  const uint64_t rr = splat2(r);
  return e2m1x8_pairs(mul2(v0, v1, rr), mul2(v2, v3, rr), mul2(v4, v5, rr), mul2(v6, v7, rr));
}

// 8x8 transpose of 4-bit elements held as 8 words (word k = row k, element
// c at bits 4c..4c+3): afterwards word c holds column c, row k at bits 4k.
__device__ __forceinline__ void transpose_nibbles8x8(uint32_t (&w)[8]) {
  // swap the off-diagonal elements of every 2x2 block of nibbles
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
    const uint32_t a = w[k], b = w[k + 1];
    w[k] = (a & 0x0F0F0F0Fu) | ((b << 4) & 0xF0F0F0F0u);
    w[k + 1] = ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
  }
  // then of every 2x2 block of bytes (2x2-nibble blocks)
#pragma unroll
  for (int k = 0; k < 8; k += 4) {
#pragma unroll
    for (int d = 0; d < 2; ++d) {
      const uint32_t a = w[k + d], b = w[k + d + 2];
      w[k + d] = __byte_perm(a, b, 0x6240);
      w[k + d + 2] = __byte_perm(a, b, 0x7351);
    }
  }
  // then of the 2x2 block of half-words (4x4-nibble blocks)
#pragma unroll
  for (int d = 0; d < 4; ++d) {
    const uint32_t a = w[d], b = w[d + 4];
    w[d] = __byte_perm(a, b, 0x5410);
    w[d + 4] = __byte_perm(a, b, 0x7632);
  }
}

// ---------------------------------------------------------------------------
// 8x8 sub-block pass.  Warp w: bx = w & 1 (tile columns 64bx .. +63),
// q = w >> 1 (tile rows 32q .. +31); lane l: j = l & 7 (columns 64bx + 8j ..
// +7), i = l >> 3 (rows 32q + 8i .. +7).  For BF16 the eight lanes of one
// shared-memory phase read eight different 16-byte chunks (conflict-free).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Packed BF16 pair: per half max(|a|, |b|) (the sign bits are junk and are
// cleared where the value is used).
__device__ __forceinline__ uint32_t xsa(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// (lo of a, lo of b) and (hi of a, hi of b) -> per-half max of |.|: a packed
// pair (max|a|, max|b|) from two packed pairs.
__device__ __forceinline__ uint32_t xsa_pairs(uint32_t a, uint32_t b) {
  return xsa(__byte_perm(a, b, 0x5410), __byte_perm(a, b, 0x7632));
}

// The 8x8 sub-block in registers.  BF16: w[k][p] holds columns 2p (low half)
// and 2p+1 of row k.  FP32: w[k][c] is column c of row k.
template <typename T>
struct Sub {
  static constexpr int kW = sizeof(T) == 2 ? 4 : 8;
  uint32_t w[8][kW];
  __device__ __forceinline__ float v(int k, int c) const {
    if constexpr (sizeof(T) == 2)
      return (c & 1) ? bf16_hi(w[k][c >> 1]) : bf16_lo(w[k][c >> 1]);
    else
      return __uint_as_float(w[k][c]);
  }
};

// Loads rows trow..trow+7 of the sub-block; trow is a multiple of 8, so the
// swizzled chunk of row trow + k is chunk ^ k, i.e. the address bits 4..6 of
// the unswizzled address XOR k.
template <typename T>
__device__ __forceinline__ void load_sub(uint32_t stage, int bx, int trow, int j, Sub<T>& s) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t base = stage + bx * kBoxBytes + trow * 128 + (j << 4);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 c = lds128((base + 128 * k) ^ (k << 4));
      s.w[k][0] = c.x; s.w[k][1] = c.y; s.w[k][2] = c.z; s.w[k][3] = c.w;
    }
  } else {
    const uint32_t base = stage + (2 * bx + (j >> 2)) * kBoxBytes + trow * 128 + ((2 * (j & 3)) << 4);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint4 c0 = lds128((base + 128 * k) ^ (k << 4));
      const uint4 c1 = lds128((base + 16 + 128 * k) ^ (k << 4));
      s.w[k][0] = c0.x; s.w[k][1] = c0.y; s.w[k][2] = c0.z; s.w[k][3] = c0.w;
      s.w[k][4] = c1.x; s.w[k][5] = c1.y; s.w[k][6] = c1.z; s.w[k][7] = c1.w;
    }
  }
}

template <typename T>
__device__ __forceinline__ uint32_t encode_row(const Sub<T>& s, int k, float r) {
  return encode8(s.v(k, 0), s.v(k, 1), s.v(k, 2), s.v(k, 3), s.v(k, 4), s.v(k, 5), s.v(k, 6), s.v(k, 7), r);
}
template <typename T>
__device__ __forceinline__ uint32_t encode_col(const Sub<T>& s, int c, float r) {
  return encode8(s.v(0, c), s.v(1, c), s.v(2, c), s.v(3, c), s.v(4, c), s.v(5, c), s.v(6, c), s.v(7, c), r);
}

// Packed pair (max|x| of row 2t, of row 2t+1) over the sub-block's columns,
// combined with lane l^1 (the other half of each 1x16 block).  BF16 only.
__device__ __forceinline__ uint32_t row_pair_max(const Sub<uint16_t>& s, int t) {
  const uint32_t a = xsa(xsa(s.w[2 * t][0], s.w[2 * t][1]), xsa(s.w[2 * t][2], s.w[2 * t][3]));
  const uint32_t b = xsa(xsa(s.w[2 * t + 1][0], s.w[2 * t + 1][1]), xsa(s.w[2 * t + 1][2], s.w[2 * t + 1][3]));
  const uint32_t pr = xsa_pairs(a, b);
  return xsa(pr, __shfl_xor_sync(0xFFFFFFFFu, pr, 1)) & 0x7FFF7FFFu;
}
// Packed pair (max|x| of column 2p, of column 2p+1) over the sub-block's 8
// rows, combined with lane l^8 (the other half of each 16-row block).
__device__ __forceinline__ uint32_t col_pair_max(const Sub<uint16_t>& s, int p) {
  const uint32_t acc = xsa(xsa(xsa(s.w[0][p], s.w[1][p]), xsa(s.w[2][p], s.w[3][p])),
                           xsa(xsa(s.w[4][p], s.w[5][p]), xsa(s.w[6][p], s.w[7][p])));
  return xsa(acc, __shfl_xor_sync(0xFFFFFFFFu, acc, 8)) & 0x7FFF7FFFu;
}
__device__ __forceinline__ float row_max_f32(const Sub<float>& s, int k) {
  float m = 0.0f;
#pragma unroll
  for (int c = 0; c < 8; ++c) m = fmaxf(m, fabsf(s.v(k, c)));
  return fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
}
__device__ __forceinline__ float col_max_f32(const Sub<float>& s, int c) {
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(s.v(k, c)));
  return fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
}

// 16x16 tile maximum: the sub-block's max combined over lanes l^1, l^8.
template <typename T>
__device__ __forceinline__ float tile_max(const Sub<T>& s) {
  float m;
  if constexpr (sizeof(T) == 2) {
    uint32_t acc = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) acc = xsa(acc, xsa(xsa(s.w[k][0], s.w[k][1]), xsa(s.w[k][2], s.w[k][3])));
    acc &= 0x7FFF7FFFu;
    m = fmaxf(bf16_lo(acc), bf16_hi(acc));
  } else {
    m = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int c = 0; c < 8; ++c) m = fmaxf(m, fabsf(s.v(k, c)));
  }
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  return fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
}

// Casts this thread's 8x8 sub-block of the staged tile at shared address
// `stage`: stores its code words and stages its scales in the shared
// regions at sc_row and sc_col (layouts: staged_scale).  `warp` is the
// warp's index within the 8 warps casting the tile.
// kDirs: 3 = both directions, 1 = row-wise only, 2 = column-wise only.
// kInterior: the whole 128x128 tile lies inside x (no bounds checks).
template <typename T, int MODE, int kDirs, bool kInterior>
__device__ __forceinline__ void block_pass(uint32_t stage, const float* rtab_row, const float* rtab_col,
                                           uint32_t sc_row, uint32_t sc_col, const CastArgs& a, int64_t r0,
                                           int64_t c0, float g_row, float g_col, int warp) {
  constexpr bool kRow = (kDirs & 1) != 0, kCol = (kDirs & 2) != 0;
  const int lane = threadIdx.x & 31;
  const int bx = warp & 1, q = warp >> 1, j = lane & 7, i = lane >> 3;
  const int trow = 32 * q + 8 * i;   // first tile row of the sub-block
  const int tcol = 64 * bx + 8 * j;  // first tile column
  Sub<T> s;
  load_sub<T>(stage, bx, trow, j, s);

  // Output cursors: codes of row k at prow + k * srow, of column c at
  // pcol + c * scol.  Outside x (edge tiles only) the stores are predicated
  // off: bit k of row_ok / col_ok.
  const int64_t M = a.M, N = a.N, y0 = r0 + trow, x0 = c0 + tcol;
  const int64_t srow = N / 2, scol = M / 2;
  uint8_t* prow = kRow ? a.data_row + y0 * srow + x0 / 2 : nullptr;
  uint8_t* pcol = kCol ? a.data_col + x0 * scol + y0 / 2 : nullptr;
  uint32_t row_ok = 0xFFu, col_ok = 0xFFu;
  if (!kInterior) {
    const int64_t rows_in = M - y0, cols_in = N - x0;
    const uint32_t rk = rows_in >= 8 ? 0xFFu : (rows_in <= 0 ? 0u : (1u << rows_in) - 1u);
    const uint32_t ck = cols_in >= 8 ? 0xFFu : (cols_in <= 0 ? 0u : (1u << cols_in) - 1u);
    row_ok = cols_in > 0 ? rk : 0u;
    col_ok = rows_in > 0 ? ck : 0u;
  }
  auto put_row = [&](int k, uint32_t w) {
    if (kInterior)
      st_cs_u32(prow, w);
    else
      st_cs_u32_if(prow, w, (row_ok >> k) & 1u);
    prow += srow;
  };
  auto put_col = [&](int c, uint32_t w) {
    if (kInterior)
      st_cs_u32(pcol, w);
    else
      st_cs_u32_if(pcol, w, (col_ok >> c) & 1u);
    pcol += scol;
  };
  // The first of the two lanes of a 1x16 row block (j even) stages its rows'
  // scales, the first of the two of a 16x1 column block (i even) its
  // columns' scales; in 2D the first of the four lanes of a 16x16 tile.
  const bool stage_row = (j & 1) == 0, stage_col = (i & 1) == 0;

  if constexpr (MODE == kCast2D) {
    const float m = tile_max<T>(s);
    const uint32_t sr = block_scale(m, g_row);
    const uint32_t sc = (g_col == g_row) ? sr : block_scale(m, g_col);
    const float rr = rtab_row[sr], rc = rtab_col[sc];
    uint32_t wc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t wr = encode_row<T>(s, k, kRow ? rr : rc);
      if (kRow) put_row(k, wr);
      if (kCol) wc[k] = (!kRow || rc == rr) ? wr : encode_row<T>(s, k, rc);
    }
    if (kCol) {
      transpose_nibbles8x8(wc);
#pragma unroll
      for (int c = 0; c < 8; ++c) put_col(c, wc[c]);
    }
    if (stage_row && stage_col) {
      if (kRow) sts_u8(sc_row + (uint32_t)((trow >> 4) * 8 + (tcol >> 4)), sr);
      if (kCol) sts_u8(sc_col + (uint32_t)((tcol >> 4) * 8 + (trow >> 4)), sc);
    }
  } else {
    // 1D: row blocks 1x16 (lanes l, l^1), column blocks 16x1 (lanes l, l^8).
    if (kRow) {
      uint32_t packed[2] = {0u, 0u};  // byte k: scale of row trow + k
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float m0, m1;
        if constexpr (sizeof(T) == 2) {
          const uint32_t pr = row_pair_max(s, t);
          m0 = bf16_lo(pr);
          m1 = bf16_hi(pr);
        } else {
          m0 = row_max_f32(s, 2 * t);
          m1 = row_max_f32(s, 2 * t + 1);
        }
        const uint32_t s01 = block_scale2(m0, m1, g_row), s0 = s01 & 0xFFu, s1 = s01 >> 8;
        put_row(2 * t, encode_row<T>(s, 2 * t, rtab_row[s0]));
        put_row(2 * t + 1, encode_row<T>(s, 2 * t + 1, rtab_row[s1]));
        packed[t >> 1] |= (s0 | (s1 << 8)) << (16 * (t & 1));
      }
      if (stage_row) sts_v2(sc_row + (uint32_t)((tcol >> 4) * kScPitchRow + trow), packed[0], packed[1]);
    }
    if (kCol) {
      uint32_t packed[2] = {0u, 0u};  // byte c: scale of column tcol + c
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        float m0, m1;
        if constexpr (sizeof(T) == 2) {
          const uint32_t pc = col_pair_max(s, p);
          m0 = bf16_lo(pc);
          m1 = bf16_hi(pc);
        } else {
          m0 = col_max_f32(s, 2 * p);
          m1 = col_max_f32(s, 2 * p + 1);
        }
        const uint32_t s01 = block_scale2(m0, m1, g_col), s0 = s01 & 0xFFu, s1 = s01 >> 8;
        put_col(2 * p, encode_col<T>(s, 2 * p, rtab_col[s0]));
        put_col(2 * p + 1, encode_col<T>(s, 2 * p + 1, rtab_col[s1]));
        packed[p >> 1] |= (s0 | (s1 << 8)) << (16 * (p & 1));
      }
      if (stage_col) sts_v2(sc_col + (uint32_t)((trow >> 4) * kScPitchCol + tcol), packed[0], packed[1]);
    }
  }
}

// block_pass for the directions and tile position at hand.
template <typename T, int MODE>
__device__ __forceinline__ void block_pass_any(uint32_t stage, const float* rtab_row, const float* rtab_col,
                                               uint32_t sc_row, uint32_t sc_col, const CastArgs& a, int64_t r0,
                                               int64_t c0, float g_row, float g_col, bool do_row, bool do_col,
                                               int warp) {
  const bool interior = (r0 + kTile <= a.M) && (c0 + kTile <= a.N);
  if (do_row && do_col) {
    if (interior)
      block_pass<T, MODE, 3, true>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
    else
      block_pass<T, MODE, 3, false>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
  } else if (do_row) {
    if (interior)
      block_pass<T, MODE, 1, true>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
    else
      block_pass<T, MODE, 1, false>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
  } else if (do_col) {
    if (interior)
      block_pass<T, MODE, 2, true>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
    else
      block_pass<T, MODE, 2, false>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
  }
}

// ---------------------------------------------------------------------------
// Wide sub-tiles (BF16): four warps cast a 128x128 tile, warp w owning the
// 64x64 quarter at rows 64 (w >> 1), columns 64 (w & 1) (box w & 1); lane l
// owns 8 rows x 16 columns: rows 64 (w >> 1) + 8 i, columns 64 (w & 1) + 16 j,
// i = l >> 2, j = l & 3.  Every code store of a warp then fills whole 32-byte
// sectors: a row-wise store writes 16 columns (8 bytes) per lane and the four
// lanes of a row are adjacent; a column-wise store writes 8 rows (4 bytes)
// per lane and the eight lanes of a column are adjacent.  A 1x16 row block
// lies inside one lane; a 16x1 column block and a 16x16 tile span lanes l
// and l ^ 4.
//
// The 16 columns are two 16-byte chunks (2j and 2j + 1 of the 128-byte row
// of box w & 1).  Lanes with odd i load them in the other order ("A" is
// chunk 2j + (i & 1), "B" the other one), so that each quarter-warp of a
// 16-byte shared load touches eight different chunks (no bank conflicts).
// ---------------------------------------------------------------------------
struct SubW {
  uint32_t a[8][4], b[8][4];  // [row k][BF16 pair]: halves A and B
};

// Returns a token computed from one word of every load: each 16-byte load
// writes its four registers when it completes, so anything that depends on
// the token comes after all sixteen loads have read shared memory.
__device__ __forceinline__ uint32_t load_sub_w(uint32_t stage, int wc, int trow, int j, int par, SubW& s) {
  const uint32_t base = stage + wc * kBoxBytes + trow * 128;
  const uint32_t ca = (uint32_t)(2 * j + par) << 4, cb = ca ^ 16u;
  uint32_t tok = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 va = lds128(base + 128 * k + (ca ^ (k << 4)));
    const uint4 vb = lds128(base + 128 * k + (cb ^ (k << 4)));
    s.a[k][0] = va.x; s.a[k][1] = va.y; s.a[k][2] = va.z; s.a[k][3] = va.w;
    s.b[k][0] = vb.x; s.b[k][1] = vb.y; s.b[k][2] = vb.z; s.b[k][3] = vb.w;
    tok ^= va.x ^ vb.x;
  }
  return tok;
}

// Codes of row k of one half (8 values), v0 in the low nibble.
__device__ __forceinline__ uint32_t encode_half_row(const uint32_t (&w)[4], float r) {
  return encode8(bf16_lo(w[0]), bf16_hi(w[0]), bf16_lo(w[1]), bf16_hi(w[1]), bf16_lo(w[2]), bf16_hi(w[2]),
                 bf16_lo(w[3]), bf16_hi(w[3]), r);
}
// Codes of column c (0..7) of one half over the 8 rows, row 0 in the low nibble.
__device__ __forceinline__ uint32_t encode_half_col(const uint32_t (&w)[8][4], int c, float r) {
  const int p = c >> 1;
  if (c & 1)
    return encode8(bf16_hi(w[0][p]), bf16_hi(w[1][p]), bf16_hi(w[2][p]), bf16_hi(w[3][p]), bf16_hi(w[4][p]),
                   bf16_hi(w[5][p]), bf16_hi(w[6][p]), bf16_hi(w[7][p]), r);
  return encode8(bf16_lo(w[0][p]), bf16_lo(w[1][p]), bf16_lo(w[2][p]), bf16_lo(w[3][p]), bf16_lo(w[4][p]),
                 bf16_lo(w[5][p]), bf16_lo(w[6][p]), bf16_lo(w[7][p]), r);
}
// Packed (max|.| of row k0, of row k1) over both halves (16 columns).
__device__ __forceinline__ uint32_t row_pair_max_w(const SubW& s, int k0, int k1) {
  const uint32_t x = xsa(xsa(xsa(s.a[k0][0], s.a[k0][1]), xsa(s.a[k0][2], s.a[k0][3])),
                         xsa(xsa(s.b[k0][0], s.b[k0][1]), xsa(s.b[k0][2], s.b[k0][3])));
  const uint32_t y = xsa(xsa(xsa(s.a[k1][0], s.a[k1][1]), xsa(s.a[k1][2], s.a[k1][3])),
                         xsa(xsa(s.b[k1][0], s.b[k1][1]), xsa(s.b[k1][2], s.b[k1][3])));
  return xsa_pairs(x, y) & 0x7FFF7FFFu;
}
// Packed (max|.| of column 2p, of column 2p+1) of one half over its 8 rows.
__device__ __forceinline__ uint32_t col_pair_acc_w(const uint32_t (&w)[8][4], int p) {
  return xsa(xsa(xsa(w[0][p], w[1][p]), xsa(w[2][p], w[3][p])), xsa(xsa(w[4][p], w[5][p]), xsa(w[6][p], w[7][p])));
}

// No-op stage hooks (see wide_pass).
struct NoHooks {
  __device__ __forceinline__ void data_done(uint32_t) const {}
  __device__ __forceinline__ void scale_wait() const {}
  __device__ __forceinline__ void scales_staged() const {}
  __device__ __forceinline__ const uint16_t* tile_max() const { return nullptr; }
};

// 2D: max|x| of the 16x16 tile this lane's wide sub-tile belongs to (this
// lane's 128 values and lane l ^ 4's), as a packed BF16 pair with both
// halves non-negative; `acc_out` gets the lane's own packed maximum.
__device__ __forceinline__ float wide_tile_max(const uint32_t (&a)[8][4], const uint32_t (&b)[8][4],
                                               uint32_t& acc_out) {
  uint32_t acc = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    acc = xsa(acc, xsa(xsa(xsa(a[k][0], a[k][1]), xsa(a[k][2], a[k][3])),
                       xsa(xsa(b[k][0], b[k][1]), xsa(b[k][2], b[k][3]))));
  acc &= 0x7FFF7FFFu;
  acc_out = acc;
  const float m = fmaxf(bf16_lo(acc), bf16_hi(acc));
  return fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
}

// Byte offset, in a tile's staged atoms of the 128x4 layout, of the word of
// scale row `r` (0..127: a tile row for row-wise scales, a tile column for
// column-wise ones) in atom `h` (0, 1: column blocks 4h..4h+3 of that row):
// 16-byte line r & 31, word r >> 5.
__device__ __forceinline__ uint32_t stage_swz_offset(int r, int h) {
  return (uint32_t)(h * 512 + (r & 31) * 16 + (r >> 5) * 4);
}

// Casts this lane's 8x16 sub-tile (wide mapping) of the staged tile at shared
// address `stage`: stores its codes and stages its scales (staged_scale
// layouts) at sc_row / sc_col.  `warp` is the warp's index (0..3) among the
// four casting the tile.  Both directions share the global encode scale g
// (the amax is per tensor) and its table rtab[s] = encode factor of scale
// code s.  kDirs: 3 both directions, 1 row-wise, 2 column-wise.
// kInterior: the tile lies inside x.  The warp calls
// hooks.data_done(token) once its reads of the staged tile have completed
// (token is computed from every word it read, so anything that depends on
// it comes after those reads; the caller can then reuse the stage), and
// hooks.scale_wait() before its first write to sc_row / sc_col.  In 2D,
// hooks.tile_max() may give the tile's 16x16 maxima (BF16 bits, [ty][tx])
// found while the tile was first read; else they are computed here.
// kSwz (tiles inside x, 128x4 layout): the scales are staged as the tile's
// two 512-byte atoms per direction, byte for byte as they are stored (see
// stage_swz_offset), so that one bulk copy per direction writes them; in 2D
// the warp calls hooks.scales_staged() once its share is staged, before it
// computes and stores any code (the bulk copy then runs meanwhile, and its
// proxy fence waits on the staging stores only).
template <int MODE, int kDirs, bool kInterior, bool kSwz = false, class Hooks = NoHooks>
__device__ __forceinline__ void wide_pass(uint32_t stage, const float* rtab, uint32_t sc_row, uint32_t sc_col,
                                          const CastArgs& a, int64_t r0, int64_t c0, float g, int warp,
                                          const Hooks& hooks = Hooks()) {
  constexpr bool kRow = (kDirs & 1) != 0, kCol = (kDirs & 2) != 0;
  const int lane = threadIdx.x & 31;
  const int wr = warp >> 1, wc = warp & 1, i = lane >> 2, j = lane & 3, par = i & 1;
  const int trow = 64 * wr + 8 * i, tcol = 64 * wc + 16 * j;
  SubW s;
  const uint32_t ltok = load_sub_w(stage, wc, trow, j, par, s);

  const int64_t M = a.M, N = a.N, y0 = r0 + trow, x0 = c0 + tcol;
  const int64_t srow = N / 2, scol = M / 2;
  uint8_t* prow = kRow ? a.data_row + y0 * srow + x0 / 2 : nullptr;
  uint8_t* pcol = kCol ? a.data_col + x0 * scol + y0 / 2 : nullptr;
  // Outside x (edge tiles only): N % 16 == 0, so the 16 columns are all in
  // or all out; column-wise output needs M % 16 == 0, so then the 8 rows
  // are too; row-wise alone allows any M (per-row predicates).
  const bool cols_in = kInterior || x0 < N;
  const bool rows_in = kInterior || y0 < M;
  auto put_row = [&](int k, uint32_t wa, uint32_t wb) {
    const uint32_t lo = par ? wb : wa, hi = par ? wa : wb;
    if (kInterior)
      st_cs_v2(prow + k * srow, lo, hi);
    else
      st_cs_v2_if(prow + k * srow, lo, hi, cols_in && y0 + k < M);
  };
  // column cc (0..15) of the lane's 16; half A holds columns 8 par .. 8 par + 7
  auto put_col = [&](int cc, uint32_t w) {
    if (kInterior)
      st_cs_u32(pcol + cc * scol, w);
    else
      st_cs_u32_if(pcol + cc * scol, w, (cols_in && rows_in) ? 1u : 0u);
  };

  if constexpr (MODE == kCast2D) {
    const uint16_t* pre = hooks.tile_max();
    float m;
    if (pre != nullptr) {
      m = __uint_as_float((uint32_t)pre[(trow >> 4) * 8 + (tcol >> 4)] << 16);
      hooks.data_done(ltok);  // the loads are complete: the stage may be refilled
    } else {
      uint32_t acc;
      m = wide_tile_max(s.a, s.b, acc);
      hooks.data_done(acc);  // every word of the sub-tile is in acc
    }
    // one scale and one set of codes serve both directions (the column-wise
    // codes are the row-wise ones transposed)
    const uint32_t sb = block_scale(m, g);
    const float rf = rtab[sb];
    // the scales first, so that their write-back overlaps the codes
    if constexpr (kSwz) {
      // the four column blocks of a row (lanes j) and the four row blocks of
      // a column (lanes i >> 1) gathered into the 4-byte word they share
      uint32_t wrow = sb << (8 * j), wcol = sb << (8 * (i >> 1));
      wrow |= __shfl_xor_sync(0xFFFFFFFFu, wrow, 1);
      wrow |= __shfl_xor_sync(0xFFFFFFFFu, wrow, 2);
      wcol |= __shfl_xor_sync(0xFFFFFFFFu, wcol, 8);
      wcol |= __shfl_xor_sync(0xFFFFFFFFu, wcol, 16);
      hooks.scale_wait();
#pragma unroll
      for (int t = 0; t < 2; ++t) {  // rows trow + 2j + t; columns tcol + 2i + t
        if (kRow) sts_u32(sc_row + stage_swz_offset(trow + 2 * j + t, tcol >> 6), wrow);
        if (kCol) sts_u32(sc_col + stage_swz_offset(tcol + 2 * i + t, trow >> 6), wcol);
      }
      hooks.scales_staged();
    } else {
      hooks.scale_wait();
      if (par == 0) {
        if (kRow) sts_u8(sc_row + (uint32_t)((trow >> 4) * 8 + (tcol >> 4)), sb);
        if (kCol) sts_u8(sc_col + (uint32_t)((tcol >> 4) * 8 + (trow >> 4)), sb);
      }
    }
    uint32_t ca[8], cb[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t wa = encode_half_row(s.a[k], rf);
      const uint32_t wb = encode_half_row(s.b[k], rf);
      if (kRow) put_row(k, wa, wb);
      ca[k] = wa;
      cb[k] = wb;
    }
    if (kCol) {
      transpose_nibbles8x8(ca);
      transpose_nibbles8x8(cb);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        put_col(c, par ? cb[c] : ca[c]);
        put_col(8 + c, par ? ca[c] : cb[c]);
      }
    }
  } else {
    // column pass first, then the row pass: only the data stay live between
    // them.  Both directions: the column scales are staged after the row
    // pass, so that the sub-tile's data are released (hooks.data_done)
    // before the warp waits for the scale region (hooks.scale_wait), as on
    // every other path.
    uint32_t col_pl[2] = {0u, 0u}, col_pr[2] = {0u, 0u};
    // lanes l and l ^ 4 hold the same column-block scales: the lanes with
    // par == 0 stage them (byte c of left / right: column tcol + c / + 8 + c)
    auto stage_col = [&] {
      if constexpr (kSwz) {
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const uint32_t w = (cc < 8 ? col_pl : col_pr)[(cc & 7) >> 2];
          sts_u8(sc_col + stage_swz_offset(tcol + cc, trow >> 6) + ((trow >> 4) & 3), w >> (8 * (cc & 3)));
        }
      } else {
        sts_v4(sc_col + (uint32_t)((trow >> 4) * kScPitchCol + tcol), col_pl[0], col_pl[1], col_pr[0], col_pr[1]);
      }
    };
    if (kCol) {
      // column blocks span lanes l and l ^ 4, whose halves A are the other
      // side of the 16 columns: combine left with left, right with right
      uint32_t pl[2] = {0u, 0u}, pr[2] = {0u, 0u};  // byte c: scale of left / right column c
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t xa = col_pair_acc_w(s.a, p), xb = col_pair_acc_w(s.b, p);
        uint32_t ml = par ? xb : xa, mr = par ? xa : xb;
        ml = xsa(ml, __shfl_xor_sync(0xFFFFFFFFu, ml, 4)) & 0x7FFF7FFFu;
        mr = xsa(mr, __shfl_xor_sync(0xFFFFFFFFu, mr, 4)) & 0x7FFF7FFFu;
        const uint32_t sl = block_scale2(bf16_lo(ml), bf16_hi(ml), g), sr = block_scale2(bf16_lo(mr), bf16_hi(mr), g);
        const uint32_t sl0 = sl & 0xFFu, sl1 = sl >> 8, sr0 = sr & 0xFFu, sr1 = sr >> 8;  // columns 2p, 2p + 1
        const float fl0 = rtab[sl0], fl1 = rtab[sl1], fr0 = rtab[sr0], fr1 = rtab[sr1];
        const uint32_t wa0 = encode_half_col(s.a, 2 * p, par ? fr0 : fl0);
        const uint32_t wa1 = encode_half_col(s.a, 2 * p + 1, par ? fr1 : fl1);
        const uint32_t wb0 = encode_half_col(s.b, 2 * p, par ? fl0 : fr0);
        const uint32_t wb1 = encode_half_col(s.b, 2 * p + 1, par ? fl1 : fr1);
        put_col(2 * p, par ? wb0 : wa0);
        put_col(2 * p + 1, par ? wb1 : wa1);
        put_col(8 + 2 * p, par ? wa0 : wb0);
        put_col(8 + 2 * p + 1, par ? wa1 : wb1);
        pl[p >> 1] |= sl << (16 * (p & 1));
        pr[p >> 1] |= sr << (16 * (p & 1));
      }
      col_pl[0] = pl[0]; col_pl[1] = pl[1]; col_pr[0] = pr[0]; col_pr[1] = pr[1];
      if (!kRow) {
        hooks.data_done(pl[0] ^ pl[1] ^ pr[0] ^ pr[1]);  // scales of every column
        hooks.scale_wait();
        if (par == 0) stage_col();
      }
    }
    if (kRow) {
      // with both directions, re-read the sub-tile (still staged): keeping
      // its 64 data registers live through the column pass exceeds the
      // register budget
      if (kCol) load_sub_w(stage, wc, trow, j, par, s);
      uint32_t packed[2] = {0u, 0u};  // byte k: scale of row trow + k
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const uint32_t pr = row_pair_max_w(s, 2 * t, 2 * t + 1);
        const uint32_t s01 = block_scale2(bf16_lo(pr), bf16_hi(pr), g), s0 = s01 & 0xFFu, s1 = s01 >> 8;
        const float f0 = rtab[s0], f1 = rtab[s1];
        put_row(2 * t, encode_half_row(s.a[2 * t], f0), encode_half_row(s.b[2 * t], f0));
        put_row(2 * t + 1, encode_half_row(s.a[2 * t + 1], f1), encode_half_row(s.b[2 * t + 1], f1));
        packed[t >> 1] |= s01 << (16 * (t & 1));
      }
      hooks.data_done(packed[0] ^ packed[1]);  // scales of every row
      hooks.scale_wait();
      if (kCol && par == 0) stage_col();
      if constexpr (kSwz) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          sts_u8(sc_row + stage_swz_offset(trow + k, tcol >> 6) + j, packed[k >> 2] >> (8 * (k & 3)));
      } else {
        sts_v2(sc_row + (uint32_t)((tcol >> 4) * kScPitchRow + trow), packed[0], packed[1]);
      }
    }
    if constexpr (kSwz) hooks.scales_staged();
  }
}

// wide_pass for the directions and tile position at hand; kSwz: scales
// staged in the 128x4 layout's byte order (every tile inside x).
template <int MODE, bool kSwz = false, class Hooks = NoHooks>
__device__ __forceinline__ void wide_pass_any(uint32_t stage, const float* rtab, uint32_t sc_row, uint32_t sc_col,
                                              const CastArgs& a, int64_t r0, int64_t c0, float g, bool do_row,
                                              bool do_col, int warp, const Hooks& h = Hooks()) {
  if constexpr (kSwz) {
    if (do_row && do_col)
      wide_pass<MODE, 3, true, true>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
    else if (do_row)
      wide_pass<MODE, 1, true, true>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
    else if (do_col)
      wide_pass<MODE, 2, true, true>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
    return;
  }
  const bool interior = (r0 + kTile <= a.M) && (c0 + kTile <= a.N);
  if (do_row && do_col) {
    if (interior)
      wide_pass<MODE, 3, true>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
    else
      wide_pass<MODE, 3, false>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
  } else if (do_row) {
    if (interior)
      wide_pass<MODE, 1, true>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
    else
      wide_pass<MODE, 1, false>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
  } else if (do_col) {
    if (interior)
      wide_pass<MODE, 2, true>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
    else
      wide_pass<MODE, 2, false>(stage, rtab, sc_row, sc_col, a, r0, c0, g, warp, h);
  }
}

// Stores one direction's staged scales (layout: staged_scale<MODE, kColDir>)
// for tile rows R0 .. R0 + 127 and scale columns C0 .. C0 + 7 of an R x C
// scale matrix; t = 0..127.
template <int MODE, bool kColDir>
__device__ __forceinline__ void store_scale_tile(const uint8_t* s, uint8_t* out, int64_t R0, int64_t C0, int64_t R,
                                                 int64_t C, bool swizzled, int t) {
  if (swizzled) {
    // Two 512-byte tiles of the 128x4 layout, contiguous (R, C aligned):
    // 16-byte line L of tile h holds rows L, L+32, L+64, L+96, 4 scales each.
    if (t >= 64) return;
    const int h = t >> 5, L = t & 31;
    uint32_t w[4];
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int r = 32 * qq + L;
      if constexpr (MODE == kCast2D) {
        w[qq] = *reinterpret_cast<const uint32_t*>(s + (r >> 4) * 8 + 4 * h);
      } else {
        w[qq] = staged_scale<MODE, kColDir>(s, r, 4 * h) | (staged_scale<MODE, kColDir>(s, r, 4 * h + 1) << 8) |
                (staged_scale<MODE, kColDir>(s, r, 4 * h + 2) << 16) |
                (staged_scale<MODE, kColDir>(s, r, 4 * h + 3) << 24);
      }
    }
    uint8_t* base = out + ((R0 >> 7) * (C >> 2) + (C0 >> 2) + h) * 512 + L * 16;
    st_cs_v4(base, w[0], w[1], w[2], w[3]);
  } else {
    const int64_t r = R0 + t;
    if (r >= R) return;
    const int64_t n = (C - C0) < 8 ? (C - C0) : 8;
    if (n <= 0) return;
    uint8_t* p = out + r * C + C0;
    uint32_t v[2];
    if constexpr (MODE == kCast2D) {
      const uint2 u = *reinterpret_cast<const uint2*>(s + (t >> 4) * 8);
      v[0] = u.x;
      v[1] = u.y;
    } else {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        v[hh] = staged_scale<MODE, kColDir>(s, t, 4 * hh) | (staged_scale<MODE, kColDir>(s, t, 4 * hh + 1) << 8) |
                (staged_scale<MODE, kColDir>(s, t, 4 * hh + 2) << 16) |
                (staged_scale<MODE, kColDir>(s, t, 4 * hh + 3) << 24);
    }
    if (n == 8 && (reinterpret_cast<uintptr_t>(p) & 7) == 0) {
      st_cs_v2(p, v[0], v[1]);
    } else {
      for (int b = 0; b < n; ++b) st_cs_u8(p + b, v[b >> 2] >> (8 * (b & 3)));
    }
  }
}

}  // namespace tile
}  // namespace nvfp4
