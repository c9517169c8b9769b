// sr.cu -- NVFP4 quantize with stochastically rounded E2M1 codes ("Fuse NVFP4
// scale swizzling on SM120 and SM121", Tests: stochastic rounding is one axis
// of the comparisons).  The random numbers are an input: one byte per element
// of x, used by the row-wise and the column-wise code of that element.  Block
// scales, the amax and the layouts are those of the plain cast; only the
// rounding of each product p = x * r to E2M1 changes: between neighbouring
// magnitudes lo <= |p| < hi the magnitude becomes hi iff
// byte < 256 (|p| - lo) / (hi - lo), decided exactly by the carry form of
// e2m1_sr (common.cuh): an offset made from the byte is added to the bits of
// |p|, and the carry into the kept bit is the decision.
//
// The kernel is the two-pass cast (TMA-staged 128x128 tiles, persistent CTAs
// in reverse tile order after the amax kernel) with the 8x8 sub-block mapping
// of tile_ops.cuh.  Each stage holds the x tile and, beside it, the tile's
// 128 x 128 random bytes (one more TMA box on the same barrier); each thread
// reads its sub-block's 64 bytes from there once, for both directions.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "sr.h"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace {

using namespace tile;

constexpr int kSThreads = 256;

// prmt.b32 with the selector's high bit per byte: that byte of the result is
// the sign bit of the selected input byte, replicated.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Bit 4c + 3 set where column c of row k of the sub-block is negative: the
// eight sign bits moved to where the codes of a row keep theirs.
template <typename T>
__device__ __forceinline__ uint32_t sign_nibbles(const Sub<T>& s, int k) {
  uint32_t even, odd;  // byte i: the sign of column 2i / 2i + 1, replicated
  if constexpr (sizeof(T) == 2) {
    const uint32_t p = prmt(s.w[k][0], s.w[k][1], 0xFBD9u);  // columns 0, 2, 1, 3
    const uint32_t q = prmt(s.w[k][2], s.w[k][3], 0xFBD9u);  // columns 4, 6, 5, 7
    even = prmt(p, q, 0x5410u);
    odd = prmt(p, q, 0x7632u);
  } else {
    even = prmt(prmt(s.w[k][0], s.w[k][2], 0xFBFBu), prmt(s.w[k][4], s.w[k][6], 0xFBFBu), 0x5410u);
    odd = prmt(prmt(s.w[k][1], s.w[k][3], 0xFBFBu), prmt(s.w[k][5], s.w[k][7], 0xFBFBu), 0x5410u);
  }
  return ((even & 0x0F0F0F0Fu) | (odd & 0xF0F0F0F0u)) & 0x88888888u;
}

// Packing eight codes-plus-252 four bits apart and subtracting this once
// leaves the eight codes (the sums wrap mod 2^32, which the subtraction
// undoes exactly).
constexpr uint32_t kCode252x8 = 252u * 0x11111111u;

// Codes of row k of the sub-block (column c in nibble c) times the factor
// of column c, fr[c] (1D column-wise: the column's factor; otherwise one
// factor for the row), with the row's random bytes rb.
template <typename T>
__device__ __forceinline__ uint32_t sr_row_word(const Sub<T>& s, int k, const float (&f)[8], const uint2& rb,
                                                uint32_t sgn) {
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    acc += sr_code252(__fmul_rn(fabsf(s.v(k, c)), f[c]), sr_offset_w(c < 4 ? rb.x : rb.y, c & 3)) << (4 * c);
  return (acc - kCode252x8) | sgn;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// A stage: the x tile, then the tile's random bytes (128 rows of 128 bytes,
// 128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r & 7)).
constexpr uint32_t kRbTileBytes = 128 * 128;
template <typename T>
__host__ __device__ constexpr uint32_t sr_stage_bytes() {
  return (uint32_t)tile_bytes<T>() + kRbTileBytes;
}
// Stages per CTA: two (BF16: two CTAs of 2 x 48 KB per SM; FP32: one CTA of
// 2 x 80 KB).
template <typename T, int MODE>
__host__ __device__ constexpr int sr_stages() {
  return 2;
}
// stages | 2 encode-factor tables | 2 x 2 staged scale regions | barriers | flag
template <typename T, int MODE>
__host__ __device__ constexpr size_t sr_smem_bytes() {
  return 1024 + (size_t)sr_stages<T, MODE>() * sr_stage_bytes<T>() + 2 * 128 * 4 + 4 * kScRegion +
         8 * sr_stages<T, MODE>() + 16;
}

// The sub-block pass of tile_ops.cuh (same mapping, scales, staging and
// stores) with stochastically rounded codes.
template <typename T, int MODE, int kDirs, bool kInterior>
__device__ __forceinline__ void sr_pass(uint32_t stage, const float* rtab_row, const float* rtab_col,
                                        uint32_t sc_row, uint32_t sc_col, const CastArgs& a, int64_t r0, int64_t c0,
                                        float g_row, float g_col, int warp) {
  constexpr bool kRow = (kDirs & 1) != 0, kCol = (kDirs & 2) != 0;
  const int lane = threadIdx.x & 31;
  const int bx = warp & 1, q = warp >> 1, j = lane & 7, i = lane >> 3;
  const int trow = 32 * q + 8 * i;
  const int tcol = 64 * bx + 8 * j;
  Sub<T> s;
  load_sub<T>(stage, bx, trow, j, s);

  const int64_t M = a.M, N = a.N, y0 = r0 + trow, x0 = c0 + tcol;
  // the sub-block's random bytes: row k at rb[k], column c in byte c;
  // outside x they are the zero fill, unused
  uint2 rb[8];
  const uint32_t rstage = stage + (uint32_t)tile_bytes<T>();
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int r = trow + k;
    rb[k] = lds64(rstage + (uint32_t)(r * 128 + ((((tcol >> 4) ^ (r & 7)) << 4) | (tcol & 8))));
  }

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
  const bool stage_row = (j & 1) == 0, stage_col = (i & 1) == 0;

  // Every code of a row is made in row order, the column-wise ones too (with
  // their columns' factors), and the column-wise words are transposed at the
  // end; the signs of a row serve both directions.
  uint32_t wc[8];
  if constexpr (MODE == kCast2D) {
    const float m = tile_max<T>(s);
    const uint32_t sr = block_scale(m, g_row);
    const uint32_t sc = (g_col == g_row) ? sr : block_scale(m, g_col);
    const float rr = rtab_row[sr], rc = rtab_col[sc];
    float fr[8], fc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      fr[c] = kRow ? rr : rc;
      fc[c] = rc;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t sgn = sign_nibbles(s, k);
      const uint32_t wr = sr_row_word(s, k, fr, rb[k], sgn);
      if (kRow) put_row(k, wr);
      // an element keeps its byte in both directions, so with one factor the
      // column codes are the transposed row codes
      if (kCol) wc[k] = (!kRow || rc == rr) ? wr : sr_row_word(s, k, fc, rb[k], sgn);
    }
    if (stage_row && stage_col) {
      if (kRow) sts_u8(sc_row + (uint32_t)((trow >> 4) * 8 + (tcol >> 4)), sr);
      if (kCol) sts_u8(sc_col + (uint32_t)((tcol >> 4) * 8 + (trow >> 4)), sc);
    }
  } else {
    float fr[8], fc[8];  // factors of the sub-block's rows / columns
    if (kRow) {
      uint32_t packed[2] = {0u, 0u};
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
        fr[2 * t] = rtab_row[s0];
        fr[2 * t + 1] = rtab_row[s1];
        packed[t >> 1] |= (s0 | (s1 << 8)) << (16 * (t & 1));
      }
      if (stage_row) sts_v2(sc_row + (uint32_t)((tcol >> 4) * kScPitchRow + trow), packed[0], packed[1]);
    }
    if (kCol) {
      uint32_t packed[2] = {0u, 0u};
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
        fc[2 * p] = rtab_col[s0];
        fc[2 * p + 1] = rtab_col[s1];
        packed[p >> 1] |= (s0 | (s1 << 8)) << (16 * (p & 1));
      }
      if (stage_col) sts_v2(sc_col + (uint32_t)((trow >> 4) * kScPitchCol + tcol), packed[0], packed[1]);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t sgn = sign_nibbles(s, k);
      if (kRow) {
        float f[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) f[c] = fr[k];
        put_row(k, sr_row_word(s, k, f, rb[k], sgn));
      }
      if (kCol) wc[k] = sr_row_word(s, k, fc, rb[k], sgn);
    }
  }
  if (kCol) {
    transpose_nibbles8x8(wc);
#pragma unroll
    for (int c = 0; c < 8; ++c) put_col(c, wc[c]);
  }
}

template <typename T, int MODE>
__device__ __forceinline__ void sr_pass_any(uint32_t stage, const float* rtab_row, const float* rtab_col,
                                            uint32_t sc_row, uint32_t sc_col, const CastArgs& a, int64_t r0,
                                            int64_t c0, float g_row, float g_col, bool do_row, bool do_col,
                                            int warp) {
  const bool interior = (r0 + kTile <= a.M) && (c0 + kTile <= a.N);
  if (do_row && do_col) {
    if (interior)
      sr_pass<T, MODE, 3, true>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
    else
      sr_pass<T, MODE, 3, false>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
  } else if (do_row) {
    if (interior)
      sr_pass<T, MODE, 1, true>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
    else
      sr_pass<T, MODE, 1, false>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
  } else if (do_col) {
    if (interior)
      sr_pass<T, MODE, 2, true>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
    else
      sr_pass<T, MODE, 2, false>(stage, rtab_row, rtab_col, sc_row, sc_col, a, r0, c0, g_row, g_col, warp);
  }
}

struct SSmem {
  uint8_t* stages;
  float* rtab_row;  // [128]
  float* rtab_col;  // [128]
  uint8_t* sc_row;  // [2][kScRegion]
  uint8_t* sc_col;  // [2][kScRegion]
  uint64_t* bars;   // [kStages]
  int* abort_flag;
};

template <typename T, int MODE>
__device__ __forceinline__ SSmem scarve(uint8_t* raw) {
  SSmem s;
  uint8_t* p = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  s.stages = p;
  p += (size_t)sr_stages<T, MODE>() * sr_stage_bytes<T>();
  s.rtab_row = reinterpret_cast<float*>(p);
  s.rtab_col = s.rtab_row + 128;
  s.sc_row = reinterpret_cast<uint8_t*>(s.rtab_col + 128);
  s.sc_col = s.sc_row + 2 * kScRegion;
  s.bars = reinterpret_cast<uint64_t*>(s.sc_col + 2 * kScRegion);
  s.abort_flag = reinterpret_cast<int*>(s.bars + sr_stages<T, MODE>());
  return s;
}

// CTAs per SM the register budget is set for: two for BF16 (128 registers,
// no spills), one for FP32.
template <typename T, int MODE>
constexpr int sr_min_blocks() {
  return sizeof(T) == 2 ? 2 : 1;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kSThreads, sr_min_blocks<T, MODE>())
    sr_cast_kernel(const __grid_constant__ CUtensorMap tmap, const CastArgs a,
                   const __grid_constant__ CUtensorMap rmap) {
  using C = TileCfg<T>;
  constexpr int S = sr_stages<T, MODE>();
  extern __shared__ uint8_t smem_raw[];
  const SSmem sm = scarve<T, MODE>(smem_raw);
  const int tid = threadIdx.x;
  if (a.noop != nullptr && *a.noop == 1.0f) return;

  const int num_tiles = a.num_tiles;
  const int bid = blockIdx.x, nb = gridDim.x;
  const int my_count = (bid < num_tiles) ? (num_tiles - 1 - bid) / nb + 1 : 0;
  auto tile_of = [&](int k) { return num_tiles - 1 - (bid + k * nb); };

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&sm.bars[s], 1);
    *sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap);
    tma_prefetch_desc(&rmap);
  }
  __syncthreads();
  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int k) {
    const int t = tile_of(k);
    const int tr = t / a.tiles_n, tc = t - tr * a.tiles_n;
    uint8_t* dst = sm.stages + (size_t)(k % S) * sr_stage_bytes<T>();
    uint64_t* bar = &sm.bars[k % S];
    mbar_arrive_expect_tx(bar, sr_stage_bytes<T>());
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_2d(dst + b * kBoxBytes, &tmap, tc * kTile + b * C::kBoxCols, tr * kTile, bar, policy);
    tma_load_2d(dst + tile_bytes<T>(), &rmap, tc * kTile, tr * kTile, bar, policy);
  };
  if (tid == 0)
    for (int k = 0; k < S && k < my_count; ++k) issue(k);

  grid_dependency_wait();  // the amax written by the preceding kernel is visible
  const float g_row = global_encode_scale(a.amax_row ? *a.amax_row : 0.0f);
  const float g_col = global_encode_scale(a.amax_col ? *a.amax_col : 0.0f);
  if (tid < 128)
    sm.rtab_row[tid] = encode_factor((uint32_t)tid, g_row);
  else
    sm.rtab_col[tid - 128] = encode_factor((uint32_t)(tid - 128), g_col);
  __syncthreads();

  const bool do_row = a.rowwise != 0, do_col = a.colwise != 0;
  int k = 0;
  for (; k < my_count; ++k) {
    const int s = k % S;
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&sm.bars[s], (uint32_t)((k / S) & 1), a.status));
    if (!ok) *sm.abort_flag = 1;
    const int t = tile_of(k);
    const int tr = t / a.tiles_n, tc = t - tr * a.tiles_n;
    const int64_t r0 = (int64_t)tr * kTile, c0 = (int64_t)tc * kTile;
    const uint8_t* st = sm.stages + (size_t)s * sr_stage_bytes<T>();
    const int parity = k & 1;
    if (ok)
      sr_pass_any<T, MODE>(smem_u32(st), sm.rtab_row, sm.rtab_col, smem_u32(sm.sc_row + parity * kScRegion),
                           smem_u32(sm.sc_col + parity * kScRegion), a, r0, c0, g_row, g_col, do_row, do_col,
                           tid >> 5);
    __syncthreads();  // stage s fully read; this tile's scales staged
    if (*sm.abort_flag) break;
    if (tid == 0 && k + S < my_count) issue(k + S);
    if (tid < 128) {
      if (do_row)
        store_scale_tile<MODE, false>(sm.sc_row + parity * kScRegion, a.scale_row, r0, c0 / 16, a.M, a.N / 16,
                                      a.swizzled, tid);
    } else if (do_col) {
      store_scale_tile<MODE, true>(sm.sc_col + parity * kScRegion, a.scale_col, c0, r0 / 16, a.N, a.M / 16,
                                   a.swizzled, tid - 128);
    }
  }
  if (k < my_count && tid == 0) {
    // A wait ran out: wait (bounded) for this CTA's copies still in flight
    // before the shared memory is released.
    const int issued = (k + S < my_count) ? k + S : my_count;
    for (int jj = k; jj < issued; ++jj) mbar_wait_bounded(&sm.bars[jj % S], (uint32_t)((jj / S) & 1), a.status);
  }
}

template <typename T, int MODE>
cudaError_t launch_t(const CUtensorMap& map, const CastArgs& a, const CUtensorMap& rmap, bool pdl,
                     const LaunchCtx& ctx) {
  constexpr size_t kSmem = sr_smem_bytes<T, MODE>();
  auto fn = sr_cast_kernel<T, MODE>;
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  // the CTAs per SM that fit (registers, shared memory), at most two
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessorWithFlags(&per_sm, fn, kSThreads, kSmem, cudaOccupancyDefault);
  if (e != cudaSuccess) return e;
  const int cap = ctx.num_sms * (per_sm < 1 ? 1 : (per_sm > 2 ? 2 : per_sm));
  const int grid = a.num_tiles < cap ? a.num_tiles : cap;
  if (grid == 0) return cudaSuccess;
  void* args[] = {(void*)&map, (void*)&a, (void*)&rmap};
  if (pdl) return launch_pdl((const void*)fn, dim3(grid), dim3(kSThreads), kSmem, ctx.stream, args);
  fn<<<grid, kSThreads, kSmem, ctx.stream>>>(map, a, rmap);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cast_sr(const CUtensorMap& map, bool bf16, int mode, CastArgs args, const CUtensorMap& rmap,
                           bool pdl, const LaunchCtx& ctx) {
  const int64_t tiles_m = (args.M + kTile - 1) / kTile, tiles_n = (args.N + kTile - 1) / kTile;
  args.tiles_n = (int)tiles_n;
  args.num_tiles = (int)(tiles_m * tiles_n);
  if (bf16) {
    if (mode == kCast1D) return launch_t<uint16_t, kCast1D>(map, args, rmap, pdl, ctx);
    return launch_t<uint16_t, kCast2D>(map, args, rmap, pdl, ctx);
  }
  if (mode == kCast1D) return launch_t<float, kCast1D>(map, args, rmap, pdl, ctx);
  return launch_t<float, kCast2D>(map, args, rmap, pdl, ctx);
}

}  // namespace nvfp4
