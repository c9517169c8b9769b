// cast.cu -- fused NVFP4 cast with row-wise and column-wise (transposed)
// outputs from one read of each 128x128 tile of x.
//
// Per tile (TMA-loaded into shared memory with the 128-byte swizzle, a
// multi-stage mbarrier pipeline, persistent CTAs walking the tiles in
// reverse so the first ones hit the part of x the amax pass left in L2):
//   row pass:    thread = one row x 64 columns (4 blocks of 1x16); block
//                max, E4M3 scale, codes; 32 bytes of codes per thread.
//   column pass: thread = 2 columns x 32 rows (BF16) or 1 column x 64 rows
//                (FP32); the same per 16x1 block of x, i.e. per 1x16 block
//                of x transposed.  With the random Hadamard transform the
//                16 values of a column block are transformed first.
//   2D:          one scale per 16x16 tile: the row pass reduces the block
//                maxima over the tile's 16 rows (half-warp shuffles) and
//                leaves the tile max in shared memory for the column pass.
// Scales are stored compact or in the cuBLAS 128x4 layout ("Fuse NVFP4
// scale swizzling on SM120 and SM121", Changes: groups of four scales as one
// 32-bit store).  The encode factor g/float(s) comes from a 128-entry table
// per CTA (one IEEE division per E4M3 code instead of one per block).
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;           // tile rows = tile columns (elements)
constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 128 bytes

template <typename T>
struct TileCfg;
template <>
struct TileCfg<uint16_t> {
  static constexpr int kEB = 2, kBoxCols = 64, kBoxes = 2, kStages = 3, kMinBlocks = 2;
};
template <>
struct TileCfg<float> {
  static constexpr int kEB = 4, kBoxCols = 32, kBoxes = 4, kStages = 3, kMinBlocks = 1;
};

template <typename T>
__host__ __device__ constexpr int tile_bytes() {
  return TileCfg<T>::kBoxes * kBoxBytes;
}
template <typename T>
__host__ __device__ constexpr size_t smem_bytes() {
  return 1024 + (size_t)TileCfg<T>::kStages * tile_bytes<T>() + 2 * 128 * 4 + 64 * 4 +
         8 * TileCfg<T>::kStages + 16;
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in box `box` of a
// stage: the TMA 128-byte swizzle XORs the chunk index with row % 8.
__device__ __forceinline__ uint32_t swz(int box, int row, int chunk) {
  return (uint32_t)(box * kBoxBytes + row * 128 + (((chunk ^ row) & 7) << 4));
}

template <typename T>
__device__ __forceinline__ float elem(const uint32_t* w, int i) {
  if constexpr (sizeof(T) == 2)
    return (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
  else
    return __uint_as_float(w[i]);
}

// E4M3 scale code of a block with maximum b under global scale g.
__device__ __forceinline__ uint32_t block_scale(float b, float g) {
  return e4m3_rn_satfinite(__fmul_rn(div6_rn(b), g));
}

// 16 values times r -> two words of 8 E2M1 codes.
__device__ __forceinline__ void encode16(const float* v, float r, uint32_t& lo, uint32_t& hi) {
  lo = e2m1x8(__fmul_rn(v[0], r), __fmul_rn(v[1], r), __fmul_rn(v[2], r), __fmul_rn(v[3], r),
              __fmul_rn(v[4], r), __fmul_rn(v[5], r), __fmul_rn(v[6], r), __fmul_rn(v[7], r));
  hi = e2m1x8(__fmul_rn(v[8], r), __fmul_rn(v[9], r), __fmul_rn(v[10], r), __fmul_rn(v[11], r),
              __fmul_rn(v[12], r), __fmul_rn(v[13], r), __fmul_rn(v[14], r), __fmul_rn(v[15], r));
}

struct Smem {
  uint8_t* stages;
  float* rtab_row;  // [128] encode factor per E4M3 code, row-wise g
  float* rtab_col;  // [128] same, column-wise g
  float* tmax;      // [8][8] 16x16 tile maxima (2D)
  uint64_t* bars;   // [kStages]
  int* abort_flag;
};

template <typename T>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
  Smem s;
  uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~(uintptr_t)1023);
  s.stages = p;
  p += (size_t)TileCfg<T>::kStages * tile_bytes<T>();
  s.rtab_row = reinterpret_cast<float*>(p);
  s.rtab_col = s.rtab_row + 128;
  s.tmax = s.rtab_col + 128;
  s.bars = reinterpret_cast<uint64_t*>(s.tmax + 64);
  s.abort_flag = reinterpret_cast<int*>(s.bars + TileCfg<T>::kStages);
  return s;
}

// ---------------------------------------------------------------------------
// Row pass: thread (rr = tid % 128, h = tid / 128) owns tile row rr, tile
// columns [64h, 64h + 64) = four 1x16 blocks.
// ---------------------------------------------------------------------------
template <typename T, int MODE>
__device__ __forceinline__ void row_pass(const uint8_t* st, const Smem& sm, const CastArgs& a, int64_t r0,
                                         int64_t c0, float g_row) {
  using C = TileCfg<T>;
  const int tid = threadIdx.x;
  const int rr = tid & 127, h = tid >> 7;
  constexpr int kWords = 64 * C::kEB / 4;  // 32 (BF16) or 64 (FP32)
  uint32_t w[kWords];
#pragma unroll
  for (int j = 0; j < kWords / 4; ++j) {
    // BF16: box h, chunks 0..7.  FP32: boxes 2h, 2h+1, chunks 0..7 each.
    const int box = (sizeof(T) == 2) ? h : 2 * h + (j >> 3);
    const uint4 v = *reinterpret_cast<const uint4*>(st + swz(box, rr, j & 7));
    w[4 * j] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
  }
  float b[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(elem<T>(w, 16 * k + i)));
    b[k] = m;
  }
  if constexpr (MODE == kCast2D) {
    // 16x16 tile max: the tile's 16 rows are the 16 lanes of this half-warp.
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) b[k] = fmaxf(b[k], __shfl_xor_sync(0xFFFFFFFFu, b[k], o));
    if ((tid & 15) == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) sm.tmax[(rr >> 4) * 8 + 4 * h + k] = b[k];
    }
  }
  const int64_t y = r0 + rr;
  const int64_t cb = c0 + 64 * h;  // first column of this segment
  if (!a.rowwise || y >= a.M || cb >= a.N) return;
  uint32_t code[8];
  uint32_t scales = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t s = block_scale(b[k], g_row);
    const float r = sm.rtab_row[s];
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = elem<T>(w, 16 * k + i);
    encode16(v, r, code[2 * k], code[2 * k + 1]);
    scales |= s << (8 * k);
  }
  uint8_t* dst = a.data_row + y * (a.N / 2) + cb / 2;
  const int nblk = (cb + 64 <= a.N) ? 4 : (int)((a.N - cb) / 16);
  if (nblk == 4) {
    if (((a.N / 2) & 15) == 0) {
      st_cs_v4(dst, code[0], code[1], code[2], code[3]);
      st_cs_v4(dst + 16, code[4], code[5], code[6], code[7]);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) st_cs_v2(dst + 8 * k, code[2 * k], code[2 * k + 1]);
    }
    store_scales(a.scale_row, y, cb / 16, a.N / 16, a.swizzled, 4, scales);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (k < nblk) {
        st_cs_v2(dst + 8 * k, code[2 * k], code[2 * k + 1]);
        store_scales(a.scale_row, y, cb / 16 + k, a.N / 16, a.swizzled, 1, scales >> (8 * k));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Column pass.  BF16: warp w -> box w % 2, rows 32 (w / 2) .. +32; lane l ->
// tile columns 64 (w % 2) + 2l, +1; two 16-row blocks per column.
// FP32: warp w -> box w % 4, rows 64 (w / 4) .. +64; lane l -> tile column
// 32 (w % 4) + l; four 16-row blocks.
// ---------------------------------------------------------------------------
template <typename T, int MODE>
__device__ __forceinline__ void col_pass(const uint8_t* st, const Smem& sm, const CastArgs& a, int64_t r0,
                                         int64_t c0, float g_col, const float* sgn) {
  using C = TileCfg<T>;
  constexpr int kCols = (sizeof(T) == 2) ? 2 : 1;   // columns per thread
  constexpr int kBlk = (sizeof(T) == 2) ? 2 : 4;    // 16-row blocks per column
  constexpr int kRows = 16 * kBlk;
  constexpr int kWarpsPerBox = 8 / C::kBoxes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int box = warp % C::kBoxes;
  const int rbase = (warp / C::kBoxes) * kRows;  // first tile row
  (void)kWarpsPerBox;
  uint32_t w[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int row = rbase + i;
    w[i] = *reinterpret_cast<const uint32_t*>(st + swz(box, row, lane >> 2) + ((lane & 3) << 2));
  }
  const int64_t rg = r0 + rbase;  // first row of x
#pragma unroll
  for (int cc = 0; cc < kCols; ++cc) {
    const int tcol = box * C::kBoxCols + kCols * lane + cc;  // tile column
    const int64_t x = c0 + tcol;
    uint32_t code[2 * kBlk];
    uint32_t scales = 0;
#pragma unroll
    for (int blk = 0; blk < kBlk; ++blk) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t word = w[16 * blk + i];
        if constexpr (sizeof(T) == 2)
          v[i] = cc ? bf16_hi(word) : bf16_lo(word);
        else
          v[i] = __uint_as_float(word);
      }
      if constexpr (MODE == kCastRHT) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], sgn[i]);
        fwht16(v);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = round_bf16(v[i]);
      }
      float bm;
      if constexpr (MODE == kCast2D) {
        bm = sm.tmax[((rbase >> 4) + blk) * 8 + (tcol >> 4)];
      } else {
        bm = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) bm = fmaxf(bm, fabsf(v[i]));
      }
      const uint32_t s = block_scale(bm, g_col);
      encode16(v, sm.rtab_col[s], code[2 * blk], code[2 * blk + 1]);
      scales |= s << (8 * blk);
    }
    if (!a.colwise || x >= a.N || rg >= a.M) continue;
    uint8_t* dst = a.data_col + x * (a.M / 2) + rg / 2;
    const int nblk = (rg + kRows <= a.M) ? kBlk : (int)((a.M - rg) / 16);
    if (nblk == kBlk) {
      if (((a.M / 2) & 15) == 0) {
#pragma unroll
        for (int q = 0; q < kBlk / 2; ++q)
          st_cs_v4(dst + 16 * q, code[4 * q], code[4 * q + 1], code[4 * q + 2], code[4 * q + 3]);
      } else {
#pragma unroll
        for (int q = 0; q < kBlk; ++q) st_cs_v2(dst + 8 * q, code[2 * q], code[2 * q + 1]);
      }
      store_scales(a.scale_col, x, rg / 16, a.M / 16, a.swizzled, kBlk, scales);
    } else {
#pragma unroll
      for (int q = 0; q < kBlk; ++q) {
        if (q < nblk) {
          st_cs_v2(dst + 8 * q, code[2 * q], code[2 * q + 1]);
          store_scales(a.scale_col, x, rg / 16 + q, a.M / 16, a.swizzled, 1, scales >> (8 * q));
        }
      }
    }
  }
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kThreads, TileCfg<T>::kMinBlocks)
    cast_kernel(const __grid_constant__ CUtensorMap tmap, const CastArgs a) {
  using C = TileCfg<T>;
  extern __shared__ uint8_t smem_raw[];
  const Smem sm = carve<T>(smem_raw);
  const int tid = threadIdx.x;
  if (a.noop != nullptr && *a.noop == 1.0f) return;

  const int num_tiles = a.num_tiles;
  const int bid = blockIdx.x, nb = gridDim.x;
  const int my_count = (bid < num_tiles) ? (num_tiles - 1 - bid) / nb + 1 : 0;
  auto tile_of = [&](int k) { return num_tiles - 1 - (bid + k * nb); };

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) mbar_init(&sm.bars[s], 1);
    *sm.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap);
  }
  __syncthreads();
  const uint64_t policy = l2_policy_evict_first();
  auto issue = [&](int k) {
    const int t = tile_of(k);
    const int tr = t / a.tiles_n, tc = t - tr * a.tiles_n;
    uint8_t* dst = sm.stages + (size_t)(k % C::kStages) * tile_bytes<T>();
    uint64_t* bar = &sm.bars[k % C::kStages];
    mbar_arrive_expect_tx(bar, tile_bytes<T>());
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_2d(dst + b * kBoxBytes, &tmap, tc * kTile + b * C::kBoxCols, tr * kTile, bar, policy);
  };
  // x does not depend on the amax kernel, so the first tiles are requested
  // before waiting for it.
  if (tid == 0)
    for (int k = 0; k < C::kStages && k < my_count; ++k) issue(k);

  grid_dependency_wait();  // the amax written by the preceding kernel is visible
  const float g_row = global_encode_scale(a.amax_row ? *a.amax_row : 0.0f);
  const float g_col = global_encode_scale(a.amax_col ? *a.amax_col : 0.0f);
  if (tid < 128)
    sm.rtab_row[tid] = encode_factor((uint32_t)tid, g_row);
  else
    sm.rtab_col[tid - 128] = encode_factor((uint32_t)(tid - 128), g_col);
  float sgn[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) sgn[i] = ((a.sign_mask >> i) & 1u) ? -0.25f : 0.25f;
  __syncthreads();

  int k = 0;
  for (; k < my_count; ++k) {
    const int s = k % C::kStages;
    // Warp-uniform so that the shuffles of the row pass see whole warps.
    const bool ok =
        __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&sm.bars[s], (uint32_t)((k / C::kStages) & 1), a.status));
    if (!ok) *sm.abort_flag = 1;
    const int t = tile_of(k);
    const int tr = t / a.tiles_n, tc = t - tr * a.tiles_n;
    const int64_t r0 = (int64_t)tr * kTile, c0 = (int64_t)tc * kTile;
    const uint8_t* st = sm.stages + (size_t)s * tile_bytes<T>();
    if (ok && (a.rowwise || MODE == kCast2D)) row_pass<T, MODE>(st, sm, a, r0, c0, g_row);
    if constexpr (MODE == kCast2D) __syncthreads();
    if (ok && a.colwise) col_pass<T, MODE>(st, sm, a, r0, c0, g_col, sgn);
    __syncthreads();  // stage s fully read
    if (*sm.abort_flag) break;
    if (tid == 0 && k + C::kStages < my_count) issue(k + C::kStages);
  }
  if (k < my_count && tid == 0) {
    // A wait ran out: wait (bounded) for this CTA's copies still in flight
    // before the shared memory is released.
    const int issued = (k + C::kStages < my_count) ? k + C::kStages : my_count;
    for (int j = k; j < issued; ++j)
      mbar_wait_bounded(&sm.bars[j % C::kStages], (uint32_t)((j / C::kStages) & 1), a.status);
  }
}

template <typename T, int MODE>
cudaError_t launch_t(const CUtensorMap& map, const CastArgs& a, bool pdl, const LaunchCtx& ctx) {
  using C = TileCfg<T>;
  auto fn = cast_kernel<T, MODE>;
  // The shared-memory opt-in is per device; remembered per instantiation.
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<T>());
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  const int cap = ctx.num_sms * C::kMinBlocks;
  const int grid = a.num_tiles < cap ? a.num_tiles : cap;
  if (grid == 0) return cudaSuccess;
  void* args[] = {(void*)&map, (void*)&a};
  if (pdl) return launch_pdl((const void*)fn, dim3(grid), dim3(kThreads), smem_bytes<T>(), ctx.stream, args);
  fn<<<grid, kThreads, smem_bytes<T>(), ctx.stream>>>(map, a);
  return cudaGetLastError();
}

}  // namespace

// Tensor map of x: dims {N, M}, box {128 bytes, 128 rows}, 128-byte swizzle,
// zero fill outside the tensor.
cudaError_t make_x_tensor_map(CUtensorMap* map, const void* x, bool bf16, int64_t M, int64_t N);

cudaError_t launch_cast(const void* x, bool bf16, int mode, CastArgs args, bool pdl, const LaunchCtx& ctx) {
  CUtensorMap map;
  cudaError_t e = make_x_tensor_map(&map, x, bf16, args.M, args.N);
  if (e != cudaSuccess) return e;
  const int64_t tiles_m = (args.M + kTile - 1) / kTile, tiles_n = (args.N + kTile - 1) / kTile;
  args.tiles_n = (int)tiles_n;
  args.num_tiles = (int)(tiles_m * tiles_n);
  if (bf16) {
    if (mode == kCast1D) return launch_t<uint16_t, kCast1D>(map, args, pdl, ctx);
    if (mode == kCast2D) return launch_t<uint16_t, kCast2D>(map, args, pdl, ctx);
    return launch_t<uint16_t, kCastRHT>(map, args, pdl, ctx);
  }
  if (mode == kCast1D) return launch_t<float, kCast1D>(map, args, pdl, ctx);
  return launch_t<float, kCast2D>(map, args, pdl, ctx);
}

}  // namespace nvfp4
