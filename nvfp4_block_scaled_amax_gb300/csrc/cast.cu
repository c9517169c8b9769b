// cast.cu -- fused NVFP4 cast with row-wise and column-wise (transposed)
// outputs from one read of each 128x128 tile of x.
//
// Tiles are TMA-loaded into shared memory (128-byte swizzle, a 3-stage
// mbarrier pipeline); persistent CTAs walk the tiles in reverse order so the
// first tiles they read are the ones the amax pass read last (most likely
// still in L2).
//
// Per tile each thread owns an 8x8 sub-block (8 rows x 8 columns):
//   * a 1x16 row block is the sub-blocks of lanes l and l^1; a 16x1 column
//     block those of lanes l and l^8; a 16x16 tile lanes l, l^1, l^8, l^9;
//     block maxima are combined with one or two shuffles;
//   * row-wise codes: one 32-bit word (8 codes) per row of the sub-block;
//   * column-wise codes: one word per column of the sub-block, computed from
//     the same registers (1D, with the column block's scale) or, in 2D, the
//     8x8 nibble transpose of the row-wise words (same scale per tile);
//   * scales are staged in shared memory and stored once per tile by 128
//     threads: 16-byte lines of the cuBLAS 128x4 layout ("Fuse NVFP4 scale
//     swizzling on SM120 and SM121", Changes: aligned groups of four scales
//     written together), or 8-byte runs of the compact layout.
// With the random Hadamard transform the column blocks are transformed on
// the tensor cores (see the Hadamard column pass below) while warps 0-3 cast
// the rows with the wide mapping of tile_ops.cuh.
#include <atomic>

#include "common.cuh"
#include "hadamard.cuh"
#include "kernels.h"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace {

using namespace tile;

constexpr int kThreads = 256;

struct Smem {
  uint8_t* stages;
  float* rtab_row;  // [128] encode factor per E4M3 code, row-wise g
  float* rtab_col;  // [128] same, column-wise g
  uint8_t* sc_row;  // [2][kScRegion] staged row-wise scales of a tile (by tile parity)
  uint8_t* sc_col;  // [2][kScRegion] staged column-wise scales
  uint64_t* bars;   // [kStages]
  int* abort_flag;
  // Hadamard column transform (BF16): operand B, its MMA barrier and the
  // tensor-memory address live in the unused tails of the staging regions
  // (a row-wise region uses bytes 0..7 * kScPitchRow + 127, a column-wise
  // one 0..7 * kScPitchCol + 127), so the cast keeps two CTAs per SM.
  uint8_t* hmat;    // n-group g (8 columns of B, 256 bytes) at hmat + g * kScRegion
  uint64_t* mma_bar;
  uint32_t* tmem_slot;
};
constexpr int kHmatOffset = 1280, kMmaBarOffset = 1472;
static_assert(7 * kScPitchRow + 128 <= kHmatOffset && kHmatOffset + 256 <= kScRegion, "row staging tail");
static_assert(7 * kScPitchCol + 128 <= kMmaBarOffset && kMmaBarOffset + 12 <= kScRegion, "column staging tail");

template <typename T>
__device__ __forceinline__ Smem carve(uint8_t* raw) {
  Smem s;
  // offset arithmetic on the shared array itself, so that every carved
  // pointer stays a known shared-memory pointer (ld.shared / atom.shared)
  uint8_t* p = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  s.stages = p;
  p += (size_t)TileCfg<T>::kStages * tile_bytes<T>();
  s.rtab_row = reinterpret_cast<float*>(p);
  s.rtab_col = s.rtab_row + 128;
  s.sc_row = reinterpret_cast<uint8_t*>(s.rtab_col + 128);
  s.sc_col = s.sc_row + 2 * kScRegion;
  s.bars = reinterpret_cast<uint64_t*>(s.sc_col + 2 * kScRegion);
  s.abort_flag = reinterpret_cast<int*>(s.bars + TileCfg<T>::kStages);
  s.hmat = s.sc_row + kHmatOffset;
  s.mma_bar = reinterpret_cast<uint64_t*>(s.sc_col + kMmaBarOffset);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.sc_col + kMmaBarOffset + 8);
  return s;
}

// ---------------------------------------------------------------------------
// Hadamard column pass (BF16): hadamard.cuh.  One thread issues the tile's
// eight block transforms, which run beside the row-wise pass of warps 0..3;
// warps 4..7 then cast the columns (warp w owns tile columns 32 (w % 4) ..).
// ---------------------------------------------------------------------------

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
  // Hadamard column pass: the operand, the MMA barrier and 128 tensor-memory
  // columns (one tile's eight 128 x 16 FP32 results; two CTAs per SM use 256
  // of the 512).
  const bool tc_cols = MODE == kCastRHT && a.colwise != 0;
  uint32_t tmem = 0;
  if (tc_cols) {
    fill_hadamard_operand(sm.hmat, kScRegion, a.sign_mask);
    fence_proxy_async_shared();  // the operand, before the tensor cores read it
    if (tid == 0) {
      mbar_init(sm.mma_bar, 1);
      fence_mbar_init();
    }
    if ((tid >> 5) == 0) tmem_alloc(sm.tmem_slot, 128);
    tcgen05_before_sync();
  }
  __syncthreads();
  if (tc_cols) {
    tcgen05_after_sync();
    tmem = *reinterpret_cast<volatile uint32_t*>(sm.tmem_slot);
  }

  const bool do_row = a.rowwise != 0;
  const bool do_col_blk = a.colwise != 0 && MODE != kCastRHT;
  int k = 0;
  for (; k < my_count; ++k) {
    const int s = k % C::kStages;
    // Warp-uniform so that the shuffles below see whole warps.
    const bool ok =
        __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&sm.bars[s], (uint32_t)((k / C::kStages) & 1), a.status));
    if (!ok) *sm.abort_flag = 1;
    const int t = tile_of(k);
    const int tr = t / a.tiles_n, tc = t - tr * a.tiles_n;
    const int64_t r0 = (int64_t)tr * kTile, c0 = (int64_t)tc * kTile;
    const uint8_t* st = sm.stages + (size_t)s * tile_bytes<T>();
    const int parity = k & 1;
    bool tc_done = false;
    if constexpr (MODE == kCastRHT && sizeof(T) == 2) {
      if (tc_cols) {
        tc_done = true;
        const int warp = tid >> 5;
        if (ok && tid == 0) rht_issue_mma(smem_u32(st), smem_u32(sm.hmat), kScRegion, tmem, sm.mma_bar);
        if (ok && warp < 4) {
          if (do_row)
            wide_pass_any<kCast1D>(smem_u32(st), sm.rtab_row, smem_u32(sm.sc_row + parity * kScRegion),
                                   smem_u32(sm.sc_col + parity * kScRegion), a, r0, c0, g_row, true, false, warp);
        } else if (ok) {
          // the transforms of tile k complete (k-th phase of the MMA barrier)
          const bool done = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(sm.mma_bar, (uint32_t)(k & 1), a.status));
          if (done) {
            tcgen05_after_sync();
            rht_col_epilogue<false>(tmem, warp & 3, sm.rtab_col, sm.sc_col + parity * kScRegion, a, r0, c0, g_col);
          } else {
            *sm.abort_flag = 1;
          }
        }
        tcgen05_before_sync();
      }
    }
    if (ok && !tc_done && (do_row || do_col_blk))
      block_pass_any<T, MODE>(smem_u32(st), sm.rtab_row, sm.rtab_col, smem_u32(sm.sc_row + parity * kScRegion),
                              smem_u32(sm.sc_col + parity * kScRegion), a, r0, c0, g_row, g_col, do_row, do_col_blk,
                              threadIdx.x >> 5);
    __syncthreads();  // stage s fully read; this tile's scales staged
    if (*sm.abort_flag) break;
    if (tid == 0 && k + C::kStages < my_count) issue(k + C::kStages);
    // this tile's scales: threads 0..127 row-wise, 128..255 column-wise
    if (tid < 128) {
      if (do_row)
        store_scale_tile<MODE, false>(sm.sc_row + parity * kScRegion, a.scale_row, r0, c0 / 16, a.M, a.N / 16,
                                      a.swizzled, tid);
    } else if (a.colwise) {
      store_scale_tile<MODE, true>(sm.sc_col + parity * kScRegion, a.scale_col, c0, r0 / 16, a.N, a.M / 16,
                                   a.swizzled, tid - 128);
    }
  }
  if (tc_cols && (tid >> 5) == 0) {
    tcgen05_after_sync();
    tmem_dealloc(tmem, 128);
  }
  if (k < my_count && tid == 0) {
    // A wait ran out: wait (bounded) for this CTA's copies still in flight
    // before the shared memory is released.
    const int issued = (k + C::kStages < my_count) ? k + C::kStages : my_count;
    for (int jj = k; jj < issued; ++jj)
      mbar_wait_bounded(&sm.bars[jj % C::kStages], (uint32_t)((jj / C::kStages) & 1), a.status);
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

cudaError_t launch_cast(const CUtensorMap& map, bool bf16, int mode, CastArgs args, bool pdl, const LaunchCtx& ctx) {
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
