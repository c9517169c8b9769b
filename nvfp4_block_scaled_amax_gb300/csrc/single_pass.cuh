// single_pass.cuh -- the pieces the single-pass kernels (fused.cu,
// fused_rht.cu) share: bounded hand-overs between warps, the TMA stage ring
// with its refill counting, and the per-tile scale write-back (a share per
// warp, or bulk copies for the 128x4 layout).
#pragma once

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace sp {

using tile::kBoxBytes;
using tile::kTile;
using tile::TileCfg;

// Bounded wait of lane 0 until the counter *p reaches `want` (a shared-memory
// hand-over between warps); warp-uniform result, false when it ran out.
__device__ __forceinline__ bool warp_wait_count(const unsigned* p, unsigned want, unsigned* status) {
  unsigned good = 1;
  if ((threadIdx.x & 31) == 0) {
    const volatile unsigned* c = p;
    if (*c < want) {
      const long long t0 = clock64();
      while (*c < want) {
        if (clock64() - t0 > kWaitLimitCycles) {
          atomicOr(status, kStatusWaitTimeout);
          good = 0;
          break;
        }
      }
    }
  }
  const bool ok = __shfl_sync(0xFFFFFFFFu, good, 0) != 0;
  __threadfence_block();  // the counted warps' shared-memory writes are visible past this point
  return ok;
}
// The same until *slot == want.
__device__ __forceinline__ bool warp_wait_slot(const int* p, int want, unsigned* status) {
  unsigned good = 1;
  if ((threadIdx.x & 31) == 0) {
    const volatile int* slot = p;
    if (*slot != want) {
      const long long t0 = clock64();
      while (*slot != want) {
        if (clock64() - t0 > kWaitLimitCycles) {
          atomicOr(status, kStatusWaitTimeout);
          good = 0;
          break;
        }
      }
    }
  }
  return __shfl_sync(0xFFFFFFFFu, good, 0) != 0;
}

// TMA coordinates (x = first column, y = first row) of tile t of a plain
// tensor with tiles_n tile columns (row-major tile order).
struct PlainTiles {
  int tiles_n;
  __device__ __forceinline__ void xy(int t, int32_t& x, int32_t& y) const {
    const int tr = t / tiles_n;
    x = (t - tr * tiles_n) * kTile;
    y = tr * kTile;
  }
};

// The ring of S shared-memory stages a CTA streams its tiles through: tile k
// of the CTA (t_k = b + k * G) uses stage k % S; its TMA completion is
// full[s] with phase parity (k / S) & 1 (the fills of a stage are
// sequential: in phase A fill number k / S, in phase B a stage's F phase-A
// fills are followed by its tiles in reverse, tile s + m S as fill
// 2F - 2 - m, the same parity).
template <typename T, int S, int WPT, class Tiles = PlainTiles>
struct StageRing {
  uint8_t* stages;
  uint64_t* full;     // [S]
  unsigned* loaded;   // [S] warps done with the stage's tile
  unsigned* issued;   // [S] loads issued into the stage so far
  int* tile_in;       // [S] tile index of the stage's latest issued load
  const CUtensorMap* tmap;
  int b, G;
  Tiles tiles;        // where tile t lies in the tensor map
  unsigned* status;

  // Tile k's first row and column in the tensor map.
  __device__ __forceinline__ void tile_rc(int k, int64_t& r0, int64_t& c0) const {
    int32_t x, y;
    tiles.xy(b + k * G, x, y);
    r0 = y;
    c0 = x;
  }
  __device__ __forceinline__ uint32_t stage(int s) const {
    return smem_u32(stages + (size_t)s * tile::tile_bytes<T>());
  }
  // One thread, before the CTA's first barrier.
  __device__ __forceinline__ void init() const {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      loaded[s] = 0;
      issued[s] = 0;
      tile_in[s] = -1;
    }
  }
  // One thread: load tile k into its stage.
  __device__ __forceinline__ void issue(int k, uint64_t pol) const {
    const int s = k % S;
    int32_t c0, r0;
    tiles.xy(b + k * G, c0, r0);
    uint8_t* dst = stages + (size_t)s * tile::tile_bytes<T>();
    issued[s] += 1;
    *reinterpret_cast<volatile int*>(&tile_in[s]) = k;  // before the arrival (see wait_full)
    mbar_arrive_expect_tx(&full[s], tile::tile_bytes<T>());
#pragma unroll
    for (int bb = 0; bb < TileCfg<T>::kBoxes; ++bb)
      tma_load_2d(dst + bb * kBoxBytes, tmap, c0 + bb * TileCfg<T>::kBoxCols, r0, &full[s], pol);
  }
  // Warp (all lanes): done with stage s's tile.  The group's last warp
  // loads tile `next` (if any) into the stage.  `token` is a value each lane
  // computed from every word it read.  Lane 0 counts the warp out, but the
  // lanes need not have run in step up to here (a lane-0-only branch
  // earlier on can leave lane 0 ahead of the others), so the lanes' tokens
  // are first combined by a warp-wide reduction, which waits for every lane
  // and for its reads, and the count's address depends on the result.
  __device__ __forceinline__ void release(int s, int next, uint64_t pol, uint32_t token) const {
    const uint32_t all = __reduce_or_sync(0xFFFFFFFFu, token);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      uint32_t zero;
      asm volatile("and.b32 %0, %1, 0;" : "=r"(zero) : "r"(all));
      if (atomicAdd(&loaded[s] + zero, 1u) == (unsigned)(WPT - 1)) {
        loaded[s] = 0;
        __threadfence_block();
        if (next >= 0) issue(next, pol);
      }
    }
  }
  // Warp: until tile k is in its stage.  The stage's previous tile belongs
  // to another group, which may not be done with it yet: a parity wait
  // issued before tile k's load would refer to that earlier phase.  So lane
  // 0 first waits (bounded) until tile k's load has been issued (tile_in[s]
  // is set before its arrival), which also means the earlier phase is
  // complete.
  __device__ __forceinline__ bool wait_full(int k) const {
    const int s = k % S;
    if (!warp_wait_slot(&tile_in[s], k, status)) return false;
    return __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[s], (uint32_t)((k / S) & 1), status)) != 0;
  }
  // One thread, when a CTA leaves early: let the latest load into each stage
  // land (bounded) before the shared memory is released.
  __device__ __forceinline__ void drain() const {
    for (int s = 0; s < S; ++s)
      if (issued[s] > 0) mbar_wait_bounded(&full[s], (issued[s] - 1u) & 1u, status);
  }
};

// Warp: this warp's scales of the tile are staged in the buffer.
__device__ __forceinline__ void count_staged(unsigned* staged_q) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    __threadfence_block();  // this warp's staged scales before its count
    atomicAdd(staged_q, 1u);
  }
}

// Warp cw of a group: its share of the write-back of a tile's staged scales
// (compact: 8-byte runs; 128x4: 16-byte lines) once all WPT warps of the
// group have staged them (staged counts every use of the buffer); then it
// counts itself in wb (the buffer may be reused once all have).
template <int MODE, int WPT>
__device__ __forceinline__ bool write_back_share(const uint8_t* sc, const unsigned* staged, unsigned* wb,
                                                 unsigned want_staged, int cw, const CastArgs& a, int64_t r0,
                                                 int64_t c0, bool do_row, bool do_col) {
  if (!warp_wait_count(staged, want_staged, a.status)) return false;
  const int lane = threadIdx.x & 31;
  const int per = a.swizzled ? 64 / WPT : 128 / WPT;  // 16-byte lines or rows per warp
  if (lane < per) {
    const int t = cw * per + lane;
    if (do_row) tile::store_scale_tile<MODE, false>(sc, a.scale_row, r0, c0 / 16, a.M, a.N / 16, a.swizzled, t);
    if (do_col)
      tile::store_scale_tile<MODE, true>(sc + tile::kScRegion, a.scale_col, c0, r0 / 16, a.N, a.M / 16, a.swizzled,
                                         t);
  }
  __syncwarp();  // the lanes' reads of the buffer are complete (their stores used them)
  if (lane == 0) atomicAdd(wb, 1u);
  return true;
}

// 128x4 layout, warp: this warp has staged its part of the tile's scales in
// the stored byte order; the group's last warp to do so writes each
// direction's two 512-byte atoms with one bulk copy and remembers the
// buffer (pending_q, lane 0) to free it later (bulk_free).
template <int WPT>
__device__ __forceinline__ void bulk_staged(unsigned* staged_q, int q, const uint8_t* sc, const CastArgs& a,
                                            int64_t r0, int64_t c0, bool do_row, bool do_col, int& pending_q) {
  fence_proxy_async_shared();  // this lane's staging stores, before the copy engine reads them
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    __threadfence_block();
    if (atomicAdd(staged_q, 1u) % WPT == (unsigned)(WPT - 1)) {
      __threadfence_block();
      if (do_row) bulk_store(a.scale_row + ((r0 >> 7) * (a.N >> 6) + (c0 >> 6)) * 512, smem_u32(sc), 1024);
      if (do_col)
        bulk_store(a.scale_col + ((c0 >> 7) * (a.M >> 6) + (r0 >> 6)) * 512, smem_u32(sc + tile::kScRegion), 1024);
      bulk_commit();
      pending_q = q;
    }
  }
  __syncwarp();
}
// Lane 0: once the bulk copies this warp issued have read their buffer,
// free it for the group (wb of the buffer += WPT).
template <int WPT>
__device__ __forceinline__ void bulk_free(int& pending_q, unsigned* wb) {
  if ((threadIdx.x & 31) == 0 && pending_q >= 0) {
    bulk_wait_read_all();
    __threadfence_block();
    atomicAdd(&wb[pending_q], (unsigned)WPT);
    pending_q = -1;
  }
}

// Host: one CTA of `threads` threads per SM (at most one per tile), as a
// cooperative launch so that all CTAs are co-resident (the grid barrier
// needs them all).  The dynamic shared-memory limit is raised once per
// kernel and device.
template <auto Fn, class Args>
cudaError_t launch_persistent(size_t smem, int threads, const CUtensorMap& map, const Args& a, int num_tiles,
                              SinglePassWorkspace* ws, const LaunchCtx& ctx) {
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(Fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  const int grid = num_tiles < ctx.num_sms ? num_tiles : ctx.num_sms;
  if (grid == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {(void*)&map, (void*)&a, (void*)&ws};
  return cudaLaunchKernelExC(&cfg, (const void*)Fn, args);
}

}  // namespace sp
}  // namespace nvfp4
