// grouped.cu -- grouped (multi-tensor) NVFP4 quantize: x stacks several
// tensors along its first dimension and each is quantized as a tensor of its
// own (its own amax, and so its own global scale; "Implement row-scaled NVFP4
// fprop recipe", Important Files Changed: a grouped tensor keeps one amax
// slice per member).  Three launches whatever the number of members:
//   * zero the members' amax buffers;
//   * max|x| per member: every member's rows are a contiguous, 16-byte
//     aligned range of x, cut into chunks of 2048 vectors; a grid-stride loop
//     over all members' chunks keeps a CTA's running maximum while its chunks
//     stay in one member and publishes it (one atomic max per buffer) when
//     the member changes;
//   * the fused row-wise + column-wise cast of every member's 128x128 tiles
//     (the tile code of the plain cast, tile_ops.cuh), one tensor map over
//     all of x: a member's tile starts at row row0 + 128 tr, and the rows of
//     the next member that a boundary tile also loads are masked off like the
//     rows below the end of a plain tensor (a member's rows are a multiple of
//     16, so no 16-row block straddles two members).  The encode-factor tables
//     are rebuilt when a CTA's next tile belongs to another member.
#include <atomic>

#include "common.cuh"
#include "grouped.h"
#include "kernels.h"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace {

using namespace tile;

constexpr int kGThreads = 256;  // amax and cast kernels
constexpr int kGUnroll = 8;     // 16-byte loads in flight per thread and chunk
static_assert(kGroupChunkVecs == (int64_t)kGThreads * kGUnroll, "chunk = one batch of the CTA's loads");

__global__ void grouped_zero_kernel(const __grid_constant__ GroupedArgs ga) {
  grid_launch_dependents();
  if (ga.noop != nullptr && *ga.noop == 1.0f) return;
  const int g = threadIdx.x;
  if (g < ga.num_groups) {
    if (ga.amax_row[g] != nullptr) *ga.amax_row[g] = 0.0f;
    if (ga.amax_col[g] != nullptr) *ga.amax_col[g] = 0.0f;
  }
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// CTA-wide max of non-negative floats, published with one atomic max into
// each of member g's buffers.  Barriers on both sides, so it may be called
// again right away.
__device__ __forceinline__ void publish_member_max(float m, float* red, const GroupedArgs& ga, int g) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // an earlier call's reads of red are done
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    m = lane < kGThreads / 32 ? red[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if (lane == 0) {
      grid_dependency_wait();  // the zeroing kernel has completed
      // non-negative floats order like their bit patterns read as integers
      if (ga.amax_row[g] != nullptr) atomicMax(reinterpret_cast<int*>(ga.amax_row[g]), __float_as_int(m));
      if (ga.amax_col[g] != nullptr) atomicMax(reinterpret_cast<int*>(ga.amax_col[g]), __float_as_int(m));
    }
  }
}

template <bool kBF16>
__global__ void __launch_bounds__(kGThreads, 4)
    grouped_amax_kernel(const void* __restrict__ x, const __grid_constant__ GroupedArgs ga) {
  __shared__ float red[kGThreads / 32];
  grid_launch_dependents();
  if (ga.noop != nullptr && *ga.noop == 1.0f) return;
  constexpr int kEpv = kBF16 ? 8 : 4;  // elements per 16-byte vector
  const uint4* xv = static_cast<const uint4*>(x);
  const int64_t vecs_per_row = ga.N / kEpv;
  int cur = -1;
  uint32_t acc0 = 0, acc1 = 0;  // BF16: packed |x| maxima
  float m0 = 0.0f, m1 = 0.0f;   // FP32
  auto running = [&] {
    if constexpr (kBF16) {
      uint32_t acc;
      asm("max.bf16x2 %0, %1, %2;" : "=r"(acc) : "r"(acc0), "r"(acc1));
      return bf16x2_hmax_to_f32(acc);
    } else {
      return fmaxf(m0, m1);
    }
  };
  for (int c = blockIdx.x; c < ga.num_chunks; c += gridDim.x) {
    const int g = member_of(ga.chunk_start, ga.num_groups, c);  // the same in every thread
    if (g != cur) {
      if (cur >= 0) publish_member_max(running(), red, ga, cur);
      cur = g;
      acc0 = acc1 = 0;
      m0 = m1 = 0.0f;
    }
    const int64_t first = ga.row0[g] * vecs_per_row;
    const int64_t end = first + ga.rows[g] * vecs_per_row;
    const int64_t base = first + (int64_t)(c - ga.chunk_start[g]) * kGroupChunkVecs + threadIdx.x;
    uint4 v[kGUnroll];
#pragma unroll
    for (int u = 0; u < kGUnroll; ++u) {
      const int64_t i = base + (int64_t)u * kGThreads;
      v[u] = i < end ? ld_stream(xv + i) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kGUnroll; ++u) {
      if constexpr (kBF16) {
        uint32_t t0, t1;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(t0) : "r"(v[u].x & 0x7FFF7FFFu), "r"(v[u].y & 0x7FFF7FFFu));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(t1) : "r"(v[u].z & 0x7FFF7FFFu), "r"(v[u].w & 0x7FFF7FFFu));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(acc0) : "r"(t0));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(acc1) : "r"(t1));
      } else {
        m0 = fmaxf(m0, fmaxf(fabsf(__uint_as_float(v[u].x)), fabsf(__uint_as_float(v[u].y))));
        m1 = fmaxf(m1, fmaxf(fabsf(__uint_as_float(v[u].z)), fabsf(__uint_as_float(v[u].w))));
      }
    }
  }
  if (cur >= 0) publish_member_max(running(), red, ga, cur);
}

struct GSmem {
  uint8_t* stages;
  float* rtab_row;  // [128] encode factor per E4M3 code, the current member's g
  float* rtab_col;  // [128]
  uint8_t* sc_row;  // [2][kScRegion] staged scales of a tile (by tile parity)
  uint8_t* sc_col;  // [2][kScRegion]
  uint64_t* bars;   // [kStages]
  int* abort_flag;
  float* g;         // [2] the current member's row-wise and column-wise global encode scales
};

template <typename T>
__device__ __forceinline__ GSmem gcarve(uint8_t* raw) {
  GSmem s;
  uint8_t* p = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  s.stages = p;
  p += (size_t)TileCfg<T>::kStages * tile_bytes<T>();
  s.rtab_row = reinterpret_cast<float*>(p);
  s.rtab_col = s.rtab_row + 128;
  s.sc_row = reinterpret_cast<uint8_t*>(s.rtab_col + 128);
  s.sc_col = s.sc_row + 2 * kScRegion;
  s.bars = reinterpret_cast<uint64_t*>(s.sc_col + 2 * kScRegion);
  s.abort_flag = reinterpret_cast<int*>(s.bars + TileCfg<T>::kStages);
  s.g = reinterpret_cast<float*>(s.abort_flag + 1);
  return s;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kGThreads, TileCfg<T>::kMinBlocks)
    grouped_cast_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ GroupedArgs ga) {
  using C = TileCfg<T>;
  extern __shared__ uint8_t smem_raw[];
  const GSmem sm = gcarve<T>(smem_raw);
  const int tid = threadIdx.x;
  if (ga.noop != nullptr && *ga.noop == 1.0f) return;

  const int num_tiles = ga.num_tiles;
  const int bid = blockIdx.x, nb = gridDim.x;
  const int my_count = (bid < num_tiles) ? (num_tiles - 1 - bid) / nb + 1 : 0;
  // reverse order: the first tiles read are the ones the amax pass read last
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
    const MemberTile p = member_tile(ga, tile_of(k));
    uint8_t* dst = sm.stages + (size_t)(k % C::kStages) * tile_bytes<T>();
    uint64_t* bar = &sm.bars[k % C::kStages];
    mbar_arrive_expect_tx(bar, tile_bytes<T>());
#pragma unroll
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_2d(dst + b * kBoxBytes, &tmap, (int32_t)p.c0 + b * C::kBoxCols, (int32_t)(ga.row0[p.g] + p.r0), bar,
                  policy);
  };
  // x does not depend on the amax kernel: the first tiles are requested
  // before waiting for it.
  if (tid == 0)
    for (int k = 0; k < C::kStages && k < my_count; ++k) issue(k);
  grid_dependency_wait();  // the members' amaxes written by the preceding kernel are visible

  const bool do_row = ga.rowwise != 0, do_col = ga.colwise != 0;
  int cur = -1;
  int k = 0;
  for (; k < my_count; ++k) {
    const int s = k % C::kStages;
    const MemberTile p = member_tile(ga, tile_of(k));  // the same in every thread
    if (p.g != cur) {
      // every thread is past the previous tile's cast (the barrier at the end
      // of its iteration), so the tables may be rewritten
      cur = p.g;
      const float* ar = ga.amax_row[cur];
      const float* ac = ga.amax_col[cur];
      const float gr = global_encode_scale(ar ? *ar : 0.0f), gc = global_encode_scale(ac ? *ac : 0.0f);
      if (tid < 128)
        sm.rtab_row[tid] = encode_factor((uint32_t)tid, gr);
      else
        sm.rtab_col[tid - 128] = encode_factor((uint32_t)(tid - 128), gc);
      if (tid == 0) {
        sm.g[0] = gr;
        sm.g[1] = gc;
      }
      __syncthreads();
    }
    // the member's view as a plain tensor (read from the parameter table)
    CastArgs a = {};
    a.M = ga.rows[p.g];
    a.N = ga.N;
    a.data_row = ga.data_row[p.g];
    a.scale_row = ga.scale_row[p.g];
    a.data_col = ga.data_col[p.g];
    a.scale_col = ga.scale_col[p.g];
    a.status = ga.status;
    a.rowwise = ga.rowwise;
    a.colwise = ga.colwise;
    a.swizzled = ga.swizzled;
    const float g_row = sm.g[0], g_col = sm.g[1];
    // warp-uniform so that the shuffles of the cast see whole warps
    const bool ok =
        __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&sm.bars[s], (uint32_t)((k / C::kStages) & 1), ga.status));
    if (!ok) *sm.abort_flag = 1;
    const uint8_t* st = sm.stages + (size_t)s * tile_bytes<T>();
    const int parity = k & 1;
    if (ok)
      block_pass_any<T, MODE>(smem_u32(st), sm.rtab_row, sm.rtab_col, smem_u32(sm.sc_row + parity * kScRegion),
                              smem_u32(sm.sc_col + parity * kScRegion), a, p.r0, p.c0, g_row, g_col, do_row, do_col,
                              tid >> 5);
    __syncthreads();  // stage s fully read; this tile's scales staged
    if (*sm.abort_flag) break;
    if (tid == 0 && k + C::kStages < my_count) issue(k + C::kStages);
    // this tile's scales: threads 0..127 row-wise, 128..255 column-wise
    if (tid < 128) {
      if (do_row)
        store_scale_tile<MODE, false>(sm.sc_row + parity * kScRegion, a.scale_row, p.r0, p.c0 / 16, a.M, a.N / 16,
                                      a.swizzled, tid);
    } else if (do_col) {
      store_scale_tile<MODE, true>(sm.sc_col + parity * kScRegion, a.scale_col, p.c0, p.r0 / 16, a.N, a.M / 16,
                                   a.swizzled, tid - 128);
    }
  }
  if (k < my_count && tid == 0) {
    // A wait ran out: wait (bounded) for this CTA's copies still in flight
    // before the shared memory is released.
    const int issued = (k + C::kStages < my_count) ? k + C::kStages : my_count;
    for (int jj = k; jj < issued; ++jj)
      mbar_wait_bounded(&sm.bars[jj % C::kStages], (uint32_t)((jj / C::kStages) & 1), ga.status);
  }
}

template <typename T, int MODE>
cudaError_t launch_cast_t(const CUtensorMap& map, const GroupedArgs& ga, bool pdl, const LaunchCtx& ctx) {
  using C = TileCfg<T>;
  auto fn = grouped_cast_kernel<T, MODE>;
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
  const int grid = ga.num_tiles < cap ? ga.num_tiles : cap;
  if (grid == 0) return cudaSuccess;
  void* args[] = {(void*)&map, (void*)&ga};
  if (pdl) return launch_pdl((const void*)fn, dim3(grid), dim3(kGThreads), smem_bytes<T>(), ctx.stream, args);
  fn<<<grid, kGThreads, smem_bytes<T>(), ctx.stream>>>(map, ga);
  return cudaGetLastError();
}

}  // namespace

void grouped_prefix_sums(GroupedArgs& ga, bool bf16) {
  const int epv = bf16 ? 8 : 4;
  ga.tiles_n = (int)((ga.N + kTile - 1) / kTile);
  ga.tile_start[0] = 0;
  ga.chunk_start[0] = 0;
  for (int g = 0; g < ga.num_groups; ++g) {
    const int64_t tiles_m = (ga.rows[g] + kTile - 1) / kTile;
    const int64_t chunks = (ga.rows[g] * (ga.N / epv) + kGroupChunkVecs - 1) / kGroupChunkVecs;
    ga.tile_start[g + 1] = ga.tile_start[g] + (int)(tiles_m * ga.tiles_n);
    ga.chunk_start[g + 1] = ga.chunk_start[g] + (int)chunks;
  }
  ga.num_tiles = ga.tile_start[ga.num_groups];
  ga.num_chunks = ga.chunk_start[ga.num_groups];
}

cudaError_t launch_grouped_zero(const GroupedArgs& ga, const LaunchCtx& ctx) {
  grouped_zero_kernel<<<1, kMaxGroups, 0, ctx.stream>>>(ga);
  return cudaGetLastError();
}

cudaError_t launch_grouped(const void* x, const CUtensorMap* map, bool bf16, int mode, GroupedArgs ga,
                           bool skip_amax, const LaunchCtx& ctx) {
  grouped_prefix_sums(ga, bf16);
  cudaError_t e;
  if (!skip_amax) {
    if ((e = launch_grouped_zero(ga, ctx)) != cudaSuccess) return e;
    if (ga.num_chunks > 0) {
      const void* fn = bf16 ? (const void*)grouped_amax_kernel<true> : (const void*)grouped_amax_kernel<false>;
      static std::atomic<int> occ[2] = {0, 0};  // CTAs per SM
      int per_sm = occ[bf16].load();
      if (per_sm == 0) {
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kGThreads, 0)) != cudaSuccess) return e;
        occ[bf16].store(per_sm);
      }
      const int cap = ctx.num_sms * (per_sm > 0 ? per_sm : 1);
      const int grid = ga.num_chunks < cap ? ga.num_chunks : cap;
      void* args[] = {(void*)&x, (void*)&ga};
      if ((e = launch_pdl(fn, dim3(grid), dim3(kGThreads), 0, ctx.stream, args)) != cudaSuccess) return e;
    }
  }
  if (ga.num_tiles == 0 || map == nullptr) return cudaSuccess;
  const bool pdl = !skip_amax;
  if (bf16) {
    if (mode == kCast1D) return launch_cast_t<uint16_t, kCast1D>(*map, ga, pdl, ctx);
    return launch_cast_t<uint16_t, kCast2D>(*map, ga, pdl, ctx);
  }
  if (mode == kCast1D) return launch_cast_t<float, kCast1D>(*map, ga, pdl, ctx);
  return launch_cast_t<float, kCast2D>(*map, ga, pdl, ctx);
}

}  // namespace nvfp4
