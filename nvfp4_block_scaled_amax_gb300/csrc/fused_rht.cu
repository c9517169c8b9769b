// fused_rht.cu -- single-launch NVFP4 quantize with the random Hadamard
// transform of column blocks (BF16): max|x| (row-wise amax) and max|RHT(x)|
// (column-wise amax), then the row-wise cast of x and the column-wise cast of
// the transformed columns, in one persistent kernel ("Write both NVFP4 amax
// buffers", review reply: with RHT the row amax is max|x| and the column
// amax is max|RHT(x)|).
//
// The structure of fused.cu, with the same stage ring and scale write-back
// (single_pass.cuh): one CTA per SM, cooperative launch, 16 warps in
// 4 groups of 4, a 6-stage TMA ring, phase A / grid barrier / phase B, the
// last 6 tiles of a CTA resident.  The transform runs on the tensor cores
// (hadamard.cuh): every tile's eight 16-row blocks are transformed by
// tcgen05.mma into the group's 128 tensor-memory columns (4 groups x 128 =
// all 512), once in phase A for the column amax and again in phase B for the
// cast, so x is read from HBM once and the transform never leaves the chip.
// In both phases warp cw of a group reads tensor-memory lanes 32 cw .. +31
// (tile columns), the lane quarter its warp index allows.
#include "common.cuh"
#include "grid.cuh"
#include "hadamard.cuh"
#include "kernels.h"
#include "single_pass.cuh"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace {

using namespace tile;

constexpr int kRWarps = 16, kRThreads = 32 * kRWarps;
constexpr int kRStages = 6, kRWPT = 4, kRGroups = kRWarps / kRWPT;
constexpr uint32_t kTmemCols = 128 * kRGroups;  // 512: the whole tensor memory of the SM

struct RSmem {
  uint8_t* stages;    // [S][tile]
  uint8_t* sc;        // [groups][2][2][kScRegion] staged row / column scales, two buffers per group
  float* rtab_row;    // [128] encode factor per E4M3 code, g of max|x|
  float* rtab_col;    // [128] same, g of max|RHT(x)|
  uint64_t* full;     // [S] TMA completion per stage
  uint64_t* mma_bar;  // [groups] transform completion per group
  unsigned* loaded;   // [S] warps done with the stage's tile
  unsigned* issued;   // [S] loads issued into the stage so far
  int* tile_in;       // [S] tile index of the stage's latest issued load
  unsigned* staged;   // [groups][2] warps done staging into the buffer (all uses so far)
  unsigned* wb;       // [groups][2] warps done writing the buffer's scales back
  unsigned* tfree;    // [groups] warps done reading the group's tensor memory (all tiles so far)
  unsigned* exited;   // [1]
  unsigned* gen;      // [1] this call's barrier generation
  unsigned* cta_max;  // [2] the CTA's max|x| and max|RHT(x)| bits (phase A)
  unsigned* cta_in;   // [1] warps done with phase A
  float* g;           // [2] broadcast of the two global encode scales
  int* abort_flag;    // [1]
  uint32_t* tmem_slot;
  uint8_t* hmat;      // [512] Hadamard operand (16-byte aligned)
};

constexpr size_t rht_smem_bytes() {
  return 1024 + (size_t)kRStages * tile_bytes<uint16_t>() + (size_t)kRGroups * 2 * 2 * kScRegion + 2 * 128 * 4 +
         8 * (kRStages + kRGroups) + 4 * (3 * kRStages + 5 * kRGroups + 9) + 16 + 512;
}

__device__ __forceinline__ RSmem rcarve(uint8_t* raw) {
  RSmem s;
  uint8_t* p = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  s.stages = p;
  p += (size_t)kRStages * tile_bytes<uint16_t>();
  s.sc = p;
  p += (size_t)kRGroups * 2 * 2 * kScRegion;
  s.rtab_row = reinterpret_cast<float*>(p);
  s.rtab_col = s.rtab_row + 128;
  s.full = reinterpret_cast<uint64_t*>(s.rtab_col + 128);
  s.mma_bar = s.full + kRStages;
  s.loaded = reinterpret_cast<unsigned*>(s.mma_bar + kRGroups);
  s.issued = s.loaded + kRStages;
  s.tile_in = reinterpret_cast<int*>(s.issued + kRStages);
  s.staged = reinterpret_cast<unsigned*>(s.tile_in + kRStages);
  s.wb = s.staged + 2 * kRGroups;
  s.tfree = s.wb + 2 * kRGroups;
  s.exited = s.tfree + kRGroups;
  s.gen = s.exited + 1;
  s.cta_max = s.exited + 2;
  s.cta_in = s.exited + 4;
  s.g = reinterpret_cast<float*>(s.exited + 5);
  s.abort_flag = reinterpret_cast<int*>(s.exited + 7);
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.exited + 8);
  uint8_t* h = reinterpret_cast<uint8_t*>(s.exited + 9);
  s.hmat = h + ((16u - (smem_u32(h) & 15u)) & 15u);
  return s;
}

// max|x| over a quarter of a staged BF16 tile (warp cw: 8 KB, sixteen
// 16-byte loads per lane, consecutive lanes on consecutive chunks).
__device__ __forceinline__ float quarter_absmax(uint32_t stage, int cw) {
  const int lane = threadIdx.x & 31;
  const uint32_t base = stage + (uint32_t)cw * 8192u + (uint32_t)lane * 16u;
  uint32_t acc = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint4 v = lds128(base + 512u * k);
    acc = xsa(acc, xsa(xsa(v.x, v.y), xsa(v.z, v.w)));
  }
  acc &= 0x7FFF7FFFu;
  return fmaxf(bf16_lo(acc), bf16_hi(acc));
}

struct RowHooks {  // the row-wise wide pass: the stage is released after the column pass
  uint32_t* tok;
  const unsigned* wbq;
  unsigned want;
  bool* ok;
  unsigned* status;
  __device__ __forceinline__ void data_done(uint32_t token) const { *tok ^= token; }
  __device__ __forceinline__ void scale_wait() const;
  // the tile's scales (both directions) leave after the column pass
  __device__ __forceinline__ void scales_staged() const {}
};
__device__ __forceinline__ void RowHooks::scale_wait() const { *ok = sp::warp_wait_count(wbq, want, status) && *ok; }

template <bool kBulk>
__global__ void __launch_bounds__(kRThreads, 1)
    fused_rht_kernel(const __grid_constant__ CUtensorMap tmap, const CastArgs a, SinglePassWorkspace* ws) {
  constexpr int S = kRStages, WPT = kRWPT, kGroups = kRGroups;
  extern __shared__ uint8_t smem_raw[];
  const RSmem sm = rcarve(smem_raw);
  if (a.noop != nullptr && *a.noop == 1.0f) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int n = (a.num_tiles - 1 - b) / G + 1;  // tiles t_k = b + k * G, k < n (grid <= tiles)
  const int kept_from = n > S ? n - S : 0;
  const sp::StageRing<uint16_t, S, WPT> ring{sm.stages, sm.full, sm.loaded, sm.issued, sm.tile_in, &tmap, b, G,
                                             sp::PlainTiles{a.tiles_n}, a.status};
  const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
  fill_hadamard_operand(sm.hmat, 256, a.sign_mask);
  fence_proxy_async_shared();  // the operand, before the tensor cores read it
  if (tid == 0) {
    *sm.gen = ld_acquire_gpu(&ws->gen);
    ring.init();
    for (int q = 0; q < kGroups; ++q) {
      mbar_init(&sm.mma_bar[q], 1);
      sm.tfree[q] = 0;
    }
    for (int q = 0; q < 2 * kGroups; ++q) {
      sm.staged[q] = 0;
      sm.wb[q] = 0;
    }
    *sm.abort_flag = 0;
    *sm.exited = 0;
    sm.cta_max[0] = 0;
    sm.cta_max[1] = 0;
    *sm.cta_in = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap);
    for (int k = 0; k < S && k < n; ++k) ring.issue(k, k >= kept_from ? stream : keep);
  }
  if (warp == 0) tmem_alloc(sm.tmem_slot, kTmemCols);
  tcgen05_before_sync();
  __syncthreads();
  tcgen05_after_sync();
  const uint32_t tmem_all = *reinterpret_cast<volatile uint32_t*>(sm.tmem_slot);

  const int grp = warp / WPT, cw = warp % WPT;
  const uint32_t tmem = tmem_all + 128u * (uint32_t)grp;  // the group's columns
  int jt = 0;             // transforms of this group so far (the same count in each of its warps)
  int mma_issued = 0;     // warp cw == 0: transforms it issued
  // Warp cw == 0 of the group: the transform of the tile in stage `st`, once
  // all four warps have read the group's previous transform.
  auto transform = [&](uint32_t st) {
    if (cw != 0) return true;
    if (!sp::warp_wait_count(&sm.tfree[grp], (unsigned)(WPT * jt), a.status)) return false;
    if (lane == 0) rht_issue_mma(st, smem_u32(sm.hmat), 256, tmem, &sm.mma_bar[grp]);
    ++mma_issued;
    return true;
  };
  // Every warp of the group: wait for transform jt, then (after reading)
  // count itself out of the group's tensor memory.
  auto transform_wait = [&] {
    const bool done = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&sm.mma_bar[grp], (uint32_t)(jt & 1), a.status));
    tcgen05_after_sync();
    return done;
  };
  auto transform_done = [&] {
    tcgen05_before_sync();
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      atomicAdd(&sm.tfree[grp], 1u);
    }
    ++jt;
  };

  // phase A: max|x| and max|RHT(x)| of this group's tiles
  bool ok = true;
  float m_row = 0.0f, m_col = 0.0f;
  for (int k = grp; k < n; k += kGroups) {
    const int s = k % S;
    if (!ring.wait_full(k)) {
      ok = false;
      break;
    }
    const uint32_t st = ring.stage(s);
    if (!transform(st)) {
      ok = false;
      break;
    }
    const float mr = quarter_absmax(st, cw);
    if (!transform_wait()) {
      ok = false;
      break;
    }
    const float mc = rht_col_max(tmem, cw);
    transform_done();
    m_row = fmaxf(m_row, mr);
    m_col = fmaxf(m_col, mc);
    if (k + S < n)  // tile k leaves shared memory (the transform has read it too)
      ring.release(s, k + S, k + S >= kept_from ? stream : keep, __float_as_uint(mr) ^ __float_as_uint(mc));
  }
  if (!ok) *sm.abort_flag = 1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m_row = fmaxf(m_row, __shfl_xor_sync(0xFFFFFFFFu, m_row, o));
    m_col = fmaxf(m_col, __shfl_xor_sync(0xFFFFFFFFu, m_col, o));
  }
  const unsigned gen = *sm.gen;
  if (lane == 0) {
    atomicMax(&sm.cta_max[0], __float_as_uint(m_row));
    atomicMax(&sm.cta_max[1], __float_as_uint(m_col));
    __threadfence_block();
    if (atomicAdd(sm.cta_in, 1u) == (unsigned)(kRWarps - 1)) {
      __threadfence_block();
      const volatile unsigned* cm = sm.cta_max;
      grid_arrive2(ws, gen, __uint_as_float(cm[0]), __uint_as_float(cm[1]));
    }
  }
  if (tid == 0) {
    float amax_row = 0.0f, amax_col = 0.0f;
    const bool gok = grid_wait_max(ws, gen, (unsigned)G, a.status, &amax_row, &amax_col);
    if (!gok) *sm.abort_flag = 1;
    if (b == 0 && gok && !*sm.abort_flag) {
      if (a.amax_row) *const_cast<float*>(a.amax_row) = amax_row;
      if (a.amax_col) *const_cast<float*>(a.amax_col) = amax_col;
    }
    sm.g[0] = global_encode_scale(amax_row);
    sm.g[1] = global_encode_scale(amax_col);
  }
  __syncthreads();
  const bool early_exit = *sm.abort_flag != 0;
  const float g_row = sm.g[0], g_col = sm.g[1];
  if (!early_exit) {
    if (tid < 128)
      sm.rtab_row[tid] = encode_factor((uint32_t)tid, g_row);
    else if (tid < 256)
      sm.rtab_col[tid - 128] = encode_factor((uint32_t)(tid - 128), g_col);
  }
  __syncthreads();

  // phase B: descending k, this group's tiles: transform (one thread), rows
  // (wide pass), columns (tensor-memory epilogue); the stage is released once
  // both have read it; scales as in fused.cu (bulk copies for the 128x4
  // layout, else each warp writes back its share of the previous tile's).
  const bool do_row = a.rowwise != 0, do_col = a.colwise != 0;
  const int k_top = n - 1 - ((n - 1 - grp) % kGroups + kGroups) % kGroups;
  const volatile int* abort_flag = sm.abort_flag;
  auto buffer = [&](int it) { return sm.sc + (size_t)((grp * 2 + (it & 1)) * 2) * kScRegion; };
  auto write_back = [&](int kk, int it) {
    const int q = grp * 2 + (it & 1);
    int64_t r0, c0;
    ring.tile_rc(kk, r0, c0);
    return sp::write_back_share<kCast1D, WPT>(buffer(it), &sm.staged[q], &sm.wb[q],
                                              (unsigned)(WPT * ((it >> 1) + 1)), cw, a, r0, c0, do_row, do_col);
  };
  int it = 0, k_prev = -1;
  int pending_q = -1;  // lane 0, kBulk: buffer of the copies this warp issued, not yet freed
  for (int k = early_exit ? -1 : k_top; k >= 0; k -= kGroups, ++it) {
    const int s = k % S;
    if constexpr (kBulk) sp::bulk_free<WPT>(pending_q, sm.wb);
    if (*abort_flag) break;
    if (k < kept_from && !ring.wait_full(k)) {
      *sm.abort_flag = 1;
      break;
    }
    int64_t r0, c0;
    ring.tile_rc(k, r0, c0);
    uint8_t* sc = buffer(it);
    const uint32_t st = ring.stage(s);
    bool good = true;
    if (do_col) good = transform(st);
    uint32_t tok = 0;
    RowHooks hooks{&tok, &sm.wb[grp * 2 + (it & 1)], (unsigned)(WPT * (it >> 1)), &good, a.status};
    if (do_row)
      wide_pass_any<kCast1D, kBulk>(st, sm.rtab_row, smem_u32(sc), smem_u32(sc + kScRegion), a, r0, c0, g_row,
                                    true, false, cw, hooks);
    else
      hooks.scale_wait();
    if (do_col && good) {
      if (transform_wait())
        tok ^= rht_col_epilogue<kBulk>(tmem, cw, sm.rtab_col, sc + kScRegion, a, r0, c0, g_col);
      else
        good = false;
      transform_done();
    }
    ring.release(s, k - S, stream, tok);
    if (!good) {
      *sm.abort_flag = 1;
      break;
    }
    if constexpr (kBulk) {
      sp::bulk_staged<WPT>(&sm.staged[grp * 2 + (it & 1)], grp * 2 + (it & 1), sc, a, r0, c0, do_row, do_col,
                           pending_q);
    } else {
      sp::count_staged(&sm.staged[grp * 2 + (it & 1)]);
      if (k_prev >= 0 && !write_back(k_prev, it - 1)) {
        *sm.abort_flag = 1;
        break;
      }
      k_prev = k;
    }
  }
  if (!kBulk && k_prev >= 0 && !*abort_flag && !write_back(k_prev, it - 1)) *sm.abort_flag = 1;
  if constexpr (kBulk) {
    sp::bulk_free<WPT>(pending_q, sm.wb);
    if (lane == 0) bulk_wait_all();
  }
  // A transform this warp issued and nobody waited for (after an abort) ends
  // before the tensor memory is released (bounded).
  if (cw == 0 && mma_issued > jt && lane == 0)
    mbar_wait_bounded(&sm.mma_bar[grp], (uint32_t)((mma_issued - 1) & 1), a.status);
  tcgen05_before_sync();
  __syncwarp();
  unsigned last = 0;
  if (lane == 0) last = (atomicAdd(sm.exited, 1u) == (unsigned)(kRWarps - 1)) ? 1u : 0u;
  last = __shfl_sync(0xFFFFFFFFu, last, 0);
  if (last) {
    // the last warp out: every other warp is done with tensor memory and,
    // after an abort, lets the CTA's copies still in flight land (bounded)
    tcgen05_after_sync();
    tmem_dealloc(tmem_all, kTmemCols);
    if (lane == 0 && *abort_flag) ring.drain();
  }
}

template <bool kBulk>
cudaError_t launch_rht_t(const CUtensorMap& map, const CastArgs& a, SinglePassWorkspace* ws, const LaunchCtx& ctx) {
  return sp::launch_persistent<fused_rht_kernel<kBulk>>(rht_smem_bytes(), kRThreads, map, a, a.num_tiles, ws, ctx);
}

}  // namespace

cudaError_t launch_single_pass_rht(const CUtensorMap& map, CastArgs args, SinglePassWorkspace* ws,
                                   const LaunchCtx& ctx) {
  const int64_t tiles_m = (args.M + kTile - 1) / kTile, tiles_n = (args.N + kTile - 1) / kTile;
  args.tiles_n = (int)tiles_n;
  args.num_tiles = (int)(tiles_m * tiles_n);
  if (args.swizzled) return launch_rht_t<true>(map, args, ws, ctx);  // M, N multiples of 128 (validated)
  return launch_rht_t<false>(map, args, ws, ctx);
}

}  // namespace nvfp4
