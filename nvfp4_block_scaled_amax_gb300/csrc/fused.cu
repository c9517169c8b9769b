// fused.cu -- single-launch NVFP4 quantize: per-tensor amax and the fused
// row-wise + column-wise cast in one persistent kernel.
//
// One CTA per SM (cooperative launch, all CTAs co-resident), 16 warps in
// groups; a group casts one 128x128 tile at a time (BF16: groups of 4 warps
// with the wide 8x16-per-lane mapping, FP32: groups of 8 with 8x8 sub-blocks):
//   * tile k of the CTA (t_k = blockIdx + k * gridDim) goes through stage
//     k % S of a shared-memory ring and is handled by group k % groups; its
//     TMA completion is an mbarrier whose phase parity is (k / S) & 1 in both
//     phases (the fills of a stage are sequential);
//   * when the warps of a group are done with a stage, the last of them (a
//     shared-memory counter per stage) writes the tile's staged scales back
//     and issues the next load into the stage, so no warp ever waits for the
//     whole CTA;
//   * phase A streams the CTA's tiles through the ring computing max|x|; the
//     last S tiles stay in shared memory;
//   * a grid barrier in the caller's workspace combines the CTA maxima
//     (the amax is written to both direction buffers, "Write both NVFP4 amax
//     buffers");
//   * phase B casts the resident tiles first, then reloads the others in
//     reverse order (most recently read first, so mostly from L2; phase A
//     marked them evict-last), writing codes, and scales in the compact or
//     cuBLAS 128x4 layout.
// x is read from HBM once; the call is one launch.  The stage ring, the
// scale write-back and the cooperative launch are shared with fused_rht.cu
// (single_pass.cuh).
#include "common.cuh"
#include "grid.cuh"
#include "kernels.h"
#include "single_pass.cuh"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace {

using namespace tile;

constexpr int kWarps = 16;
constexpr int kFusedThreads = 32 * kWarps;

template <typename T>
struct FusedCfg;
template <>
struct FusedCfg<uint16_t> {
  static constexpr int kStages = 6;
  static constexpr int kWarpsPerTile = 4;  // wide mapping
};
template <>
struct FusedCfg<float> {
  static constexpr int kStages = 3;  // 3 x 64 KB tiles (more loads in flight than 2: phase A -1 µs at 4096x3072)
  static constexpr int kWarpsPerTile = 8;  // 8x8 sub-blocks
};

// Phase A keeps the 16x16 maxima of the tiles of each CTA (2D, BF16, up to
// kPreTiles tiles per CTA), so that phase B need not find them again.
constexpr int kPreTiles = 32;

template <typename T>
__host__ __device__ constexpr int fused_groups() {
  return kWarps / FusedCfg<T>::kWarpsPerTile;
}
// stages | per group two staged-scale buffers (row and column regions) |
// encode-factor tables | mbarriers | stage and scale-buffer counters | misc
template <typename T>
__host__ __device__ constexpr size_t fused_smem_bytes() {
  return 1024 + (size_t)FusedCfg<T>::kStages * tile_bytes<T>() + (size_t)fused_groups<T>() * 2 * 2 * kScRegion +
         2 * 128 * 4 + 20 * FusedCfg<T>::kStages + 16 * fused_groups<T>() + 16 + 64 +
         (sizeof(T) == 2 ? kPreTiles * 64 * 2 : 0);
}

struct FSmem {
  uint8_t* stages;   // [S][tile]
  uint8_t* sc;       // [groups][2][2][kScRegion] staged row / column scales, two buffers per group
  float* rtab_row;   // [128]
  float* rtab_col;   // [128]
  uint64_t* full;    // [S]
  unsigned* loaded;  // [S] warps done reading the stage's tile data
  unsigned* issued;  // [S] loads issued into the stage so far
  int* tile_in;      // [S] tile index of the stage's latest issued load
  unsigned* staged;  // [groups][2] warps done staging into the buffer (all uses so far)
  unsigned* wb;      // [groups][2] warps done writing the buffer's scales back (all uses so far)
  unsigned* exited;  // [1] warps done with phase B
  unsigned* gen;     // [1] this call's barrier generation
  unsigned* cta_max; // [1] the CTA's max|x| bits (phase A)
  unsigned* cta_in;  // [1] warps done with phase A
  float* amax;       // [1] broadcast of the global amax
  int* abort_flag;   // [1]
  uint16_t* pre;     // [kPreTiles][64] 2D (BF16): 16x16 tile maxima found in phase A
};

// The stage hooks the cast passes call (see wide_pass).
template <class D, class W, class St>
struct StageHooksT {
  D done_fn;
  W wait_fn;
  St staged_fn;
  const uint16_t* pre;  // 2D: the tile's 16x16 maxima found in phase A, or null
  __device__ __forceinline__ void data_done(uint32_t token) const { done_fn(token); }
  __device__ __forceinline__ void scale_wait() const { wait_fn(); }
  __device__ __forceinline__ void scales_staged() const { staged_fn(); }
  __device__ __forceinline__ const uint16_t* tile_max() const { return pre; }
};
template <class D, class W, class St>
__device__ __forceinline__ StageHooksT<D, W, St> make_hooks(D d, W w, St st, const uint16_t* pre = nullptr) {
  return StageHooksT<D, W, St>{d, w, st, pre};
}


template <typename T>
__device__ __forceinline__ FSmem fcarve(uint8_t* raw) {
  constexpr int S = FusedCfg<T>::kStages;
  FSmem s;
  // offset arithmetic on the shared array itself, so that every carved
  // pointer stays a known shared-memory pointer (ld.shared / atom.shared)
  uint8_t* p = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
  s.stages = p;
  p += (size_t)S * tile_bytes<T>();
  s.sc = p;
  p += (size_t)fused_groups<T>() * 2 * 2 * kScRegion;
  s.rtab_row = reinterpret_cast<float*>(p);
  s.rtab_col = s.rtab_row + 128;
  s.full = reinterpret_cast<uint64_t*>(s.rtab_col + 128);
  s.loaded = reinterpret_cast<unsigned*>(s.full + S);
  s.issued = s.loaded + S;
  s.tile_in = reinterpret_cast<int*>(s.issued + S);
  s.staged = reinterpret_cast<unsigned*>(s.tile_in + S);
  s.wb = s.staged + 2 * fused_groups<T>();
  s.exited = s.wb + 2 * fused_groups<T>();
  s.gen = s.exited + 1;
  s.cta_max = s.exited + 2;
  s.cta_in = s.exited + 3;
  s.amax = reinterpret_cast<float*>(s.exited + 4);
  s.abort_flag = reinterpret_cast<int*>(s.amax + 1);
  s.pre = reinterpret_cast<uint16_t*>(s.abort_flag + 1);
  return s;
}

// max|x| over this warp's share of a staged tile: BF16, a quarter of the
// tile (8 KB, sixteen 16-byte loads per lane, consecutive lanes on
// consecutive chunks); FP32, its 8x8 sub-block.
template <typename T>
__device__ __forceinline__ float share_absmax(uint32_t stage, int cw) {
  const int lane = threadIdx.x & 31;
  if constexpr (sizeof(T) == 2) {
    const uint32_t base = stage + (uint32_t)cw * 8192u + (uint32_t)lane * 16u;
    uint32_t acc = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint4 v = lds128(base + 512u * k);
      acc = xsa(acc, xsa(xsa(v.x, v.y), xsa(v.z, v.w)));
    }
    acc &= 0x7FFF7FFFu;
    return fmaxf(bf16_lo(acc), bf16_hi(acc));
  } else {
    const int bx = cw & 1, q = cw >> 1, j = lane & 7, i = lane >> 3;
    Sub<T> s;
    load_sub<T>(stage, bx, 32 * q + 8 * i, j, s);
    float m = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
#pragma unroll
      for (int c = 0; c < 8; ++c) m = fmaxf(m, fabsf(s.v(k, c)));
    return m;
  }
}

// kBulk (BF16, 128x4 layout, M and N multiples of 128): the scales are
// staged in the stored byte order and leave by bulk copies (a separate
// instantiation, so the compact path carries none of that code).
template <typename T, int MODE, bool kBulk>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tmap, const CastArgs a, SinglePassWorkspace* ws) {
  static_assert(!kBulk || sizeof(T) == 2, "bulk scale copies: BF16 wide mapping only");
  constexpr int S = FusedCfg<T>::kStages;
  constexpr int WPT = FusedCfg<T>::kWarpsPerTile;
  constexpr int kGroups = kWarps / WPT;
  extern __shared__ uint8_t smem_raw[];
  const FSmem sm = fcarve<T>(smem_raw);
  if (a.noop != nullptr && *a.noop == 1.0f) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int n = (a.num_tiles - 1 - b) / G + 1;  // tiles t_k = b + k * G, k < n (grid <= tiles)
  const int kept_from = n > S ? n - S : 0;      // tiles k >= kept_from stay staged after phase A
  const sp::StageRing<T, S, WPT> ring{sm.stages, sm.full, sm.loaded, sm.issued, sm.tile_in, &tmap, b, G,
                                      a.tiles_n, a.status};

  // Loads: phase A reads tiles 0..n-1 (the ones reloaded in phase B are kept
  // in L2 with evict-last), phase B reloads tiles kept_from-1 .. 0.
  const uint64_t keep = l2_policy_evict_last(), stream = l2_policy_evict_first();
  if (tid == 0) {
    *sm.gen = ld_acquire_gpu(&ws->gen);  // this call's barrier generation
    ring.init();
    for (int q = 0; q < 2 * kGroups; ++q) {
      sm.staged[q] = 0;
      sm.wb[q] = 0;
    }
    *sm.abort_flag = 0;
    *sm.exited = 0;
    *sm.cta_max = 0;
    *sm.cta_in = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmap);
    for (int k = 0; k < S && k < n; ++k) ring.issue(k, k >= kept_from ? stream : keep);
  }
  __syncthreads();

  const int grp = warp / WPT, cw = warp % WPT;
  bool ok = true;

  // phase A: max|x| of this group's tiles (k == grp mod kGroups)
  constexpr bool kPre = MODE == kCast2D && sizeof(T) == 2;
  const bool use_pre = kPre && n <= kPreTiles;
  float m = 0.0f;
  for (int k = grp; k < n; k += kGroups) {
    const int s = k % S;
    if (!ring.wait_full(k)) {
      ok = false;
      break;
    }
    float mk;
    if (use_pre) {
      // the wide partition of phase B: record the tile's 16x16 maxima
      SubW sw;
      const int wr = cw >> 1, wc = cw & 1, i = lane >> 2, j = lane & 3;
      load_sub_w(ring.stage(s), wc, 64 * wr + 8 * i, j, i & 1, sw);
      uint32_t acc;
      mk = wide_tile_max(sw.a, sw.b, acc);
      if ((i & 1) == 0) sm.pre[k * 64 + (4 * wr + (i >> 1)) * 8 + 4 * wc + j] = (uint16_t)(__float_as_uint(mk) >> 16);
    } else {
      mk = share_absmax<T>(ring.stage(s), cw);
    }
    m = fmaxf(m, mk);
    if (k + S < n)  // tile k leaves shared memory: load tile k + S into its stage
      ring.release(s, k + S, k + S >= kept_from ? stream : keep, __float_as_uint(mk));
  }
  if (!ok) *sm.abort_flag = 1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  // Every warp counts in (a warp that lost a wait too, so the others are not
  // held up); the CTA's last one arrives at the grid barrier for the CTA;
  // thread 0 waits for all CTAs.
  const unsigned gen = *sm.gen;
  if (lane == 0) {
    atomicMax(sm.cta_max, __float_as_uint(m));
    __threadfence_block();
    if (atomicAdd(sm.cta_in, 1u) == (unsigned)(kWarps - 1)) {
      __threadfence_block();
      grid_arrive(ws, gen, __uint_as_float(*reinterpret_cast<volatile unsigned*>(sm.cta_max)));
    }
  }
  if (tid == 0) {
    float amax = 0.0f;
    const bool gok = grid_wait_max(ws, gen, (unsigned)G, a.status, &amax);
    if (!gok) *sm.abort_flag = 1;
    if (b == 0 && gok && !*sm.abort_flag) {
      if (a.amax_row) *const_cast<float*>(a.amax_row) = amax;
      if (a.amax_col) *const_cast<float*>(a.amax_col) = amax;
    }
    *sm.amax = global_encode_scale(amax);
  }
  __syncthreads();
  if (*sm.abort_flag) {
    // let this CTA's copies in flight (the last load into each stage) land,
    // bounded, before leaving
    if (tid == 0) ring.drain();
    return;
  }
  const float g = *sm.amax;
  if (tid < 128)
    sm.rtab_row[tid] = encode_factor((uint32_t)tid, g);
  else if (tid < 256)
    sm.rtab_col[tid - 128] = encode_factor((uint32_t)(tid - 128), g);
  __syncthreads();

  // phase B: descending k, this group's tiles.  A stage's data is released
  // (tile k - S loaded into it) as soon as the group's warps have read their
  // sub-tiles.  Scales are staged in the group's own two buffers, used in
  // turn; during its next tile each warp writes back its share of the
  // previous tile's scales (waiting, bounded, until all the group's warps
  // have staged them), and a buffer is reused only after every warp's share
  // of its previous contents has been written back.
  const bool do_row = a.rowwise != 0, do_col = a.colwise != 0;
  const int k_top = n - 1 - ((n - 1 - grp) % kGroups + kGroups) % kGroups;  // largest k < n, k == grp mod kGroups
  const volatile int* abort_flag = sm.abort_flag;
  auto buffer = [&](int it) { return sm.sc + (size_t)((grp * 2 + (it & 1)) * 2) * kScRegion; };
  // this warp's share of tile kk's (iteration it's) scale write-back
  auto write_back = [&](int kk, int it) {
    const int q = grp * 2 + (it & 1);
    int64_t r0, c0;
    ring.tile_rc(kk, r0, c0);
    return sp::write_back_share<MODE, WPT>(buffer(it), &sm.staged[q], &sm.wb[q], (unsigned)(WPT * ((it >> 1) + 1)),
                                           cw, a, r0, c0, do_row, do_col);
  };
  int it = 0, k_prev = -1;
  int pending_q = -1;  // lane 0, kBulk: buffer of the copies this warp issued, not yet freed
  for (int k = k_top; k >= 0; k -= kGroups, ++it) {
    const int s = k % S;
    if constexpr (kBulk) sp::bulk_free<WPT>(pending_q, sm.wb);
    if (*abort_flag) break;
    if (k < kept_from && !ring.wait_full(k)) {  // a wait ran out: outputs unfinished
      *sm.abort_flag = 1;
      break;
    }
    int64_t r0, c0;
    ring.tile_rc(k, r0, c0);
    uint8_t* sc = buffer(it);
    const uint32_t st = ring.stage(s);
    const unsigned* wbq = &sm.wb[grp * 2 + (it & 1)];
    bool scales_ok = true;
    // the buffer's previous contents (iteration it - 2) are written back
    auto scale_wait = [&] {
      scales_ok = sp::warp_wait_count(wbq, (unsigned)(WPT * (it >> 1)), a.status) && scales_ok;
    };
    // 128x4 layout: once all of the group's warps have staged their scales,
    // the last of them writes the tile's scales with one bulk copy per
    // direction; the buffer is freed once the copies have read it (at that
    // warp's next iteration)
    auto staged = [&] {
      if constexpr (kBulk)
        sp::bulk_staged<WPT>(&sm.staged[grp * 2 + (it & 1)], grp * 2 + (it & 1), sc, a, r0, c0, do_row, do_col,
                             pending_q);
    };
    if constexpr (sizeof(T) == 2) {
      const auto hooks = make_hooks([&](uint32_t token) { ring.release(s, k - S, stream, token); }, scale_wait,
                                    staged, use_pre ? sm.pre + k * 64 : nullptr);
      wide_pass_any<MODE, kBulk>(st, sm.rtab_row, smem_u32(sc), smem_u32(sc + kScRegion), a, r0, c0, g, do_row,
                                 do_col, cw, hooks);
    } else {
      scale_wait();
      block_pass_any<T, MODE>(st, sm.rtab_row, sm.rtab_col, smem_u32(sc), smem_u32(sc + kScRegion), a, r0, c0, g,
                              g, do_row, do_col, cw);
      __syncwarp();
      __threadfence_block();  // the warp's reads of the stage are done
      ring.release(s, k - S, stream, 0u);
    }
    if (!scales_ok) {  // a wait ran out: outputs unfinished
      *sm.abort_flag = 1;
      break;
    }
    if constexpr (!kBulk) {
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
    if (lane == 0) bulk_wait_all();  // this warp's scale copies (if any) are complete
  }
  // After an abort, the last warp to leave lets the copies still in flight
  // (the latest load into each stage) land, bounded, before the CTA exits.
  __syncwarp();
  if (lane == 0 && atomicAdd(&sm.exited[0], 1u) == (unsigned)(kWarps - 1) && *abort_flag) ring.drain();
}

template <typename T, int MODE, bool kBulk>
cudaError_t launch_fused_t(const CUtensorMap& map, const CastArgs& a, SinglePassWorkspace* ws, const LaunchCtx& ctx) {
  return sp::launch_persistent<fused_kernel<T, MODE, kBulk>>(fused_smem_bytes<T>(), kFusedThreads, map, a, ws, ctx);
}

}  // namespace

int single_pass_grid(int64_t M, int64_t N, const LaunchCtx& ctx) {
  const int64_t tiles = ((M + kTile - 1) / kTile) * ((N + kTile - 1) / kTile);
  return (int)(tiles < ctx.num_sms ? tiles : ctx.num_sms);
}

cudaError_t launch_single_pass(const CUtensorMap& map, bool bf16, int mode, CastArgs args, SinglePassWorkspace* ws,
                               const LaunchCtx& ctx) {
  const int64_t tiles_m = (args.M + kTile - 1) / kTile, tiles_n = (args.N + kTile - 1) / kTile;
  args.tiles_n = (int)tiles_n;
  args.num_tiles = (int)(tiles_m * tiles_n);
  if (bf16) {
    // the 128x4 layout requires M and N multiples of 128 (validated): every tile is whole
    if (args.swizzled) {
      if (mode == kCast1D) return launch_fused_t<uint16_t, kCast1D, true>(map, args, ws, ctx);
      return launch_fused_t<uint16_t, kCast2D, true>(map, args, ws, ctx);
    }
    if (mode == kCast1D) return launch_fused_t<uint16_t, kCast1D, false>(map, args, ws, ctx);
    return launch_fused_t<uint16_t, kCast2D, false>(map, args, ws, ctx);
  }
  if (mode == kCast1D) return launch_fused_t<float, kCast1D, false>(map, args, ws, ctx);
  return launch_fused_t<float, kCast2D, false>(map, args, ws, ctx);
}

}  // namespace nvfp4
