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
//
// The same kernel body quantizes a grouped tensor (grouped.h: x stacks
// member tensors, each with its own amax): the tiles of all members form one
// list, phase A keeps a maximum per member (a tile that reaches past its
// member's last row skips the next member's rows), the grid barrier combines
// the members' maxima in the workspace, and phase B casts every tile with its
// member's outputs and global scale (an encode-factor table per member).
#include "common.cuh"
#include "grid.cuh"
#include "grouped.h"
#include "kernels.h"
#include "single_pass.cuh"
#include "tile_ops.cuh"

namespace nvfp4 {
namespace {

using namespace tile;

constexpr int kWarps = 16;
constexpr int kFusedThreads = 32 * kWarps;

template <typename T, bool kGrouped = false>
struct FusedCfg;
template <bool kGrouped>
struct FusedCfg<uint16_t, kGrouped> {
  // grouped: five stages, beside the members' encode-factor tables (32 KB)
  static constexpr int kStages = kGrouped ? 5 : 6;
  static constexpr int kWarpsPerTile = 4;  // wide mapping
};
template <bool kGrouped>
struct FusedCfg<float, kGrouped> {
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
// Grouped: what a tile needs of its member, copied from the parameter
// table into shared memory once (reads through the parameter's address are
// slow).
struct MemberInfo {
  uint8_t* data_row;
  uint8_t* scale_row;
  uint8_t* data_col;
  uint8_t* scale_col;
  int64_t row0, rows;
};
// Grouped: per member an encode-factor table, a maximum, a global scale and
// its MemberInfo; the tile prefix sums.
constexpr size_t kMemberTables = (size_t)kMaxGroups * 128 * 4 + (size_t)kMaxGroups * 4 * 2 +
                                 (size_t)kMaxGroups * sizeof(MemberInfo) + (size_t)(kMaxGroups + 2) * 4 + 16;

// stages | per group two staged-scale buffers (row and column regions) |
// encode-factor tables | mbarriers | stage and scale-buffer counters | misc
// | 2D phase-A maxima | grouped: the members' tables and maxima
template <typename T, bool kGrouped = false>
__host__ __device__ constexpr size_t fused_smem_bytes() {
  return 1024 + (size_t)FusedCfg<T, kGrouped>::kStages * tile_bytes<T>() +
         (size_t)fused_groups<T>() * 2 * 2 * kScRegion + 2 * 128 * 4 + 20 * FusedCfg<T, kGrouped>::kStages +
         16 * fused_groups<T>() + 16 + 64 + (sizeof(T) == 2 ? kPreTiles * 64 * 2 : 0) +
         (kGrouped ? kMemberTables : 0);
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
  float* mtab;       // grouped: [kMaxGroups][128] each member's encode factors
  unsigned* mmax;    // grouped: [kMaxGroups] the CTA's max|x| bits per member (phase A)
  float* mg;         // grouped: [kMaxGroups] each member's global encode scale
  MemberInfo* minfo; // grouped: [kMaxGroups]
  int* mstart;       // grouped: [kMaxGroups + 1] the members' tile prefix sums
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


template <typename T, bool kGrouped>
__device__ __forceinline__ FSmem fcarve(uint8_t* raw) {
  constexpr int S = FusedCfg<T, kGrouped>::kStages;
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
  s.mtab = reinterpret_cast<float*>(s.pre + (sizeof(T) == 2 ? kPreTiles * 64 : 0));
  s.mmax = reinterpret_cast<unsigned*>(s.mtab + (kGrouped ? kMaxGroups * 128 : 0));
  s.mg = reinterpret_cast<float*>(s.mmax + kMaxGroups);
  // 16-byte aligned for the pointers and 64-bit fields
  s.minfo = reinterpret_cast<MemberInfo*>(reinterpret_cast<uint8_t*>(s.mg + kMaxGroups) +
                                          ((16u - (smem_u32(s.mg + kMaxGroups) & 15u)) & 15u));
  s.mstart = reinterpret_cast<int*>(s.minfo + kMaxGroups);
  return s;
}

// max|x| over this warp's share of a staged tile: BF16, a quarter of the
// tile (8 KB, sixteen 16-byte loads per lane, consecutive lanes on
// consecutive chunks: load k holds tile row 64 (cw & 1) + lane / 8 + 4 k of
// box cw >> 1); FP32, its 8x8 sub-block.  kMask (grouped, BF16): tile rows
// from `lim` on are not part of the tile's member and are skipped.
template <typename T, bool kMask = false>
__device__ __forceinline__ float share_absmax(uint32_t stage, int cw, int lim = kTile) {
  const int lane = threadIdx.x & 31;
  if constexpr (sizeof(T) == 2) {
    const uint32_t base = stage + (uint32_t)cw * 8192u + (uint32_t)lane * 16u;
    const int row0 = 64 * (cw & 1) + (lane >> 3);
    uint32_t acc = 0;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint4 v = lds128(base + 512u * k);
      const uint32_t m = xsa(xsa(v.x, v.y), xsa(v.z, v.w));
      if (!kMask || row0 + 4 * k < lim) acc = xsa(acc, m);
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

// Where the kernel body's tiles come from: one tensor (its arguments held by
// value: reading them through the parameter's address instead made every
// call of a small tensor several microseconds slower) ...
struct PlainSrc {
  static constexpr bool kGrouped = false;
  using Tiles = sp::PlainTiles;
  CastArgs a;
  __device__ __forceinline__ int num_tiles() const { return a.num_tiles; }
  __device__ __forceinline__ const float* noop() const { return a.noop; }
  __device__ __forceinline__ unsigned* status() const { return a.status; }
  __device__ __forceinline__ bool rowwise() const { return a.rowwise != 0; }
  __device__ __forceinline__ bool colwise() const { return a.colwise != 0; }
  __device__ __forceinline__ Tiles tiles() const { return Tiles{a.tiles_n}; }
  // tile t: its member (0), first row and first column
  __device__ __forceinline__ MemberTile at(int t) const {
    const int tr = t / a.tiles_n;
    return MemberTile{0, (int64_t)tr * kTile, (int64_t)(t - tr * a.tiles_n) * kTile};
  }
  __device__ __forceinline__ const CastArgs& member(int) const { return a; }
};
// ... or the members of a grouped tensor (grouped.h): tile t of all members,
// each member seen as a plain tensor of its own.  The scalars are held by
// value, the per-member records in shared memory (MemberInfo).
struct GroupedSrc {
  static constexpr bool kGrouped = true;
  // TMA coordinates of tile t from the shared-memory records
  struct Tiles {
    const MemberInfo* mi;
    const int* start;
    int members, tiles_n;
    __device__ __forceinline__ MemberTile at(int t) const {
      MemberTile p;
      p.g = member_of(start, members, t);
      const int lt = t - start[p.g];
      const int tr = lt / tiles_n;
      p.r0 = (int64_t)tr * kTile;
      p.c0 = (int64_t)(lt - tr * tiles_n) * kTile;
      return p;
    }
    __device__ __forceinline__ void xy(int t, int32_t& x, int32_t& y) const {
      const MemberTile p = at(t);
      x = (int32_t)p.c0;
      y = (int32_t)(mi[p.g].row0 + p.r0);
    }
  };
  Tiles tl;
  int ntiles;
  int64_t N;
  const float* noop_;
  unsigned* status_;
  int rowwise_, colwise_, swizzled_;
  const GroupedArgs* ga;  // the parameter table: the amax buffers, read once at the barrier
  __device__ __forceinline__ int num_tiles() const { return ntiles; }
  __device__ __forceinline__ const float* noop() const { return noop_; }
  __device__ __forceinline__ unsigned* status() const { return status_; }
  __device__ __forceinline__ bool rowwise() const { return rowwise_ != 0; }
  __device__ __forceinline__ bool colwise() const { return colwise_ != 0; }
  __device__ __forceinline__ Tiles tiles() const { return tl; }
  __device__ __forceinline__ MemberTile at(int t) const { return tl.at(t); }
  __device__ __forceinline__ int members() const { return tl.members; }
  __device__ __forceinline__ int64_t rows(int g) const { return tl.mi[g].rows; }
  __device__ __forceinline__ CastArgs member(int g) const {
    const MemberInfo& i = tl.mi[g];
    CastArgs m = {};
    m.M = i.rows;
    m.N = N;
    m.data_row = i.data_row;
    m.scale_row = i.scale_row;
    m.data_col = i.data_col;
    m.scale_col = i.scale_col;
    m.noop = noop_;
    m.status = status_;
    m.rowwise = rowwise_;
    m.colwise = colwise_;
    m.swizzled = swizzled_;
    m.tiles_n = tl.tiles_n;
    return m;
  }
};

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// kBulk (BF16, 128x4 layout, M and N multiples of 128): the scales are
// staged in the stored byte order and leave by bulk copies (a separate
// instantiation, so the compact path carries none of that code).
template <typename T, int MODE, bool kBulk, class Src>
__device__ __forceinline__ void fused_body(const CUtensorMap& tmap, const Src& src, SinglePassWorkspace* ws) {
  static_assert(!kBulk || sizeof(T) == 2, "bulk scale copies: BF16 wide mapping only");
  constexpr bool kGrouped = Src::kGrouped;
  static_assert(!kGrouped || sizeof(T) == 2, "grouped: BF16 wide mapping only");
  constexpr int S = FusedCfg<T, kGrouped>::kStages;
  constexpr int WPT = FusedCfg<T, kGrouped>::kWarpsPerTile;
  constexpr int kGroups = kWarps / WPT;
  extern __shared__ uint8_t smem_raw[];
  const FSmem sm = fcarve<T, kGrouped>(smem_raw);
  if (src.noop() != nullptr && *src.noop() == 1.0f) return;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, b = blockIdx.x;
  const int n = (src.num_tiles() - 1 - b) / G + 1;  // tiles t_k = b + k * G, k < n (grid <= tiles)
  const int kept_from = n > S ? n - S : 0;          // tiles k >= kept_from stay staged after phase A
  const sp::StageRing<T, S, WPT, typename Src::Tiles> ring{sm.stages, sm.full,  sm.loaded,    sm.issued,    sm.tile_in,
                                                           &tmap,     b,        G,            src.tiles(), src.status()};

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
  if (kGrouped && tid < kMaxGroups) sm.mmax[tid] = 0u;
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
    // grouped: the tile's member, and its rows in the tile (the rest belong
    // to the next member)
    MemberTile mt = {0, 0, 0};
    int lim = kTile;
    if constexpr (kGrouped) {
      mt = src.at(b + k * G);
      const int64_t left = src.rows(mt.g) - mt.r0;
      lim = left < kTile ? (int)left : kTile;
    }
    float mk;
    if (use_pre) {
      // the wide partition of phase B: record the tile's 16x16 maxima
      SubW sw;
      const int wr = cw >> 1, wc = cw & 1, i = lane >> 2, j = lane & 3;
      load_sub_w(ring.stage(s), wc, 64 * wr + 8 * i, j, i & 1, sw);
      if (kGrouped && lim < kTile) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (64 * wr + 8 * i + kk >= lim) {
#pragma unroll
            for (int p = 0; p < 4; ++p) sw.a[kk][p] = sw.b[kk][p] = 0u;
          }
      }
      uint32_t acc;
      mk = wide_tile_max(sw.a, sw.b, acc);
      if ((i & 1) == 0) sm.pre[k * 64 + (4 * wr + (i >> 1)) * 8 + 4 * wc + j] = (uint16_t)(__float_as_uint(mk) >> 16);
    } else {
      mk = share_absmax<T, kGrouped>(ring.stage(s), cw, lim);
    }
    if constexpr (kGrouped) {
      float mw = mk;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xFFFFFFFFu, mw, o));
      if (lane == 0) atomicMax(&sm.mmax[mt.g], __float_as_uint(mw));
    } else {
      m = fmaxf(m, mk);
    }
    if (k + S < n)  // tile k leaves shared memory: load tile k + S into its stage
      ring.release(s, k + S, k + S >= kept_from ? stream : keep, __float_as_uint(mk));
  }
  if (!ok) *sm.abort_flag = 1;
  const unsigned gen = *sm.gen;
  GroupedBanks* banks = reinterpret_cast<GroupedBanks*>(reinterpret_cast<uint8_t*>(ws) + kGroupedBanksOffset);
  if constexpr (kGrouped) {
    // The CTA's per-member maxima (every warp's, a warp that lost a wait
    // too) go to this call's bank, ordered before thread 0 arrives.
    __syncthreads();
    if (tid < src.members() && sm.mmax[tid] != 0u) {
      red_relaxed_max_gpu(&banks->maxbits[gen & 1u][tid], sm.mmax[tid]);
      __threadfence();
    }
    __syncthreads();
    if (tid == 0) grid_arrive(ws, gen, 0.0f);
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    // Every warp counts in (a warp that lost a wait too, so the others are
    // not held up); the CTA's last one arrives at the grid barrier for the
    // CTA; thread 0 waits for all CTAs.
    if (lane == 0) {
      atomicMax(sm.cta_max, __float_as_uint(m));
      __threadfence_block();
      if (atomicAdd(sm.cta_in, 1u) == (unsigned)(kWarps - 1)) {
        __threadfence_block();
        grid_arrive(ws, gen, __uint_as_float(*reinterpret_cast<volatile unsigned*>(sm.cta_max)));
      }
    }
  }
  if (tid == 0) {
    float amax = 0.0f;
    const bool gok = grid_wait_max(ws, gen, (unsigned)G, src.status(), &amax);
    if (!gok) *sm.abort_flag = 1;
    if constexpr (kGrouped) {
      // every member's maximum, right after the wait (whose acquire orders
      // these relaxed loads after every CTA's arrival; they overlap)
      if (gok)
        for (int q = 0; q < src.members(); ++q) sm.mmax[q] = ld_relaxed_gpu(&banks->maxbits[gen & 1u][q]);
    } else {
      const CastArgs& a = src.member(0);
      if (b == 0 && gok && !*sm.abort_flag) {
        if (a.amax_row) *const_cast<float*>(a.amax_row) = amax;
        if (a.amax_col) *const_cast<float*>(a.amax_col) = amax;
      }
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
  if constexpr (kGrouped) {
    // every member's amax (CTA 0 writes them out), global scale and table
    const int members = src.members();
    if (tid < members) {
      const float am = __uint_as_float(sm.mmax[tid]);
      sm.mg[tid] = global_encode_scale(am);
      if (b == 0) {
        if (src.ga->amax_row[tid]) src.ga->amax_row[tid][0] = am;
        if (src.ga->amax_col[tid]) src.ga->amax_col[tid][0] = am;
      }
    }
    __syncthreads();
    for (int e = tid; e < members * 128; e += kFusedThreads) sm.mtab[e] = encode_factor((uint32_t)(e & 127), sm.mg[e >> 7]);
  } else {
    if (tid < 128)
      sm.rtab_row[tid] = encode_factor((uint32_t)tid, g);
    else if (tid < 256)
      sm.rtab_col[tid - 128] = encode_factor((uint32_t)(tid - 128), g);
  }
  __syncthreads();

  // phase B: descending k, this group's tiles.  A stage's data is released
  // (tile k - S loaded into it) as soon as the group's warps have read their
  // sub-tiles.  Scales are staged in the group's own two buffers, used in
  // turn; during its next tile each warp writes back its share of the
  // previous tile's scales (waiting, bounded, until all the group's warps
  // have staged them), and a buffer is reused only after every warp's share
  // of its previous contents has been written back.
  const bool do_row = src.rowwise(), do_col = src.colwise();
  const int k_top = n - 1 - ((n - 1 - grp) % kGroups + kGroups) % kGroups;  // largest k < n, k == grp mod kGroups
  const volatile int* abort_flag = sm.abort_flag;
  auto buffer = [&](int it) { return sm.sc + (size_t)((grp * 2 + (it & 1)) * 2) * kScRegion; };
  // this warp's share of tile kk's (iteration it's) scale write-back
  auto write_back = [&](int kk, int it) {
    const int q = grp * 2 + (it & 1);
    const MemberTile mt = src.at(b + kk * G);
    const auto& ma = src.member(mt.g);
    return sp::write_back_share<MODE, WPT>(buffer(it), &sm.staged[q], &sm.wb[q], (unsigned)(WPT * ((it >> 1) + 1)),
                                           cw, ma, mt.r0, mt.c0, do_row, do_col);
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
    const MemberTile mt = src.at(b + k * G);
    const int64_t r0 = mt.r0, c0 = mt.c0;
    const auto& ma = src.member(mt.g);
    const float* rtab = kGrouped ? sm.mtab + mt.g * 128 : sm.rtab_row;
    const float gm = kGrouped ? sm.mg[mt.g] : g;
    uint8_t* sc = buffer(it);
    const uint32_t st = ring.stage(s);
    const unsigned* wbq = &sm.wb[grp * 2 + (it & 1)];
    bool scales_ok = true;
    // the buffer's previous contents (iteration it - 2) are written back
    auto scale_wait = [&] {
      scales_ok = sp::warp_wait_count(wbq, (unsigned)(WPT * (it >> 1)), src.status()) && scales_ok;
    };
    // 128x4 layout: once all of the group's warps have staged their scales,
    // the last of them writes the tile's scales with one bulk copy per
    // direction; the buffer is freed once the copies have read it (at that
    // warp's next iteration)
    auto staged = [&] {
      if constexpr (kBulk)
        sp::bulk_staged<WPT>(&sm.staged[grp * 2 + (it & 1)], grp * 2 + (it & 1), sc, ma, r0, c0, do_row, do_col,
                             pending_q);
    };
    if constexpr (sizeof(T) == 2) {
      const auto hooks = make_hooks([&](uint32_t token) { ring.release(s, k - S, stream, token); }, scale_wait,
                                    staged, use_pre ? sm.pre + k * 64 : nullptr);
      wide_pass_any<MODE, kBulk>(st, rtab, smem_u32(sc), smem_u32(sc + kScRegion), ma, r0, c0, gm, do_row, do_col,
                                 cw, hooks);
    } else {
      scale_wait();
      block_pass_any<T, MODE>(st, sm.rtab_row, sm.rtab_col, smem_u32(sc), smem_u32(sc + kScRegion), ma, r0, c0, g,
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
  // Grouped: the CTA read its bank long ago; the last CTA to count itself
  // out clears the bank for the next call of this generation's parity.
  __syncwarp();
  if (lane == 0 && atomicAdd(&sm.exited[0], 1u) == (unsigned)(kWarps - 1)) {
    if (*abort_flag) ring.drain();
    if constexpr (kGrouped) {
      GroupedBanks* bk = reinterpret_cast<GroupedBanks*>(reinterpret_cast<uint8_t*>(ws) + kGroupedBanksOffset);
      const unsigned par = *sm.gen & 1u;
      if (atom_add_acq_rel_gpu(&bk->readers[par], 1u) == (unsigned)(G - 1)) {
        for (int q = 0; q < src.members(); ++q) bk->maxbits[par][q] = 0u;
        bk->readers[par] = 0u;
      }
    }
  }
}

template <typename T, int MODE, bool kBulk>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_kernel(const __grid_constant__ CUtensorMap tmap, const CastArgs a, SinglePassWorkspace* ws) {
  fused_body<T, MODE, kBulk>(tmap, PlainSrc{a}, ws);
}

template <int MODE, bool kBulk>
__global__ void __launch_bounds__(kFusedThreads, 1)
    grouped_fused_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ GroupedArgs ga,
                         SinglePassWorkspace* ws) {
  extern __shared__ uint8_t smem_raw[];
  const FSmem sm = fcarve<uint16_t, true>(smem_raw);
  const int tid = threadIdx.x;
  if (tid < ga.num_groups) {
    MemberInfo& i = sm.minfo[tid];
    i.data_row = ga.data_row[tid];
    i.scale_row = ga.scale_row[tid];
    i.data_col = ga.data_col[tid];
    i.scale_col = ga.scale_col[tid];
    i.row0 = ga.row0[tid];
    i.rows = ga.rows[tid];
  }
  if (tid <= ga.num_groups) sm.mstart[tid] = ga.tile_start[tid];
  __syncthreads();
  GroupedSrc src;
  src.tl = GroupedSrc::Tiles{sm.minfo, sm.mstart, ga.num_groups, ga.tiles_n};
  src.ntiles = ga.num_tiles;
  src.N = ga.N;
  src.noop_ = ga.noop;
  src.status_ = ga.status;
  src.rowwise_ = ga.rowwise;
  src.colwise_ = ga.colwise;
  src.swizzled_ = ga.swizzled;
  src.ga = &ga;
  fused_body<uint16_t, MODE, kBulk>(tmap, src, ws);
}

template <typename T, int MODE, bool kBulk>
cudaError_t launch_fused_t(const CUtensorMap& map, const CastArgs& a, SinglePassWorkspace* ws, const LaunchCtx& ctx) {
  return sp::launch_persistent<fused_kernel<T, MODE, kBulk>>(fused_smem_bytes<T>(), kFusedThreads, map, a,
                                                             a.num_tiles, ws, ctx);
}

template <int MODE, bool kBulk>
cudaError_t launch_grouped_fused_t(const CUtensorMap& map, const GroupedArgs& ga, SinglePassWorkspace* ws,
                                   const LaunchCtx& ctx) {
  return sp::launch_persistent<grouped_fused_kernel<MODE, kBulk>>(fused_smem_bytes<uint16_t, true>(), kFusedThreads,
                                                                  map, ga, ga.num_tiles, ws, ctx);
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

cudaError_t launch_grouped_single_pass(const CUtensorMap& map, int mode, GroupedArgs ga, SinglePassWorkspace* ws,
                                       const LaunchCtx& ctx) {
  grouped_prefix_sums(ga, /*bf16=*/true);
  if (ga.num_tiles == 0) return launch_grouped_zero(ga, ctx);  // every member empty: amax 0
  // the 128x4 layout requires every member's rows and N multiples of 128
  // (validated): every tile is whole
  if (ga.swizzled) {
    if (mode == kCast1D) return launch_grouped_fused_t<kCast1D, true>(map, ga, ws, ctx);
    return launch_grouped_fused_t<kCast2D, true>(map, ga, ws, ctx);
  }
  if (mode == kCast1D) return launch_grouped_fused_t<kCast1D, false>(map, ga, ws, ctx);
  return launch_grouped_fused_t<kCast2D, false>(map, ga, ws, ctx);
}

}  // namespace nvfp4
