// grouped.h -- grouped (multi-tensor) quantize: the member table the three
// kernels of grouped.cu share, passed by value as a kernel parameter (no
// device-side table: a call allocates nothing and its launches carry all of
// its state).
#pragma once

#include "kernels.h"

namespace nvfp4 {

constexpr int kMaxGroups = 64;

// x (BF16 or FP32, row-major, N columns) stacks the members along its first
// dimension: member g is rows [row0[g], row0[g] + rows[g]).  Its outputs are
// its own buffers (the layouts of the plain quantize for a rows[g] x N
// tensor).  tile_start / chunk_start: prefix sums of the members' 128x128
// tiles and amax chunks (the last entry is the total).
struct GroupedArgs {
  int num_groups;
  int tiles_n;      // tiles across N
  int num_tiles;    // all members
  int num_chunks;   // all members
  int64_t N;
  const float* noop;
  unsigned* status;
  int rowwise, colwise, swizzled, pad;
  int tile_start[kMaxGroups + 1];
  int chunk_start[kMaxGroups + 1];
  int64_t row0[kMaxGroups];
  int64_t rows[kMaxGroups];
  uint8_t* data_row[kMaxGroups];
  uint8_t* scale_row[kMaxGroups];
  float* amax_row[kMaxGroups];
  uint8_t* data_col[kMaxGroups];
  uint8_t* scale_col[kMaxGroups];
  float* amax_col[kMaxGroups];
};

// Vectors (16 bytes) of x per amax chunk: 256 threads x 8 loads.
constexpr int64_t kGroupChunkVecs = 2048;

// Largest g with start[g] <= i (start[0] = 0 <= i < start[n]).
__device__ __forceinline__ int member_of(const int* start, int n, int i) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (start[mid] <= i)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Tile t of all members (tile_start filled): its member g, and its first
// row r0 and column c0 in that member (128x128 tiles, row-major within the
// member; the member's rows start at row ga.row0[g] of x).
struct MemberTile {
  int g;
  int64_t r0, c0;
};
__device__ __forceinline__ MemberTile member_tile(const GroupedArgs& ga, int t) {
  MemberTile p;
  p.g = member_of(ga.tile_start, ga.num_groups, t);
  const int lt = t - ga.tile_start[p.g];
  const int tr = lt / ga.tiles_n;
  p.r0 = (int64_t)tr * 128;
  p.c0 = (int64_t)(lt - tr * ga.tiles_n) * 128;
  return p;
}

// The single-pass grouped quantize's per-member maxima, in the caller's
// workspace right after the grid barrier's header: two banks (used by
// calls of even and odd generation), each kMaxGroups maxima (FP32 bits) and
// a count of the CTAs that have read the bank; the last CTA to read clears
// the bank and its count, so that it is zero for the next call of its
// parity whatever single-pass calls come between.
struct GroupedBanks {
  unsigned maxbits[2][kMaxGroups];
  unsigned readers[2];
};
constexpr size_t kGroupedBanksOffset = kSinglePassHeaderBytes;
static_assert(kGroupedBanksOffset + sizeof(GroupedBanks) <= 4096, "within the single-pass workspace");

// Zeroes the members' amax buffers and reduces max|x| per member into them
// (skipped with skip_amax), then casts every member (mode kCast1D or
// kCast2D): three launches whatever the number of members.  `ga` has every
// field filled but tiles_n, num_tiles, num_chunks and the prefix sums;
// `map` is the tensor map of x (all members' rows, make_x_tensor_map), or
// null when x has no element.
cudaError_t launch_grouped(const void* x, const CUtensorMap* map, bool bf16, int mode, GroupedArgs ga,
                           bool skip_amax, const LaunchCtx& ctx);

// The same in one persistent launch (BF16 x; fused.cu): per-member max|x|
// while the tiles stream through shared memory, a grid barrier that combines
// the members' maxima in the workspace (see GroupedBanks), then the cast of
// every member's tiles with its own global scale.  `ga` as for
// launch_grouped; `ws` the single-pass workspace (4096 bytes).  With no
// tile at all it only zeroes the members' amaxes.
cudaError_t launch_grouped_single_pass(const CUtensorMap& map, int mode, GroupedArgs ga, SinglePassWorkspace* ws,
                                       const LaunchCtx& ctx);
// Zeroes the members' amax buffers (unless *ga.noop == 1).
cudaError_t launch_grouped_zero(const GroupedArgs& ga, const LaunchCtx& ctx);
// Fills ga's tile and chunk prefix sums (tiles_n, tile_start, num_tiles,
// chunk_start, num_chunks) from rows[] and N.
void grouped_prefix_sums(GroupedArgs& ga, bool bf16);

}  // namespace nvfp4
