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

// Zeroes the members' amax buffers and reduces max|x| per member into them
// (skipped with skip_amax), then casts every member (mode kCast1D or
// kCast2D): three launches whatever the number of members.  `ga` has every
// field filled but tiles_n, num_tiles, num_chunks and the prefix sums;
// `map` is the tensor map of x (all members' rows, make_x_tensor_map), or
// null when x has no element.
cudaError_t launch_grouped(const void* x, const CUtensorMap* map, bool bf16, int mode, GroupedArgs ga,
                           bool skip_amax, const LaunchCtx& ctx);

}  // namespace nvfp4
