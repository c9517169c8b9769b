// sr.h -- NVFP4 quantize with stochastically rounded codes (sr.cu).
#pragma once

#include "kernels.h"

namespace nvfp4 {

// The fused row-wise + column-wise cast (mode kCast1D or kCast2D) with the
// E2M1 codes rounded stochastically: element (y, j) of x rounds with the
// random byte rbits[y * N + j] in both outputs; block scales as the plain
// cast.  `rmap`: make_byte_tensor_map of rbits (M x N bytes), whose tiles
// are staged beside x's.  Reads the per-tensor amax from args.amax_row /
// args.amax_col; `pdl`: launched as a programmatic dependent of the
// preceding amax kernel.  N % 16 == 0.
cudaError_t launch_cast_sr(const CUtensorMap& map, bool bf16, int mode, CastArgs args, const CUtensorMap& rmap,
                           bool pdl, const LaunchCtx& ctx);

}  // namespace nvfp4
