// kernels.h -- internal launchers of the NVFP4 kernels (host side).
//
// Every launcher enqueues on ctx.stream and returns the launch status; the
// arguments have been validated by the C-ABI layer (nvfp4_api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

// Launches `func` so that it may start while the preceding kernel on the
// stream is still running (programmatic dependent launch); the kernel's
// griddepcontrol.wait orders it after that kernel's memory operations.
inline cudaError_t launch_pdl(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, func, args);
}

struct LaunchCtx {
  cudaStream_t stream;
  int num_sms;
  unsigned* status;  // per-device status word (device address)
};

// Zero both amax buffers, then max|x| into both (the reduction may start
// before the zeroing kernel ends; its atomics wait for it).
cudaError_t launch_amax(const void* x, bool bf16, int64_t n, float* amax_a, float* amax_b,
                        const float* noop, const LaunchCtx& ctx);

// Zero both buffers, then max|x| into amax_row and max|RHT(x)| (BF16-rounded)
// into amax_col.  x is BF16, M % 16 == 0, N % 16 == 0.
cudaError_t launch_rht_amax(const uint16_t* x, int64_t M, int64_t N, uint32_t sign_mask, float* amax_row,
                            float* amax_col, const float* noop, const LaunchCtx& ctx);

enum CastMode : int { kCast1D = 0, kCast2D = 1, kCastRHT = 2 };

struct CastArgs {
  int64_t M, N;
  uint8_t* data_row;
  uint8_t* scale_row;
  const float* amax_row;
  uint8_t* data_col;
  uint8_t* scale_col;
  const float* amax_col;
  const float* noop;
  unsigned* status;
  int rowwise, colwise, swizzled;
  uint32_t sign_mask;
  int tiles_n, num_tiles;
};

// Tensor map of x (M x N row-major, BF16 or FP32): dims {N, M}, box {128
// bytes, 128 rows}, 128-byte swizzle, zero fill outside the tensor.  The
// C-ABI layer encodes it before it enqueues anything for a call, so that a
// call whose map cannot be encoded launches nothing.  Needs a 16-byte
// aligned x and N * element size a multiple of 16 bytes (N % 16 == 0 is
// validated first).
cudaError_t make_x_tensor_map(CUtensorMap* map, const void* x, bool bf16, int64_t M, int64_t N);
// Tensor map of an M x N byte matrix (row pitch N): box 128 x 128 bytes,
// 128-byte swizzle, zero fill outside.  Needs a 16-byte aligned base and
// N % 16 == 0.
cudaError_t make_byte_tensor_map(CUtensorMap* map, const void* p, int64_t M, int64_t N);

// Fused row-wise + column-wise cast of x (TMA tiles of 128 x 128 elements,
// `map` from make_x_tensor_map) reading the per-tensor amax from
// args.amax_row / args.amax_col.  `pdl`: launched as a programmatic
// dependent of the preceding amax kernel.
cudaError_t launch_cast(const CUtensorMap& map, bool bf16, int mode, CastArgs args, bool pdl, const LaunchCtx& ctx);

// Scratch of the single-pass kernels (a 64-byte header, zeroed before first
// use, then kept consistent by the kernels themselves): the grid barrier's
// generation, and for each of the two alternating generations the warps'
// arrival count and the maximum they published (FP32 bits; non-negative
// floats order like their bit patterns).
struct SinglePassWorkspace {
  unsigned gen;
  unsigned pad0;
  unsigned arrive[2];
  unsigned maxbits[2];
  unsigned maxbits2[2];  // a second maximum (the Hadamard quantize: max|RHT(x)|)
  unsigned pad[8];
};
constexpr size_t kSinglePassHeaderBytes = 64;
static_assert(sizeof(SinglePassWorkspace) == kSinglePassHeaderBytes, "workspace header layout");

// One persistent launch: per-tensor amax of x (written to args.amax_row /
// args.amax_col) and the fused cast (1D or 2D), x read from HBM once.
cudaError_t launch_single_pass(const CUtensorMap& map, bool bf16, int mode, CastArgs args, SinglePassWorkspace* ws,
                               const LaunchCtx& ctx);
// The same for the Hadamard quantize (BF16): max|x| into args.amax_row,
// max|RHT(x)| into args.amax_col, then the row-wise cast of x and the
// column-wise cast of the transformed columns.
cudaError_t launch_single_pass_rht(const CUtensorMap& map, CastArgs args, SinglePassWorkspace* ws,
                                   const LaunchCtx& ctx);
// CTAs the single-pass kernel uses for an M x N input.
int single_pass_grid(int64_t M, int64_t N, const LaunchCtx& ctx);

// Row-scaled cast: per-row amax (unless skip_amax), row-wise codes/scales.
cudaError_t launch_row_scaled(const void* x, bool bf16, int64_t M, int64_t N, uint8_t* data, uint8_t* scale,
                              float* amax, bool skip_amax, bool swizzled, const float* noop,
                              const LaunchCtx& ctx);

cudaError_t launch_dequantize(const uint8_t* data, const uint8_t* scale, const float* amax, int64_t rows,
                              int64_t cols, bool swizzled, bool row_scaled, void* out, bool out_bf16,
                              const LaunchCtx& ctx);

cudaError_t launch_swizzle(const uint8_t* compact, uint8_t* swizzled, int64_t rows, int64_t scale_cols,
                           const LaunchCtx& ctx);

}  // namespace nvfp4
