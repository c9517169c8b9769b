/*
 * nvfp4.h -- C ABI of libnvfp4: NVFP4 quantize-with-transpose on one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * NVFP4: FP4 E2M1 codes (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; bit 3 is the
 * sign; element 2i in the low nibble of byte i), one E4M3 decode scale per
 * 16-element block, and one FP32 amax per tensor (or per row) from which the
 * FP32 global encode scale g = 448 * 6 / amax is formed:
 *     s = E4M3_rn_satfinite((block_amax / 6) * g)        per block
 *     r = g / float(s)   (r = 0 when s = 0; clamped to FLT_MAX)
 *     q = E2M1_rn_satfinite(x * r)                       per element
 * with amax = 0 giving g = 1 and an overflowing g clamped to FLT_MAX.
 *
 * Layouts (x is M x N, row-major, M rows, N the contiguous dimension):
 *   row-wise data    [M][N/2] bytes     1x16 blocks along a row of x
 *   row-wise scales  [M][N/16] bytes    compact, or swizzled (below)
 *   column-wise data [N][M/2] bytes     the quantization of x transposed:
 *                                       row j holds column j of x
 *   column-wise scales [N][M/16] bytes  compact, or swizzled
 *   Swizzled scales: the cuBLAS 1D block-scaling-factor layout for an R x C
 *   scale matrix (R % 128 == 0, C % 4 == 0): byte offset of (r, c) =
 *   ((r/128)*(C/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4.  It is
 *   only accepted when both data dimensions are multiples of 128
 *   ("Fuse NVFP4 scale swizzling on SM120 and SM121", Description).
 *
 * Conventions for every entry point:
 *   * Pointers named x / data / scale / amax / out / noop are DEVICE pointers
 *     owned by the caller; the library never allocates, frees or keeps them.
 *     Device pointers must be 16-byte aligned (NVFP4_ERR_ALIGN otherwise).
 *   * stream is a cudaStream_t (NULL = the legacy default stream).  All work
 *     is enqueued on it asynchronously; no call synchronizes the device.
 *   * Arguments are validated, and the tensor map through which the kernels
 *     read x is encoded, on the host before anything is enqueued: every
 *     status but NVFP4_ERR_CUDA means nothing was launched and no output was
 *     written.  NVFP4_ERR_CUDA means a CUDA call failed (cudaGetLastError()
 *     reads the error): if it was the launch of a call's second kernel, the
 *     first one (the amax reduction ahead of a cast) was enqueued and may
 *     still write the amax buffers.
 *   * Quantize shapes: N % 16 == 0 always (row-wise blocks span 16 columns,
 *     and x is staged through a tensor map whose row pitch must be a multiple
 *     of 16 bytes); with COLWISE, or for 2D / RHT, also M % 16 == 0; row-wise
 *     output alone takes any M >= 0.
 *   * noop: NULL, or a device float; when it holds 1.0f at execution time the
 *     call writes nothing at all, amax buffers included ("Write both NVFP4
 *     amax buffers", Changes: with a noop flag set both buffers are left
 *     untouched).
 *   * Kernels bound every wait they perform.  If a wait ever runs out, the
 *     kernel records it in a per-device status word (read it with
 *     nvfp4_device_status) and returns without finishing its outputs.
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_NULL = 1,    /* a required pointer is NULL                        */
  NVFP4_ERR_SHAPE = 2,   /* negative size, or a dimension not % 16 (above)     */
  NVFP4_ERR_ALIGN = 3,   /* SWIZZLED on a shape not 128-aligned; bad pointer   */
  NVFP4_ERR_DTYPE = 4,   /* unknown dtype, or one the operation does not take  */
  NVFP4_ERR_FLAGS = 5,   /* unknown / contradictory flags; aliased amax buffers */
  NVFP4_ERR_CUDA = 6,    /* a CUDA call failed (see the conventions above)     */
  NVFP4_ERR_TIMEOUT = 7  /* a device-side wait ran out (nvfp4_device_status)   */
} nvfp4_status;

/* flags */
#define NVFP4_ROWWISE 1u     /* produce the row-wise output                   */
#define NVFP4_COLWISE 2u     /* produce the column-wise (transposed) output   */
#define NVFP4_SWIZZLED 4u    /* scales in the cuBLAS 128x4 layout             */
#define NVFP4_SKIP_AMAX 8u   /* use the amax already in the buffers           */
#define NVFP4_ROW_SCALED 16u /* dequantize: one amax per row                  */

/* dtypes */
#define NVFP4_BF16 0
#define NVFP4_FP32 1

typedef struct {
  uint8_t* data_row;  /* [M][N/2]                       (ROWWISE)            */
  uint8_t* scale_row; /* [M][N/16]                      (ROWWISE)            */
  float* amax_row;    /* 1 float (row-scaled: M floats) (ROWWISE)            */
  uint8_t* data_col;  /* [N][M/2]                       (COLWISE)            */
  uint8_t* scale_col; /* [N][M/16]                      (COLWISE)            */
  float* amax_col;    /* 1 float                        (COLWISE)            */
} nvfp4_output;

/* Human-readable name of a status. */
const char* nvfp4_status_string(nvfp4_status status);

/* Bytes of a scale tensor for a rows x cols data matrix (rows * cols / 16,
 * compact or swizzled alike; swizzled needs rows % 128 == 0 and cols % 128 ==
 * 0, else NVFP4_ERR_ALIGN).  Host-only, no device work. */
nvfp4_status nvfp4_scale_bytes(int64_t rows, int64_t cols, unsigned flags, size_t* bytes);

/*
 * Per-tensor amax ("Write both NVFP4 amax buffers", Description and Changes):
 * zeroes amax_row and, when non-NULL, amax_col, then reduces max|x| over the
 * M x N elements of x into both; no device-to-device copy, no extra read.
 * amax_row must not equal amax_col (distinct buffers: the same page's review
 * reply on aliasing).  M or N may be 0 (amax = 0).  dtype: BF16 or FP32.
 */
nvfp4_status nvfp4_compute_amax(const void* x, int dtype, int64_t M, int64_t N,
                                float* amax_row, float* amax_col, const float* noop,
                                void* stream);

/*
 * Per-tensor amax pair for the random-Hadamard column-wise path ("Write both
 * NVFP4 amax buffers", review reply on aliasing: row-wise amax = max|x|,
 * column-wise amax = max|RHT(x)|).  RHT(x): every 16-element column block v
 * (rows 16k..16k+15 of one column) becomes (1/4) H16 diag(sign) v, H16 the
 * Sylvester Hadamard matrix in natural order, sign_i = -1 where bit i of
 * sign_mask is set, rounded to BF16 (BF16 input only).  M % 16 == 0.
 */
nvfp4_status nvfp4_compute_amax_rht(const void* x, int dtype, int64_t M, int64_t N,
                                    uint32_t sign_mask, float* amax_row, float* amax_col,
                                    const float* noop, void* stream);

/*
 * 1D NVFP4 quantize with row-wise and/or column-wise outputs in one pass
 * over x, after the per-tensor amax (written to both buffers); scales compact
 * or swizzled ("Write both NVFP4 amax buffers"; "Fuse NVFP4 scale swizzling
 * on SM120 and SM121", Changes: the generic and tuned 1D kernels gain a
 * swizzled store).  flags: ROWWISE | COLWISE (at least one) | SWIZZLED |
 * SKIP_AMAX.  N % 16 == 0; COLWISE also needs M % 16 == 0.
 * Both amax buffers receive max|x|; with SKIP_AMAX the kernel reads them
 * instead (e.g. after a cross-rank MAX) and writes none.
 */
nvfp4_status nvfp4_quantize_1d(const void* x, int dtype, int64_t M, int64_t N,
                               const nvfp4_output* out, unsigned flags, const float* noop,
                               void* stream);

/*
 * 2D NVFP4 quantize: one E4M3 scale per 16x16 tile of x ("Fuse NVFP4 scale
 * swizzling on SM120 and SM121", Description: the 2D in-kernel path).  The
 * scale tensors keep the 1x16 shapes above with each tile's scale repeated
 * over its 16 rows (row-wise) or 16 columns (column-wise), so the
 * column-wise codes are exactly the transpose of the row-wise codes.
 * M % 16 == 0 and N % 16 == 0.  Flags as nvfp4_quantize_1d.
 */
nvfp4_status nvfp4_quantize_2d(const void* x, int dtype, int64_t M, int64_t N,
                               const nvfp4_output* out, unsigned flags, const float* noop,
                               void* stream);

/*
 * Row-scaled (per-token) NVFP4 ("Implement row-scaled NVFP4 fprop recipe",
 * Greptile summary: one FP32 amax per row; block scales recomputed relative
 * to that row's value).  Row-wise only: flags = ROWWISE [| SWIZZLED]
 * [| SKIP_AMAX]; out->amax_row has M floats and receives max|x[y,:]| (or is
 * read, with SKIP_AMAX).  A zero row encodes to zero codes and scales.
 * N % 16 == 0; any M >= 0.
 */
nvfp4_status nvfp4_quantize_row_scaled(const void* x, int dtype, int64_t M, int64_t N,
                                       const nvfp4_output* out, unsigned flags,
                                       const float* noop, void* stream);

/*
 * 1D / 2D quantize with stochastically rounded codes ("Fuse NVFP4 scale
 * swizzling on SM120 and SM121", Tests: stochastic rounding is one axis of
 * the comparisons).  Amax, block scales, layouts and flags as
 * nvfp4_quantize_1d / _2d; each product p = x * g / float(s) is rounded to
 * one of its two neighbouring E2M1 magnitudes lo <= |p| < hi: to hi iff
 * rbits[y * N + j] < 256 (|p| - lo) / (hi - lo) for element (y, j) of x, in
 * the row-wise and in the column-wise output alike (|p| >= 6 saturates; the
 * sign of x is kept).  With uniform random bytes P(hi) = ceil(256 f) / 256.
 *   rbits: M x N bytes of device memory, row-major like x, 16-byte aligned,
 *   owned by the caller (the random numbers are an input; the library draws
 *   none).  N % 16 == 0; 2D also M % 16 == 0.
 */
nvfp4_status nvfp4_quantize_1d_sr(const void* x, int dtype, int64_t M, int64_t N,
                                  const nvfp4_output* out, unsigned flags, const uint8_t* rbits,
                                  const float* noop, void* stream);
nvfp4_status nvfp4_quantize_2d_sr(const void* x, int dtype, int64_t M, int64_t N,
                                  const nvfp4_output* out, unsigned flags, const uint8_t* rbits,
                                  const float* noop, void* stream);

/*
 * Grouped (multi-tensor) 1D / 2D quantize: x (row-major, N columns) stacks
 * num_groups member tensors along its first dimension, member g being the
 * group_rows[g] rows that follow the earlier members' rows.  Every member is
 * quantized as a tensor of its own into outs[g] (the buffers and layouts of
 * nvfp4_quantize_1d / _2d for a group_rows[g] x N tensor): its own amax, so
 * its own global scale ("Implement row-scaled NVFP4 fprop recipe", Important
 * Files Changed: a grouped tensor keeps one amax slice per member), and its
 * column-wise output is the transpose of its own rows.  Three launches
 * whatever num_groups (zero the amaxes, max|x| per member, one cast over all
 * members' tiles).
 *   group_rows, outs: HOST arrays of num_groups entries, read before the call
 *   returns (the device buffers they name stay the caller's).
 *   1 <= num_groups <= NVFP4_MAX_GROUPS; group_rows[g] >= 0 (0: an empty
 *   member, amax 0); N % 16 == 0; with COLWISE, or for 2D, group_rows[g] %
 *   16 == 0; with SWIZZLED, group_rows[g] % 128 == 0 and N % 128 == 0.
 *   Every member's outputs are checked as nvfp4_quantize_1d checks them, and
 *   no two amax buffers of the call may be the same (NVFP4_ERR_FLAGS).
 *   flags: ROWWISE | COLWISE | SWIZZLED | SKIP_AMAX, for every member.
 *   Validation fails before anything is enqueued.
 */
#define NVFP4_MAX_GROUPS 64
nvfp4_status nvfp4_quantize_grouped_1d(const void* x, int dtype, int64_t N, int num_groups,
                                       const int64_t* group_rows, const nvfp4_output* outs,
                                       unsigned flags, const float* noop, void* stream);
nvfp4_status nvfp4_quantize_grouped_2d(const void* x, int dtype, int64_t N, int num_groups,
                                       const int64_t* group_rows, const nvfp4_output* outs,
                                       unsigned flags, const float* noop, void* stream);
/*
 * Single-launch grouped 1D / 2D quantize: the results of
 * nvfp4_quantize_grouped_1d / _2d (every member's amax in both of its
 * buffers, its codes and scales) from one persistent kernel that reads x
 * from HBM once: the tiles of all members stream through shared memory while
 * each CTA keeps a maximum per member, a grid-wide barrier combines the
 * members' maxima in the workspace, then every member's tiles are cast with
 * that member's global scale.  (The same pages as the grouped quantize; the
 * single launch is nvfp4_quantize_1d_single_pass's design applied to every
 * member at once.)
 *   Arguments and checks as nvfp4_quantize_grouped_1d; x BF16 (FP32:
 *   NVFP4_ERR_DTYPE); flags ROWWISE | COLWISE | SWIZZLED (no SKIP_AMAX).
 *   workspace: as for nvfp4_quantize_1d_single_pass (4096 bytes, zeroed
 *   before first use, not shared by calls that can run at the same time);
 *   besides the 64-byte barrier header this call uses bytes 64..583 (two
 *   banks of per-member maxima, each cleared by the call that used it, so
 *   single-pass calls of either kind may share one workspace).  After a call
 *   that reported NVFP4_ERR_TIMEOUT, zero it again.
 */
nvfp4_status nvfp4_quantize_grouped_1d_single_pass(const void* x, int dtype, int64_t N, int num_groups,
                                                   const int64_t* group_rows, const nvfp4_output* outs,
                                                   unsigned flags, const float* noop, void* workspace,
                                                   void* stream);
nvfp4_status nvfp4_quantize_grouped_2d_single_pass(const void* x, int dtype, int64_t N, int num_groups,
                                                   const int64_t* group_rows, const nvfp4_output* outs,
                                                   unsigned flags, const float* noop, void* workspace,
                                                   void* stream);

/*
 * NVFP4 quantize with the random Hadamard transform on the column-wise path
 * ("Write both NVFP4 amax buffers", GPU work per quantize call: the RHT path
 * runs a zeroing kernel, a Hadamard-amax kernel and the quantize kernel;
 * "Fuse NVFP4 scale swizzling on SM120 and SM121", Changes: the
 * columnwise-RHT 1D kernel).  The row-wise output is the plain 1D
 * quantization of x with amax_row = max|x|; the column-wise output is the 1D
 * quantization of RHT(x) transposed (transform as nvfp4_compute_amax_rht)
 * with amax_col = max|RHT(x)|.  BF16 input; M % 16 == 0, N % 16 == 0.
 */
nvfp4_status nvfp4_quantize_rht(const void* x, int dtype, int64_t M, int64_t N,
                                const nvfp4_output* out, unsigned flags, uint32_t sign_mask,
                                const float* noop, void* stream);

/*
 * Single-launch 1D / 2D quantize: the same results as nvfp4_quantize_1d /
 * nvfp4_quantize_2d (amax written to both buffers, codes, scales), computed
 * by one persistent kernel that reads x from HBM once: it reduces max|x|
 * while staging tiles in shared memory, meets the other CTAs at a grid-wide
 * barrier, then casts the staged tiles and re-reads the rest from L2.
 * ("Write both NVFP4 amax buffers", Description: the reduction writes both
 * buffers; "Fuse NVFP4 scale swizzling on SM120 and SM121": scales written
 * directly in the GEMM layout.)
 *   workspace: NVFP4_SINGLE_PASS_WORKSPACE_BYTES of device memory, zeroed
 *   before its first use and not shared by calls that can run at the same
 *   time; the kernel leaves it ready for the next call (it uses the first 64
 *   bytes: the grid barrier's generation and, for two alternating
 *   generations, an arrival count and two maxima; the grouped single-pass
 *   quantize also uses bytes 64..583; the rest is reserved).
 *   After a call that reported NVFP4_ERR_TIMEOUT through
 *   nvfp4_device_status, zero it again.
 *   flags: ROWWISE | COLWISE | SWIZZLED (no SKIP_AMAX: use the two-pass
 *   entry points for a given amax).  All CTAs must be co-resident (one per
 *   SM); a device where that is impossible returns NVFP4_ERR_CUDA.
 */
#define NVFP4_SINGLE_PASS_WORKSPACE_BYTES 4096
nvfp4_status nvfp4_quantize_1d_single_pass(const void* x, int dtype, int64_t M, int64_t N,
                                           const nvfp4_output* out, unsigned flags, const float* noop,
                                           void* workspace, void* stream);
nvfp4_status nvfp4_quantize_2d_single_pass(const void* x, int dtype, int64_t M, int64_t N,
                                           const nvfp4_output* out, unsigned flags, const float* noop,
                                           void* workspace, void* stream);
/*
 * Single-launch Hadamard quantize: the results of nvfp4_quantize_rht (within
 * the same rounding-tie tolerance of the column-wise codes; amax_row =
 * max|x| and amax_col = max|RHT(x)| exact) from one persistent kernel that
 * reads x from HBM once: per tile it reduces max|x| and, on the tensor cores,
 * transforms the tile's 16-row column blocks for max|RHT(x)|; after the grid
 * barrier it casts the rows of x and transforms the staged or re-read tiles
 * again for the column-wise cast.  ("Write both NVFP4 amax buffers", review
 * reply: with RHT the row amax is max|x|, the column amax max|RHT(x)|.)
 * Workspace, flags and co-residency as above; BF16 input, M % 16 == 0,
 * N % 16 == 0 (NVFP4_ERR_DTYPE / NVFP4_ERR_SHAPE).  Without COLWISE the
 * transform plays no part and the call is nvfp4_quantize_1d_single_pass.
 */
nvfp4_status nvfp4_quantize_rht_single_pass(const void* x, int dtype, int64_t M, int64_t N,
                                            const nvfp4_output* out, unsigned flags, uint32_t sign_mask,
                                            const float* noop, void* workspace, void* stream);

/*
 * nvfp4_quantize_2d_single_pass for callers that cannot allocate device
 * memory.  This entry point has no counterpart on the pages this library
 * follows.  It computes exactly what nvfp4_quantize_2d_single_pass computes,
 * but takes no workspace: its scratch is a 256-byte array inside the
 * library that the CUDA runtime places on every GPU that loads it (held
 * until the process exits).  It serves callers with no device allocator of
 * their own (a plain C host embedding the library), callers on paths that
 * must not take an allocator's lock or risk a synchronizing cudaMalloc or
 * cudaFree, and processes that size all device memory up front.
 *   * The first call on a device looks up the array's device address (a
 *     runtime query, no allocation); make that first call before any stream
 *     capture on that device.  The address is kept for the life of the
 *     process: it belongs to the device's primary context, so after
 *     cudaDeviceReset() on a device this entry point must not be called on
 *     that device again (the kept address would be stale).
 *   * Every call clears the array's 64-byte barrier header on `stream` (a
 *     memset) and then launches the kernel; it calls no cudaMalloc /
 *     cudaFree.
 *   * All calls on a device share the one array: calls that can overlap on
 *     the GPU (other streams, other threads) race and give wrong results;
 *     serialize them.
 *   * Limit: the kernel needs the 64-byte header only, for any grid (one
 *     CTA per SM), so the array's size bounds no input shape.
 * Arguments, flags and errors otherwise as nvfp4_quantize_2d_single_pass.
 */
nvfp4_status nvfp4_quantize_2d_single_pass_noalloc(const void* x, int dtype, int64_t M, int64_t N,
                                                   const nvfp4_output* out, unsigned flags,
                                                   const float* noop, void* stream);

/*
 * Dequantize one direction of an NVFP4 tensor ("Implement row-scaled NVFP4
 * fprop recipe", Important Files Changed, dequantize_nvfp4.cuh: row y uses
 * tensor_amax[y] when row-scaled, else tensor_amax[0]):
 *     out[y][j] = (E2M1(q[y][j]) * float(s[y][j/16])) * (a / 2688)
 * in FP32, rounded to BF16 (out_dtype NVFP4_BF16) or kept (NVFP4_FP32).
 * data [rows][cols/2], scale [rows][cols/16] (compact, or swizzled with
 * NVFP4_SWIZZLED), amax 1 float (or rows floats with NVFP4_ROW_SCALED).
 * cols % 16 == 0.  For a column-wise output pass rows = N, cols = M.
 */
nvfp4_status nvfp4_dequantize(const uint8_t* data, const uint8_t* scale, const float* amax,
                              int64_t rows, int64_t cols, unsigned flags, void* out,
                              int out_dtype, void* stream);

/*
 * Compact -> swizzled scale permutation ("Write both NVFP4 amax buffers",
 * GPU work per quantize call: the post-quantize swizzle_row_scaling_kernel
 * that unaligned shapes still need).  compact [rows][scale_cols];
 * rows % 128 == 0, scale_cols % 4 == 0; compact and swizzled must not
 * overlap.
 */
nvfp4_status nvfp4_swizzle_scales(const uint8_t* compact, uint8_t* swizzled, int64_t rows,
                                  int64_t scale_cols, void* stream);

/*
 * Per-device status word of bounded device-side waits: bit 0 = a wait for a
 * tile copy ran out; bit 1 = a grid-wide barrier of a single-pass call ran
 * out.  Synchronizes the current device, copies the word into
 * *status and, when clear != 0, resets it.  Returns NVFP4_ERR_TIMEOUT when a
 * bit was set, NVFP4_OK otherwise, NVFP4_ERR_CUDA if the copy failed.
 */
nvfp4_status nvfp4_device_status(uint32_t* status, int clear);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_H_ */
