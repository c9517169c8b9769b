// nvfp4_api.cu -- the C ABI declared in include/nvfp4.h: host-side argument
// validation (before anything is enqueued), TMA descriptor creation and the
// launch sequence of each operation.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "grouped.h"
#include "kernels.h"
#include "nvfp4.h"
#include "sr.h"

// Per-device status word of bounded device-side waits.
__device__ unsigned int g_nvfp4_status_word;

namespace nvfp4 {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int num_sms = 0;
  unsigned* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (d.status == nullptr) {
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_nvfp4_status_word);
    if (e != cudaSuccess) return e;
    d.num_sms = sms;
    d.status = static_cast<unsigned*>(p);
  }
  *out = d;
  return cudaSuccess;
}

nvfp4_status make_ctx(void* stream, LaunchCtx* ctx) {
  DeviceInfo d;
  if (device_info(&d) != cudaSuccess) return NVFP4_ERR_CUDA;
  ctx->stream = static_cast<cudaStream_t>(stream);
  ctx->num_sms = d.num_sms;
  ctx->status = d.status;
  return NVFP4_OK;
}

nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxDim = (int64_t)1 << 31;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// Checks common to the quantize entry points.  N % 16 == 0 whatever the
// directions: row-wise blocks span 16 columns, and every cast stages x by
// TMA, whose row pitch must be a multiple of 16 bytes; column-wise blocks
// span 16 rows (M % 16 == 0).  Row-wise alone takes any M.
nvfp4_status check_quantize(const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                            unsigned flags, unsigned allowed_flags) {
  if (out == nullptr) return NVFP4_ERR_NULL;
  if (flags & ~allowed_flags) return NVFP4_ERR_FLAGS;
  if (!(flags & (NVFP4_ROWWISE | NVFP4_COLWISE))) return NVFP4_ERR_FLAGS;
  if (dtype != NVFP4_BF16 && dtype != NVFP4_FP32) return NVFP4_ERR_DTYPE;
  if (M < 0 || N < 0 || M >= kMaxDim || N >= kMaxDim) return NVFP4_ERR_SHAPE;
  if (N % 16 != 0) return NVFP4_ERR_SHAPE;
  if (M > 0 && N > 0 && x == nullptr) return NVFP4_ERR_NULL;
  if (x != nullptr && !aligned16(x)) return NVFP4_ERR_ALIGN;
  const bool row = flags & NVFP4_ROWWISE, col = flags & NVFP4_COLWISE;
  if (row) {
    if (out->amax_row == nullptr) return NVFP4_ERR_NULL;
    if (M > 0 && N > 0 && (out->data_row == nullptr || out->scale_row == nullptr)) return NVFP4_ERR_NULL;
    if (!aligned16(out->data_row) || !aligned16(out->scale_row) || !aligned16(out->amax_row))
      return NVFP4_ERR_ALIGN;
  }
  if (col) {
    if (M % 16 != 0) return NVFP4_ERR_SHAPE;
    if (out->amax_col == nullptr) return NVFP4_ERR_NULL;
    if (M > 0 && N > 0 && (out->data_col == nullptr || out->scale_col == nullptr)) return NVFP4_ERR_NULL;
    if (!aligned16(out->data_col) || !aligned16(out->scale_col) || !aligned16(out->amax_col))
      return NVFP4_ERR_ALIGN;
  }
  if (row && col && out->amax_row == out->amax_col) return NVFP4_ERR_FLAGS;
  if ((flags & NVFP4_SWIZZLED) && (M % 128 != 0 || N % 128 != 0)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

// Tensor map of x for a call, encoded before the call enqueues anything (so a
// map that cannot be encoded leaves every buffer untouched).  Encoding is a
// driver call of about a microsecond and callers quantize the same buffers
// over and over, so each thread keeps its last few maps, keyed by what the
// map encodes (address, shape, element type): a map holds no device state.
struct MapEntry {
  CUtensorMap map;
  const void* x;
  int64_t M, N;
  int kind;  // element type: 0 FP32, 1 BF16, 2 byte
  int used;
};
constexpr int kMapCache = 8;
thread_local MapEntry t_maps[kMapCache];
thread_local int t_map_next = 0;

nvfp4_status cached_map(const void* x, int kind, int64_t M, int64_t N, CUtensorMap* map) {
  for (int i = 0; i < kMapCache; ++i) {
    const MapEntry& e = t_maps[i];
    if (e.used && e.x == x && e.M == M && e.N == N && e.kind == kind) {
      *map = e.map;
      return NVFP4_OK;
    }
  }
  const cudaError_t r =
      kind == 2 ? make_byte_tensor_map(map, x, M, N) : make_x_tensor_map(map, x, kind == 1, M, N);
  if (r != cudaSuccess) return NVFP4_ERR_CUDA;
  MapEntry& e = t_maps[t_map_next];
  t_map_next = (t_map_next + 1) % kMapCache;
  e.map = *map;
  e.x = x;
  e.M = M;
  e.N = N;
  e.kind = kind;
  e.used = 1;
  return NVFP4_OK;
}
nvfp4_status x_map(const void* x, bool bf16, int64_t M, int64_t N, CUtensorMap* map) {
  return cached_map(x, bf16 ? 1 : 0, M, N, map);
}

nvfp4_status quantize_per_tensor(int mode, const void* x, int dtype, int64_t M, int64_t N,
                                 const nvfp4_output* out, unsigned flags, uint32_t sign_mask, const float* noop,
                                 void* stream) {
  const unsigned allowed = NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_SWIZZLED | NVFP4_SKIP_AMAX;
  nvfp4_status st = check_quantize(x, dtype, M, N, out, flags, allowed);
  if (st != NVFP4_OK) return st;
  if (mode == kCast2D && (M % 16 != 0 || N % 16 != 0)) return NVFP4_ERR_SHAPE;
  if (mode == kCastRHT) {
    if (dtype != NVFP4_BF16) return NVFP4_ERR_DTYPE;
    if (M % 16 != 0 || N % 16 != 0) return NVFP4_ERR_SHAPE;
  }
  if (noop != nullptr && !aligned16(noop)) return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  if ((st = make_ctx(stream, &ctx)) != NVFP4_OK) return st;
  const bool row = flags & NVFP4_ROWWISE, col = flags & NVFP4_COLWISE;
  const bool bf16 = dtype == NVFP4_BF16;
  float* a_row = row ? out->amax_row : nullptr;
  float* a_col = col ? out->amax_col : nullptr;
  const bool skip = flags & NVFP4_SKIP_AMAX;
  CUtensorMap map;
  if (M > 0 && N > 0 && (st = x_map(x, bf16, M, N, &map)) != NVFP4_OK) return st;
  if (!skip) {
    cudaError_t e;
    if (mode == kCastRHT && col && M > 0 && N > 0)
      e = launch_rht_amax(static_cast<const uint16_t*>(x), M, N, sign_mask, a_row, a_col, noop, ctx);
    else
      e = launch_amax(x, bf16, M * N, a_row ? a_row : a_col, a_row ? a_col : nullptr, noop, ctx);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (M == 0 || N == 0) return NVFP4_OK;
  CastArgs a = {};
  a.M = M;
  a.N = N;
  a.data_row = row ? out->data_row : nullptr;
  a.scale_row = row ? out->scale_row : nullptr;
  a.amax_row = a_row;
  a.data_col = col ? out->data_col : nullptr;
  a.scale_col = col ? out->scale_col : nullptr;
  a.amax_col = a_col;
  a.noop = noop;
  a.status = ctx.status;
  a.rowwise = row;
  a.colwise = col;
  a.swizzled = (flags & NVFP4_SWIZZLED) != 0;
  a.sign_mask = sign_mask & 0xFFFFu;
  // Without the column-wise output the transform plays no part: the row-wise
  // output is the 1D cast of x (amax max|x|), by the kernel that has no
  // tensor-core column pass.
  const int cast_mode = (mode == kCastRHT && !col) ? kCast1D : mode;
  return from_cuda(launch_cast(map, bf16, cast_mode, a, /*pdl=*/!skip, ctx));
}

nvfp4_status quantize_single_pass(int mode, const void* x, int dtype, int64_t M, int64_t N,
                                  const nvfp4_output* out, unsigned flags, const float* noop, void* workspace,
                                  void* stream) {
  const unsigned allowed = NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_SWIZZLED;
  nvfp4_status st = check_quantize(x, dtype, M, N, out, flags, allowed);
  if (st != NVFP4_OK) return st;
  if (mode == kCast2D && (M % 16 != 0 || N % 16 != 0)) return NVFP4_ERR_SHAPE;
  if (workspace == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(workspace) || (noop != nullptr && !aligned16(noop))) return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  if ((st = make_ctx(stream, &ctx)) != NVFP4_OK) return st;
  const bool row = flags & NVFP4_ROWWISE, col = flags & NVFP4_COLWISE;
  if (M == 0 || N == 0) {
    // nothing to cast: the amax of an empty tensor is 0
    return from_cuda(launch_amax(x, dtype == NVFP4_BF16, 0, row ? out->amax_row : out->amax_col,
                                 row && col ? out->amax_col : nullptr, noop, ctx));
  }
  CastArgs a = {};
  a.M = M;
  a.N = N;
  a.data_row = row ? out->data_row : nullptr;
  a.scale_row = row ? out->scale_row : nullptr;
  a.amax_row = row ? out->amax_row : nullptr;
  a.data_col = col ? out->data_col : nullptr;
  a.scale_col = col ? out->scale_col : nullptr;
  a.amax_col = col ? out->amax_col : nullptr;
  a.noop = noop;
  a.status = ctx.status;
  a.rowwise = row;
  a.colwise = col;
  a.swizzled = (flags & NVFP4_SWIZZLED) != 0;
  CUtensorMap map;
  if ((st = x_map(x, dtype == NVFP4_BF16, M, N, &map)) != NVFP4_OK) return st;
  return from_cuda(launch_single_pass(map, dtype == NVFP4_BF16, mode, a,
                                      static_cast<SinglePassWorkspace*>(workspace), ctx));
}

// Quantize with stochastically rounded codes: the checks of the plain
// quantize, plus the random bytes (one per element of x, 16-byte aligned).
nvfp4_status quantize_sr(int mode, const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                         unsigned flags, const uint8_t* rbits, const float* noop, void* stream) {
  const unsigned allowed = NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_SWIZZLED | NVFP4_SKIP_AMAX;
  nvfp4_status st = check_quantize(x, dtype, M, N, out, flags, allowed);
  if (st != NVFP4_OK) return st;
  if (mode == kCast2D && M % 16 != 0) return NVFP4_ERR_SHAPE;
  if (M > 0 && N > 0 && rbits == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(rbits)) return NVFP4_ERR_ALIGN;
  if (noop != nullptr && !aligned16(noop)) return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  if ((st = make_ctx(stream, &ctx)) != NVFP4_OK) return st;
  const bool row = flags & NVFP4_ROWWISE, col = flags & NVFP4_COLWISE;
  float* a_row = row ? out->amax_row : nullptr;
  float* a_col = col ? out->amax_col : nullptr;
  const bool skip = flags & NVFP4_SKIP_AMAX;
  CUtensorMap map, rmap;
  if (M > 0 && N > 0 && (st = x_map(x, dtype == NVFP4_BF16, M, N, &map)) != NVFP4_OK) return st;
  if (M > 0 && N > 0 && (st = cached_map(rbits, 2, M, N, &rmap)) != NVFP4_OK) return st;
  if (!skip && launch_amax(x, dtype == NVFP4_BF16, M * N, a_row ? a_row : a_col, a_row ? a_col : nullptr, noop,
                           ctx) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  if (M == 0 || N == 0) return NVFP4_OK;
  CastArgs a = {};
  a.M = M;
  a.N = N;
  a.data_row = row ? out->data_row : nullptr;
  a.scale_row = row ? out->scale_row : nullptr;
  a.amax_row = a_row;
  a.data_col = col ? out->data_col : nullptr;
  a.scale_col = col ? out->scale_col : nullptr;
  a.amax_col = a_col;
  a.noop = noop;
  a.status = ctx.status;
  a.rowwise = row;
  a.colwise = col;
  a.swizzled = (flags & NVFP4_SWIZZLED) != 0;
  return from_cuda(launch_cast_sr(map, dtype == NVFP4_BF16, mode, a, rmap, /*pdl=*/!skip, ctx));
}

static_assert(NVFP4_MAX_GROUPS == kMaxGroups, "member table size");

// Grouped quantize: every member is checked as a plain quantize of its rows
// (its slice of x and its outputs), then the member table is filled.
// With a workspace, the single-launch form (BF16, no SKIP_AMAX).
nvfp4_status quantize_grouped(int mode, const void* x, int dtype, int64_t N, int num_groups,
                              const int64_t* group_rows, const nvfp4_output* outs, unsigned flags,
                              const float* noop, void* workspace, bool single_pass, void* stream) {
  if (group_rows == nullptr || outs == nullptr) return NVFP4_ERR_NULL;
  if (num_groups < 1 || num_groups > kMaxGroups) return NVFP4_ERR_SHAPE;
  if (dtype != NVFP4_BF16 && dtype != NVFP4_FP32) return NVFP4_ERR_DTYPE;
  if (single_pass && dtype != NVFP4_BF16) return NVFP4_ERR_DTYPE;
  if (N < 0 || N >= kMaxDim || N % 16 != 0) return NVFP4_ERR_SHAPE;
  const unsigned allowed =
      NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_SWIZZLED | (single_pass ? 0u : (unsigned)NVFP4_SKIP_AMAX);
  const bool row = flags & NVFP4_ROWWISE, col = flags & NVFP4_COLWISE;
  const int64_t eb = dtype == NVFP4_BF16 ? 2 : 4;
  GroupedArgs ga = {};
  int64_t total = 0;
  for (int g = 0; g < num_groups; ++g) {
    const int64_t rows = group_rows[g];
    if (rows < 0 || rows >= kMaxDim) return NVFP4_ERR_SHAPE;
    if ((col || mode == kCast2D) && rows % 16 != 0) return NVFP4_ERR_SHAPE;
    const void* xg = x == nullptr ? nullptr : static_cast<const char*>(x) + total * N * eb;
    nvfp4_status st = check_quantize(xg, dtype, rows, N, &outs[g], flags, allowed);
    if (st != NVFP4_OK) return st;
    ga.row0[g] = total;
    ga.rows[g] = rows;
    ga.data_row[g] = row ? outs[g].data_row : nullptr;
    ga.scale_row[g] = row ? outs[g].scale_row : nullptr;
    ga.amax_row[g] = row ? outs[g].amax_row : nullptr;
    ga.data_col[g] = col ? outs[g].data_col : nullptr;
    ga.scale_col[g] = col ? outs[g].scale_col : nullptr;
    ga.amax_col[g] = col ? outs[g].amax_col : nullptr;
    total += rows;
    if (total >= kMaxDim) return NVFP4_ERR_SHAPE;
  }
  // Each member owns its amax buffers: two members that shared one would
  // merge their maxima.
  const float* seen[2 * kMaxGroups];
  int n_seen = 0;
  for (int g = 0; g < num_groups; ++g)
    for (const float* p : {static_cast<const float*>(ga.amax_row[g]), static_cast<const float*>(ga.amax_col[g])}) {
      if (p == nullptr) continue;
      for (int i = 0; i < n_seen; ++i)
        if (seen[i] == p) return NVFP4_ERR_FLAGS;
      seen[n_seen++] = p;
    }
  if (noop != nullptr && !aligned16(noop)) return NVFP4_ERR_ALIGN;
  if (single_pass && workspace == nullptr) return NVFP4_ERR_NULL;
  if (single_pass && !aligned16(workspace)) return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  nvfp4_status st = make_ctx(stream, &ctx);
  if (st != NVFP4_OK) return st;
  ga.num_groups = num_groups;
  ga.N = N;
  ga.noop = noop;
  ga.status = ctx.status;
  ga.rowwise = row;
  ga.colwise = col;
  ga.swizzled = (flags & NVFP4_SWIZZLED) != 0;
  CUtensorMap map = {};
  const bool any = total > 0 && N > 0;
  if (any && (st = x_map(x, dtype == NVFP4_BF16, total, N, &map)) != NVFP4_OK) return st;
  if (single_pass)
    return from_cuda(
        launch_grouped_single_pass(map, mode, ga, static_cast<SinglePassWorkspace*>(workspace), ctx));
  return from_cuda(launch_grouped(x, any ? &map : nullptr, dtype == NVFP4_BF16, mode, ga,
                                  (flags & NVFP4_SKIP_AMAX) != 0, ctx));
}

}  // namespace

// The host-side checks of the single-pass entry points (everything before
// the launch), for callers that supply their own scratch.
nvfp4_status validate_single_pass(int mode, const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                                  unsigned flags, const float* noop) {
  nvfp4_status st = check_quantize(x, dtype, M, N, out, flags, NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_SWIZZLED);
  if (st != NVFP4_OK) return st;
  if (mode == kCast2D && (M % 16 != 0 || N % 16 != 0)) return NVFP4_ERR_SHAPE;
  if (noop != nullptr && !aligned16(noop)) return NVFP4_ERR_ALIGN;
  return NVFP4_OK;
}

cudaError_t make_x_tensor_map(CUtensorMap* map, const void* x, bool bf16, int64_t M, int64_t N) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  const int eb = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)N * eb};
  cuuint32_t box[2] = {(cuuint32_t)(128 / eb), 128u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                      const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_byte_tensor_map(CUtensorMap* map, const void* p, int64_t M, int64_t N) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)M};
  cuuint64_t strides[1] = {(cuuint64_t)N};
  cuuint32_t box[2] = {128u, 128u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(p), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_NULL: return "NVFP4_ERR_NULL: a required pointer is NULL";
    case NVFP4_ERR_SHAPE: return "NVFP4_ERR_SHAPE: bad size (negative, or a blocked dimension not a multiple of 16)";
    case NVFP4_ERR_ALIGN:
      return "NVFP4_ERR_ALIGN: swizzled scales need 128-aligned dimensions; pointers must be 16-byte aligned";
    case NVFP4_ERR_DTYPE: return "NVFP4_ERR_DTYPE: unsupported dtype for this operation";
    case NVFP4_ERR_FLAGS: return "NVFP4_ERR_FLAGS: unknown or contradictory flags, or aliased amax buffers";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA: a CUDA launch failed";
    case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT: a device-side wait ran out";
  }
  return "unknown nvfp4_status";
}

nvfp4_status nvfp4_scale_bytes(int64_t rows, int64_t cols, unsigned flags, size_t* bytes) {
  if (bytes == nullptr) return NVFP4_ERR_NULL;
  if (rows < 0 || cols < 0 || cols % 16 != 0) return NVFP4_ERR_SHAPE;
  if ((flags & NVFP4_SWIZZLED) && (rows % 128 != 0 || cols % 128 != 0)) return NVFP4_ERR_ALIGN;
  *bytes = (size_t)rows * (size_t)(cols / 16);
  return NVFP4_OK;
}

nvfp4_status nvfp4_compute_amax(const void* x, int dtype, int64_t M, int64_t N, float* amax_row,
                                float* amax_col, const float* noop, void* stream) {
  if (dtype != NVFP4_BF16 && dtype != NVFP4_FP32) return NVFP4_ERR_DTYPE;
  if (M < 0 || N < 0) return NVFP4_ERR_SHAPE;
  if (amax_row == nullptr) return NVFP4_ERR_NULL;
  if (M > 0 && N > 0 && x == nullptr) return NVFP4_ERR_NULL;
  if (amax_row == amax_col) return NVFP4_ERR_FLAGS;
  if ((x != nullptr && !aligned16(x)) || !aligned16(amax_row) || (amax_col && !aligned16(amax_col)) ||
      (noop && !aligned16(noop)))
    return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  nvfp4_status st = make_ctx(stream, &ctx);
  if (st != NVFP4_OK) return st;
  return from_cuda(launch_amax(x, dtype == NVFP4_BF16, M * N, amax_row, amax_col, noop, ctx));
}

nvfp4_status nvfp4_compute_amax_rht(const void* x, int dtype, int64_t M, int64_t N, uint32_t sign_mask,
                                    float* amax_row, float* amax_col, const float* noop, void* stream) {
  if (dtype != NVFP4_BF16) return NVFP4_ERR_DTYPE;
  if (M < 0 || N < 0 || M % 16 != 0 || N % 16 != 0) return NVFP4_ERR_SHAPE;
  if (amax_row == nullptr || amax_col == nullptr) return NVFP4_ERR_NULL;
  if (M > 0 && N > 0 && x == nullptr) return NVFP4_ERR_NULL;
  if (amax_row == amax_col) return NVFP4_ERR_FLAGS;
  if ((x != nullptr && !aligned16(x)) || !aligned16(amax_row) || !aligned16(amax_col) ||
      (noop && !aligned16(noop)))
    return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  nvfp4_status st = make_ctx(stream, &ctx);
  if (st != NVFP4_OK) return st;
  if (M == 0 || N == 0) return from_cuda(launch_amax(x, true, 0, amax_row, amax_col, noop, ctx));
  return from_cuda(
      launch_rht_amax(static_cast<const uint16_t*>(x), M, N, sign_mask, amax_row, amax_col, noop, ctx));
}

nvfp4_status nvfp4_quantize_1d(const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                               unsigned flags, const float* noop, void* stream) {
  return quantize_per_tensor(kCast1D, x, dtype, M, N, out, flags, 0, noop, stream);
}

nvfp4_status nvfp4_quantize_2d(const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                               unsigned flags, const float* noop, void* stream) {
  return quantize_per_tensor(kCast2D, x, dtype, M, N, out, flags, 0, noop, stream);
}

nvfp4_status nvfp4_quantize_rht(const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                                unsigned flags, uint32_t sign_mask, const float* noop, void* stream) {
  return quantize_per_tensor(kCastRHT, x, dtype, M, N, out, flags, sign_mask, noop, stream);
}

nvfp4_status nvfp4_quantize_1d_single_pass(const void* x, int dtype, int64_t M, int64_t N,
                                           const nvfp4_output* out, unsigned flags, const float* noop,
                                           void* workspace, void* stream) {
  return quantize_single_pass(kCast1D, x, dtype, M, N, out, flags, noop, workspace, stream);
}

nvfp4_status nvfp4_quantize_2d_single_pass(const void* x, int dtype, int64_t M, int64_t N,
                                           const nvfp4_output* out, unsigned flags, const float* noop,
                                           void* workspace, void* stream) {
  return quantize_single_pass(kCast2D, x, dtype, M, N, out, flags, noop, workspace, stream);
}

nvfp4_status nvfp4_quantize_rht_single_pass(const void* x, int dtype, int64_t M, int64_t N,
                                            const nvfp4_output* out, unsigned flags, uint32_t sign_mask,
                                            const float* noop, void* workspace, void* stream) {
  if (!(flags & NVFP4_COLWISE))  // rows of x only: the transform plays no part
    return quantize_single_pass(kCast1D, x, dtype, M, N, out, flags, noop, workspace, stream);
  const unsigned allowed = NVFP4_ROWWISE | NVFP4_COLWISE | NVFP4_SWIZZLED;
  nvfp4_status st = check_quantize(x, dtype, M, N, out, flags, allowed);
  if (st != NVFP4_OK) return st;
  if (dtype != NVFP4_BF16) return NVFP4_ERR_DTYPE;
  if (M % 16 != 0 || N % 16 != 0) return NVFP4_ERR_SHAPE;
  if (workspace == nullptr) return NVFP4_ERR_NULL;
  if (!aligned16(workspace) || (noop != nullptr && !aligned16(noop))) return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  if ((st = make_ctx(stream, &ctx)) != NVFP4_OK) return st;
  const bool row = flags & NVFP4_ROWWISE;
  if (M == 0 || N == 0) {
    // nothing to cast: both maxima of an empty tensor are 0
    return from_cuda(launch_amax(x, true, 0, row ? out->amax_row : out->amax_col, row ? out->amax_col : nullptr,
                                 noop, ctx));
  }
  CastArgs a = {};
  a.M = M;
  a.N = N;
  a.data_row = row ? out->data_row : nullptr;
  a.scale_row = row ? out->scale_row : nullptr;
  a.amax_row = row ? out->amax_row : nullptr;
  a.data_col = out->data_col;
  a.scale_col = out->scale_col;
  a.amax_col = out->amax_col;
  a.noop = noop;
  a.status = ctx.status;
  a.rowwise = row;
  a.colwise = 1;
  a.swizzled = (flags & NVFP4_SWIZZLED) != 0;
  a.sign_mask = sign_mask & 0xFFFFu;
  CUtensorMap map;
  if ((st = x_map(x, true, M, N, &map)) != NVFP4_OK) return st;
  return from_cuda(launch_single_pass_rht(map, a, static_cast<SinglePassWorkspace*>(workspace), ctx));
}

nvfp4_status nvfp4_quantize_row_scaled(const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                                       unsigned flags, const float* noop, void* stream) {
  const unsigned allowed = NVFP4_ROWWISE | NVFP4_SWIZZLED | NVFP4_SKIP_AMAX;
  nvfp4_status st = check_quantize(x, dtype, M, N, out, flags, allowed);
  if (st != NVFP4_OK) return st;
  if (!(flags & NVFP4_ROWWISE)) return NVFP4_ERR_FLAGS;
  if (noop != nullptr && !aligned16(noop)) return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  if ((st = make_ctx(stream, &ctx)) != NVFP4_OK) return st;
  if (N == 0) {
    // Every row is empty: its amax is 0.
    if (flags & NVFP4_SKIP_AMAX || M == 0) return NVFP4_OK;
    return from_cuda(cudaMemsetAsync(out->amax_row, 0, sizeof(float) * (size_t)M, ctx.stream));
  }
  return from_cuda(launch_row_scaled(x, dtype == NVFP4_BF16, M, N, out->data_row, out->scale_row, out->amax_row,
                                     (flags & NVFP4_SKIP_AMAX) != 0, (flags & NVFP4_SWIZZLED) != 0, noop, ctx));
}

nvfp4_status nvfp4_quantize_1d_sr(const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                                  unsigned flags, const uint8_t* rbits, const float* noop, void* stream) {
  return quantize_sr(kCast1D, x, dtype, M, N, out, flags, rbits, noop, stream);
}

nvfp4_status nvfp4_quantize_2d_sr(const void* x, int dtype, int64_t M, int64_t N, const nvfp4_output* out,
                                  unsigned flags, const uint8_t* rbits, const float* noop, void* stream) {
  return quantize_sr(kCast2D, x, dtype, M, N, out, flags, rbits, noop, stream);
}

nvfp4_status nvfp4_quantize_grouped_1d(const void* x, int dtype, int64_t N, int num_groups,
                                       const int64_t* group_rows, const nvfp4_output* outs, unsigned flags,
                                       const float* noop, void* stream) {
  return quantize_grouped(kCast1D, x, dtype, N, num_groups, group_rows, outs, flags, noop, nullptr, false, stream);
}

nvfp4_status nvfp4_quantize_grouped_2d(const void* x, int dtype, int64_t N, int num_groups,
                                       const int64_t* group_rows, const nvfp4_output* outs, unsigned flags,
                                       const float* noop, void* stream) {
  return quantize_grouped(kCast2D, x, dtype, N, num_groups, group_rows, outs, flags, noop, nullptr, false, stream);
}

nvfp4_status nvfp4_quantize_grouped_1d_single_pass(const void* x, int dtype, int64_t N, int num_groups,
                                                   const int64_t* group_rows, const nvfp4_output* outs,
                                                   unsigned flags, const float* noop, void* workspace,
                                                   void* stream) {
  return quantize_grouped(kCast1D, x, dtype, N, num_groups, group_rows, outs, flags, noop, workspace, true, stream);
}

nvfp4_status nvfp4_quantize_grouped_2d_single_pass(const void* x, int dtype, int64_t N, int num_groups,
                                                   const int64_t* group_rows, const nvfp4_output* outs,
                                                   unsigned flags, const float* noop, void* workspace,
                                                   void* stream) {
  return quantize_grouped(kCast2D, x, dtype, N, num_groups, group_rows, outs, flags, noop, workspace, true, stream);
}

nvfp4_status nvfp4_dequantize(const uint8_t* data, const uint8_t* scale, const float* amax, int64_t rows,
                              int64_t cols, unsigned flags, void* out, int out_dtype, void* stream) {
  if (flags & ~(NVFP4_SWIZZLED | NVFP4_ROW_SCALED)) return NVFP4_ERR_FLAGS;
  if (out_dtype != NVFP4_BF16 && out_dtype != NVFP4_FP32) return NVFP4_ERR_DTYPE;
  if (rows < 0 || cols < 0 || cols % 16 != 0) return NVFP4_ERR_SHAPE;
  if ((flags & NVFP4_SWIZZLED) && (rows % 128 != 0 || (cols / 16) % 4 != 0)) return NVFP4_ERR_ALIGN;
  if (rows > 0 && cols > 0 && (data == nullptr || scale == nullptr || amax == nullptr || out == nullptr))
    return NVFP4_ERR_NULL;
  if (!aligned16(data) || !aligned16(scale) || !aligned16(amax) || !aligned16(out)) return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  nvfp4_status st = make_ctx(stream, &ctx);
  if (st != NVFP4_OK) return st;
  return from_cuda(launch_dequantize(data, scale, amax, rows, cols, (flags & NVFP4_SWIZZLED) != 0,
                                     (flags & NVFP4_ROW_SCALED) != 0, out, out_dtype == NVFP4_BF16, ctx));
}

nvfp4_status nvfp4_swizzle_scales(const uint8_t* compact, uint8_t* swizzled, int64_t rows, int64_t scale_cols,
                                  void* stream) {
  if (rows < 0 || scale_cols < 0) return NVFP4_ERR_SHAPE;
  if (rows % 128 != 0 || scale_cols % 4 != 0) return NVFP4_ERR_ALIGN;
  if (rows > 0 && scale_cols > 0 && (compact == nullptr || swizzled == nullptr)) return NVFP4_ERR_NULL;
  if (!aligned16(compact) || !aligned16(swizzled)) return NVFP4_ERR_ALIGN;
  LaunchCtx ctx;
  nvfp4_status st = make_ctx(stream, &ctx);
  if (st != NVFP4_OK) return st;
  return from_cuda(launch_swizzle(compact, swizzled, rows, scale_cols, ctx));
}

nvfp4_status nvfp4_device_status(uint32_t* status, int clear) {
  if (status == nullptr) return NVFP4_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_nvfp4_status_word, sizeof v) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (clear) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_nvfp4_status_word, &zero, sizeof zero) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  *status = v;
  return v ? NVFP4_ERR_TIMEOUT : NVFP4_OK;
}

}  // extern "C"
