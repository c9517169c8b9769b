// common.cuh -- device helpers shared by the NVFP4 kernels (sm_103a).
//
// Conversions use the hardware cvt instructions with round-to-nearest-even
// and saturation (E2M1 data, E4M3 block scales), TMA tile loads complete on
// shared-memory mbarriers, and every wait is bounded.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace nvfp4 {

// Bits of the per-device status word (see nvfp4_device_status).
constexpr unsigned kStatusWaitTimeout = 1u;  // a wait for a tile copy ran out
constexpr unsigned kStatusGridTimeout = 2u;  // a grid-wide barrier ran out
// A wait that has not completed after this many SM cycles (about 2 s at the
// GB300 boost clock) is abandoned.
constexpr long long kWaitLimitCycles = 4000000000LL;

constexpr float kFltMax = 3.402823466e38f;

// ---------------------------------------------------------------------------
// Programmatic dependent launch
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Scale arithmetic
// ---------------------------------------------------------------------------

// b / 6 correctly rounded, with Markstein's FMA correction of the reciprocal
// product (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// c = RN(1/6), q = RN(b*c) and the exact residual e = b - 6q (one FMA),
// RN(q + e*c) is the correctly rounded quotient.  Very small b, where q
// would be subnormal, use the IEEE division.  Equality with __fdiv_rn is
// checked on the GPU over every positive FP32 value.
__device__ __forceinline__ float div6_rn(float b) {
  if (b < 1.0e-30f) return __fdiv_rn(b, 6.0f);
  const float c = 1.0f / 6.0f;
  float q = __fmul_rn(b, c);
  float e = __fmaf_rn(-q, 6.0f, b);
  return __fmaf_rn(e, c, q);
}

// FP32 global encode scale 448*6/amax; amax = 0 -> 1; overflow -> FLT_MAX.
__device__ __forceinline__ float global_encode_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  return fminf(__fdiv_rn(2688.0f, amax), kFltMax);
}

// Value of an E4M3 (FN) code 0..126, from its exponent and mantissa fields.
__device__ __forceinline__ float e4m3_decode(uint32_t c) {
  uint32_t e = (c >> 3) & 15u, m = c & 7u;
  if (e == 0) return __fmul_rn(__uint2float_rn(m), 0.001953125f);   // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Per-block encode factor r = g / float(s), clamped to FLT_MAX; 0 for s = 0.
__device__ __forceinline__ float encode_factor(uint32_t s, float g) {
  if (s == 0 || s >= 127) return 0.0f;
  return fminf(__fdiv_rn(g, e4m3_decode(s)), kFltMax);
}

// E4M3 code of a non-negative FP32 value (RNE, saturating at 448).
__device__ __forceinline__ uint32_t e4m3_rn_satfinite(float v) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.0f), "f"(v));
  return h & 0xFFu;
}

// Eight FP32 values -> eight E2M1 codes (RNE, saturating), v0 in bits 0..3.
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4,
                                           float v5, float v6, float v7) {
  uint32_t out;
  asm("{\n"
      ".reg .b8 q0, q1, q2, q3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n"
      "mov.b32 %0, {q0, q1, q2, q3};\n"
      "}"
      : "=r"(out)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return out;
}

// Stochastic rounding to E2M1 with one random byte b (0..255) per value:
// between neighbouring magnitudes lo <= |p| < hi the magnitude becomes hi
// iff b < 256 f, f = (|p| - lo) / (hi - lo); |p| >= 6 gives 6; the sign of p
// is kept.
//
// Carry form.  From 1 up, the E2M1 magnitudes are the FP32 values with a
// single mantissa bit, so with u the bits of w = min(|p|, 6) the lower
// neighbour is u's bits 22 and up and f is bits 21..0 over 2^22.  Adding
// sr_offset(b) = ((255 - b) << 14) | (2^14 - 1) to u carries into bit 22
// exactly when bits 21..0 exceed b << 14, that is when b < 256 f, and
// (u + offset) >> 22 is then the code plus 252.  Below 1 the magnitudes
// 0, 0.5, 1 are evenly spaced: v = w / 2 + 1/2 rounded up has the bits
// 0x3F000000 + ceil(2^23 w), i.e. the code plus 252 in bits 22 and up and
// ceil(2^22 f) below, which carries the same way (ceil(y) > n exactly when
// y > n for an integer n).  max(v, w) is v below 1 and w from 1 up.  Every
// step is exact; sr_code252 returns the code plus 252 (252..259).
__device__ __forceinline__ uint32_t sr_offset(uint32_t b) { return ((b ^ 0xFFu) << 14) | 0x3FFFu; }
// sr_offset of byte c (0..3) of the word w.
__device__ __forceinline__ uint32_t sr_offset_w(uint32_t w, int c) {
  return ((((w >> (8 * c)) & 0xFFu) ^ 0xFFu) << 14) | 0x3FFFu;
}
__device__ __forceinline__ uint32_t sr_code252(float abs_p, uint32_t offset) {
  const float w = fminf(abs_p, 6.0f);
  return (__float_as_uint(fmaxf(__fmaf_ru(w, 0.5f, 0.5f), w)) + offset) >> 22;
}
__device__ __forceinline__ uint32_t e2m1_sr(float p, uint32_t offset) {
  return (sr_code252(fabsf(p), offset) - 252u) | ((__float_as_uint(p) >> 28) & 8u);
}

// ---------------------------------------------------------------------------
// BF16 helpers (a 32-bit word holds two BF16 values, the lower address in
// the low half)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max(|a|, |b|) per BF16 half, as a packed pair (inputs are finite).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a & 0x7FFF7FFFu), "r"(b & 0x7FFF7FFFu));
  return r;
}
__device__ __forceinline__ float bf16x2_hmax_to_f32(uint32_t w) {
  return fmaxf(bf16_lo(w), bf16_hi(w));
}

// FP32 -> BF16 (RNE) -> FP32.
__device__ __forceinline__ float round_bf16(float v) {
  uint16_t h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// In-place 16-point Walsh-Hadamard butterflies, natural (Sylvester) order:
// after the four stages v[o] = sum_i (-1)^popcount(o & i) v_in[i].
__device__ __forceinline__ void fwht16(float* v) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        float a = v[i], c = v[i + h];
        v[i] = __fadd_rn(a, c);
        v[i + h] = __fsub_rn(a, c);
      }
    }
  }
}

// The same transform on two columns at once, each value an FP32x2 pair
// (packed adds and subtracts round each half exactly as the scalar ones).
__device__ __forceinline__ void fwht16_x2(uint64_t* v) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const uint64_t a = v[i], c = v[i + h];
        asm("add.rn.f32x2 %0, %1, %2;" : "=l"(v[i]) : "l"(a), "l"(c));
        asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(v[i + h]) : "l"(a), "l"(c));
      }
    }
  }
}
// BF16x2 word -> FP32x2 pair times (r, r).
__device__ __forceinline__ uint64_t bf16x2_scaled(uint32_t w, float r) {
  uint64_t p, v, rr;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(w << 16), "r"(w & 0xFFFF0000u));
  asm("mov.b64 %0, {%1, %1};" : "=l"(rr) : "f"(r));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(v), "l"(rr));
  return p;
}
// FP32x2 pair -> BF16x2 word (RNE), low half from the pair's low value.
__device__ __forceinline__ uint32_t pair_to_bf16x2(uint64_t v) {
  float lo, hi;
  uint32_t w;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w) : "f"(hi), "f"(lo));
  return w;
}

// ---------------------------------------------------------------------------
// Shared memory, mbarrier and TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// One bounded try: the thread may be suspended (up to ~0.1 ms) until the
// phase completes, so a waiting warp costs few issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 100000;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of an mbarrier, at most `limit` SM cycles; on
// timeout records kStatusWaitTimeout in *status and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned* status,
                                                  long long limit = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      atomicOr(status, kStatusWaitTimeout);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2D tiled TMA load of the box at (c0 = innermost, c1) into shared memory,
// completing `bytes` transactions on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int32_t c0, int32_t c1,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Bulk (non-tensor) copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory, completing `bytes` transactions on
// `bar`.
__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
               "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Generic-proxy writes to shared memory by this thread, ordered before later
// async-proxy reads of them (tensor-core operands written with st.shared).
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Bulk (non-tensor) copy of `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from shared to global memory, in this thread's bulk group.  The
// shared data must have been made visible to the async proxy first
// (fence_proxy_async_shared by each thread that wrote it, then a hand-over).
__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's committed bulk copies have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's committed bulk copies are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Tensor memory and the 5th-generation tensor cores (tcgen05)
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading- and stride-
// dimension byte offsets (16-byte units), descriptor version 1, layout
// (0: no swizzle, 2: 128-byte swizzle).  For an MN-major operand in the
// 128-byte swizzle the leading offset steps between 64-element column
// groups and the stride offset between 8-row groups along K; for a K-major
// operand without swizzle (8x8 core matrices of 128 bytes) the leading
// offset steps between core matrices along K, the stride offset along M/N.
__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
// Instruction descriptor of kind::f16 with BF16 A and B, FP32 D, A MN-major
// (a_mn) or K-major, B K-major, shape M x N.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n, bool a_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}
// D (tensor memory) = A * B (+ D when accumulate), issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
               "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
               : "memory");
}
// One arrival on `bar` when every tcgen05.mma this thread issued so far is complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tcgen05_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tcgen05_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Whole warp: allocate `ncols` tensor-memory columns (a power of two >= 32);
// the address is written to the shared word `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Whole warp: 16 consecutive 32-bit columns of the lane (32 x 32-bit shape),
// then wait for them.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

// ---------------------------------------------------------------------------
// Streaming (evict-first) global stores of outputs
// ---------------------------------------------------------------------------
// 32 bytes (one whole sector) in one store; p 32-byte aligned.
__device__ __forceinline__ void st_cs_v8(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void st_cs_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ void st_cs_v2(void* p, uint32_t a, uint32_t b) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_cs_u32(void* p, uint32_t a) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(a) : "memory");
}
// The same, executed only when `pred` is non-zero (a predicated store, no
// branch).
__device__ __forceinline__ void st_cs_u32_if(void* p, uint32_t a, uint32_t pred) {
  asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %2, 0;\n @q st.global.cs.u32 [%0], %1;\n}" ::"l"(p), "r"(a),
               "r"(pred)
               : "memory");
}
__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_u8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void st_cs_v2_if(void* p, uint32_t a, uint32_t b, bool pred) {
  asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %3, 0;\n @q st.global.cs.v2.u32 [%0], {%1, %2};\n}" ::"l"(p),
               "r"(a), "r"(b), "r"((uint32_t)pred)
               : "memory");
}
__device__ __forceinline__ void st_cs_u16(void* p, uint32_t a) {
  asm volatile("st.global.cs.u16 [%0], %1;" ::"l"(p), "h"(static_cast<uint16_t>(a)) : "memory");
}
__device__ __forceinline__ void st_cs_u8(void* p, uint32_t a) {
  asm volatile("st.global.cs.u8 [%0], %1;" ::"l"(p), "h"(static_cast<uint16_t>(a & 0xFFu)) : "memory");
}

// Byte offset of scale (r, c) in the cuBLAS 128x4 block-scaling layout of a
// scale matrix with C columns.
__device__ __forceinline__ int64_t swizzled_scale_offset(int64_t r, int64_t c, int64_t C) {
  return ((r >> 7) * (C >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// Writes n (1, 2 or 4) consecutive scale bytes (packed little-endian in v)
// of row r starting at scale column c, compact [R][C] or swizzled.  In the
// swizzled layout c is a multiple of n, so the group is contiguous and
// aligned; in the compact layout the store is split into bytes when the
// address is not aligned.
__device__ __forceinline__ void store_scales(uint8_t* base, int64_t r, int64_t c, int64_t C, bool swizzled,
                                             int n, uint32_t v) {
  int64_t off = swizzled ? swizzled_scale_offset(r, c, C) : r * C + c;
  uint8_t* p = base + off;
  if (((reinterpret_cast<uintptr_t>(p)) & (uintptr_t)(n - 1)) == 0) {
    if (n == 4) { st_cs_u32(p, v); return; }
    if (n == 2) { st_cs_u16(p, v); return; }
    if (n == 1) { st_cs_u8(p, v); return; }
  }
  for (int i = 0; i < n; ++i) st_cs_u8(p + i, v >> (8 * i));
}

}  // namespace nvfp4
