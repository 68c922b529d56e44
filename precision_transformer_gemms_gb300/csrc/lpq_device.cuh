// Device helpers for liblpq: format arithmetic (exactly one IEEE rounding per
// float operation, no contraction), the counter-based generator, the 16-point
// Hadamard butterfly, and thin inline-PTX wrappers for mbarrier, TMA and the
// fifth-generation tensor core (tcgen05) on sm_103a.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lpq_internal.h"

namespace lpq {

// ------------------------------------------------------------------ bf16 / fp32
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

// 8 bf16 from a 16-byte vector into floats (exact).
__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
  f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
  f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
  f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// max(|x|) that ignores NaN (fmaxf returns the non-NaN operand).
__device__ __forceinline__ float absmax_acc(float m, float x) { return fmaxf(m, fabsf(x)); }

__device__ __forceinline__ bool finite_pos(float a) { return a > 0.f && a <= 3.402823466e38f; }

// ------------------------------------------------------------------ conversions
// Two fp32 -> packed E4M3 / E5M2 bytes, round-to-nearest-even, saturating.
// Result byte 0 encodes `lo`, byte 1 encodes `hi`.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint16_t cvt_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two fp32 -> packed E2M1 nibbles (low nibble encodes `lo`), RNE, saturating.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Eight fp32 -> eight E2M1 codes packed into 32 bits (nibble i = value i),
// RNE, saturating: four paired conversions and one byte pack.
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float v[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(r) : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}
template <bool kE5M2>
__device__ __forceinline__ uint16_t cvt_fp8x2(float lo, float hi) {
  if constexpr (kE5M2) return cvt_e5m2x2(lo, hi); else return cvt_e4m3x2(lo, hi);
}

// Value of an E4M3 code 0..0x7E as fp32 (exact: via the f16 conversion).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  uint16_t in = (uint16_t)(code & 0xFF);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

// 2^k as fp32 for k in [-127, 127]; 2^-127 is the subnormal 0x00400000.
__device__ __forceinline__ float pow2_exact(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

// MX block exponent: the smallest e with fmax * 2^e >= a (a >= 0), where the
// element format's largest value is fmax = mf * 2^EMAX (E4M3 448 = 1.75 * 2^8,
// E5M2 57344 = 1.75 * 2^15, E2M1 6 = 1.5 * 2^2).  From the exact
// decomposition a = m * 2^E: e = E - EMAX + (m > mf), clamped to [-127, 127];
// a = 0 gives -127, a non-finite amax gives 127.  kMfFrac is the 23-bit
// fraction of mf.
template <int EMAX, uint32_t kMfFrac>
__device__ __forceinline__ int mx_exponent_t(float a) {
  if (a == 0.f) return -127;
  uint32_t b = __float_as_uint(a);
  uint32_t be = (b >> 23) & 0xFF, frac = b & 0x7FFFFF;
  if (be == 0xFF) return 127;
  int E;
  if (be == 0) {  // subnormal: normalise the significand
    int p = 31 - __clz(frac);
    E = p - 149;
    frac = (frac << (23 - p)) & 0x7FFFFF;
  } else {
    E = (int)be - 127;
  }
  int e = E - EMAX + (frac > kMfFrac ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}
__device__ __forceinline__ int mx_exponent(float a) { return mx_exponent_t<8, 0x600000u>(a); }       // E4M3
__device__ __forceinline__ int mx_exponent_e5m2(float a) { return mx_exponent_t<15, 0x600000u>(a); }  // E5M2
__device__ __forceinline__ int mx_exponent_e2m1(float a) { return mx_exponent_t<2, 0x400000u>(a); }   // E2M1

// Correctly rounded x / 6 for x >= 0 (a block max) by division by a constant
// with one fused-multiply-add correction (P. Markstein, "IA-64 and Elementary
// Functions", 2000; N. Brisebarre and J.-M. Muller, "Correctly rounded
// multiplication by arbitrary precision constants", IEEE TC 2008): q = the
// product with RN(1/6), then q + RN(1/6) * (x - 6 q) with the exact residual
// x - 6 q from an FMA.  Below 2^-120, where the quotient can be subnormal and
// the correction is not exact, and for infinity, the IEEE division itself.
// Equal to the IEEE quotient for every non-negative float: the test suite
// checks all 2^31 of them on the device (lpq_selftest_arith, which 0).
__device__ __forceinline__ float div6_rn(float x) {
  if (!(x >= 7.52316385e-37f && x < __int_as_float(0x7F800000))) return __fdiv_rn(x, 6.0f);  // 2^-120
  const float q = __fmul_rn(x, 0.16666667f);
  return __fmaf_rn(__fmaf_rn(-q, 6.0f, x), 0.16666667f, q);
}

// ------------------------------------------------------------------ Philox-4x32-10
// Salmon et al., SC'11: per round the even words are multiplied by the two
// multipliers, hi/lo halves mixed with the odd words and the round key; the
// key is bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;  // one wide multiply gives both halves
    const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
    c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1, (uint32_t)p0);
  }
  return c;
}

// Philox-4x32-10 with the ten round keys precomputed (the key schedule only
// depends on the seed, so a thread that draws many words computes it once).
struct PhiloxKeys {
  uint32_t k0[10], k1[10];
  __device__ __forceinline__ explicit PhiloxKeys(uint64_t seed) {
    uint32_t a = (uint32_t)seed, b = (uint32_t)(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
      k0[r] = a;
      k1[r] = b;
      a += 0x9E3779B9u;
      b += 0xBB67AE85u;
    }
  }
  __device__ __forceinline__ uint4 operator()(uint4 c) const {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
      const uint64_t p0 = (uint64_t)0xD2511F53u * c.x;
      const uint64_t p1 = (uint64_t)0xCD9E8D57u * c.z;
      c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0[r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1[r], (uint32_t)p0);
    }
    return c;
  }
  // 4 random words for elements j = 4g .. 4g+3 of copy `copy_id`.
  __device__ __forceinline__ uint4 words(uint64_t g, uint32_t copy_id) const {
    return (*this)(make_uint4((uint32_t)g, (uint32_t)(g >> 32), copy_id, 0u));
  }
};

__device__ __forceinline__ uint32_t rht_signs(uint32_t rht_seed) {
  return philox4x32_10(make_uint4(0u, 0u, 2u, 0u), rht_seed, 0u).x & 0xFFFFu;
}

// The 16 random signs as factors +1 / -1 (bit j of `signs` set: -1), so that
// the sign flip is a multiply (exact) rather than a select.
__device__ __forceinline__ void rht_sign_factors(uint32_t signs, float sgn[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) sgn[j] = ((signs >> j) & 1u) ? -1.0f : 1.0f;
}

// 16-point random-sign Hadamard: sign flip, butterfly stages h = 1, 2, 4, 8
// ((t_i, t_{i+h}) -> (t_i + t_{i+h}, t_i - t_{i+h})), then * 1/4.
__device__ __forceinline__ void rht16(float t[16], const float sgn[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = __fmul_rn(sgn[j], t[j]);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((i & h) == 0) {
        float a = t[i], b = t[i + h];
        t[i] = __fadd_rn(a, b);
        t[i + h] = __fsub_rn(a, b);
      }
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = __fmul_rn(0.25f, t[j]);
}

// The same transform with the signs taken from a 16-bit mask (bit j set: -1)
// by flipping sign bits (exact like the multiply, without the 16 registers of
// the factors), the butterflies and the final scaling as packed two-wide
// operations: the quantizers' column-wise RHT.
__device__ __forceinline__ void rht16(float t[16], uint32_t signs) {
#pragma unroll
  for (int j = 0; j < 16; ++j) t[j] = __uint_as_float(__float_as_uint(t[j]) ^ ((signs << (31 - j)) & 0x80000000u));
  // Butterflies two at a time with packed two-wide operations, each half
  // rounded like the scalar step: (a, b) -> (a + b, a - b), the difference as
  // fma(b, -1, a) (the product is exact).
#pragma unroll
  for (int h = 1; h < 16; h <<= 1) {
    int idx[8], n = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((i & h) == 0) idx[n++] = i;
#pragma unroll
    for (int p = 0; p < 8; p += 2) {
      const int i0 = idx[p], i1 = idx[p + 1];
      const float2 a = make_float2(t[i0], t[i1]), b = make_float2(t[i0 + h], t[i1 + h]);
      const float2 sum = __fadd2_rn(a, b);
      const float2 dif = __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
      t[i0] = sum.x; t[i1] = sum.y;
      t[i0 + h] = dif.x; t[i1 + h] = dif.y;
    }
  }
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const float2 r = __fmul2_rn(make_float2(t[j], t[j + 1]), make_float2(0.25f, 0.25f));
    t[j] = r.x; t[j + 1] = r.y;
  }
}

// Stochastic E2M1 rounding of y with random word r: between adjacent
// magnitudes lo <= |y| <= hi, round up iff float(r >> 8) < ((|y| - lo) /
// (hi - lo)) * 2^24.  Returned as the rounded value (a grid point with the
// sign of y; +6 for NaN, saturating at 6), which cvt.rn.satfinite.e2m1x2
// encodes exactly.  Written for the FMA pipe (the SR quantizers are bound by
// the integer/logic pipe): the spacing d = hi - lo is 2^(k-1) for 2^k the
// power-of-two part of max(|y|, 1) (0.5 below 2, 1 in [2, 4), 2 in [4, 6]);
// q = |y| / d and floor(q) are exact, so (q - floor(q)) * 2^24 is the
// threshold of the definition, and the up/down decision is the saturated
// product of the difference thr - float(r >> 8) (its sign exact) scaled by
// 2^127 (1 when positive, else 0).
// Two values at a time: the six floating-point steps run as packed two-wide
// operations, each half rounded exactly like the scalar operation.
__device__ __forceinline__ float2 sr_e2m1_value2(float2 y, uint32_t r0, uint32_t r1) {
  const float c0 = fmaxf(fminf(y.x, 6.0f), -6.0f), c1 = fmaxf(fminf(y.y, 6.0f), -6.0f);
  const uint32_t e0 = __float_as_uint(fmaxf(fabsf(c0), 1.0f)) & 0x7F800000u;
  const uint32_t e1 = __float_as_uint(fmaxf(fabsf(c1), 1.0f)) & 0x7F800000u;
  const float2 d = __fmul2_rn(make_float2(__uint_as_float(e0), __uint_as_float(e1)), make_float2(0.5f, 0.5f));
  const float2 q = __fmul2_rn(make_float2(fabsf(c0), fabsf(c1)),
                              make_float2(__uint_as_float(0x7F800000u - e0), __uint_as_float(0x7F800000u - e1)));
  const float2 fl = make_float2(floorf(q.x), floorf(q.y));
  const float2 fr = __fadd2_rn(q, make_float2(-fl.x, -fl.y));  // q - fl, exact
  const float2 diff = __ffma2_rn(fr, make_float2(16777216.0f, 16777216.0f),
                                 make_float2(-(float)(r0 >> 8), -(float)(r1 >> 8)));
  const float2 up = make_float2(__saturatef(__fmul_rn(diff.x, 1.70141183e38f)),
                                __saturatef(__fmul_rn(diff.y, 1.70141183e38f)));
  const float2 v = __fmul2_rn(__fadd2_rn(fl, up), d);
  return make_float2(__uint_as_float(__float_as_uint(v.x) | (__float_as_uint(c0) & 0x80000000u)),
                     __uint_as_float(__float_as_uint(v.y) | (__float_as_uint(c1) & 0x80000000u)));
}

// ------------------------------------------------------------------ warp helpers
__device__ __forceinline__ float warp_max_xor(float v, int width_lanes) {
  for (int o = 1; o < width_lanes; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Non-negative floats order like their bit patterns.
__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
  atomicMax(reinterpret_cast<int*>(addr), __float_as_int(v));
}

// ------------------------------------------------------------------ GEMM scale layout
// Byte offset of scale (row r, column-block kb) in the tensor-core layout:
// 128-row groups of KT atoms of 512 bytes; inside an atom, row 32 j + i (i <
// 32) keeps its 4 consecutive column-block scales at bytes 16 i + 4 j.
__device__ __forceinline__ int64_t sf_gemm_offset(int64_t r, int64_t kb, int64_t kt_atoms) {
  return ((r >> 7) * kt_atoms + (kb >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3);
}

// ------------------------------------------------------------------ mbarrier / TMA / tcgen05
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase of `parity` to complete.  Gives up after
// `limit_ns` (or as soon as *abort is set by another thread of the CTA):
// records LPQ_ERR_TIMEOUT in *err (first writer wins), sets *abort and
// returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort, int* err,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      atomicCAS(err, 0, (int)LPQ_ERR_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned, size multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// TMA tile store shared -> global (bulk-group completion), its commit and the
// waits for the shared-memory reads / the whole stores of this thread's groups.
// The generic-proxy writes of the staged tile are made visible to the async
// proxy first.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               ::"l"(map), "r"(smem_u32(src)), "r"(x), "r"(y) : "memory");
}
// Asynchronous 4-byte copy global -> shared (non-bulk cp.async); `valid`
// false reads nothing and writes zero.  cp_async_arrive_noinc makes the
// mbarrier receive one arrival (counted against its initial count) once all
// of this thread's earlier cp.async copies have landed; the waiter of that
// phase then sees the copied values.
__device__ __forceinline__ void cp_async4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_group_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// tcgen05 ----------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive on `bar` once all earlier tcgen05 operations of this thread finish.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar)) : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address >> 4 in bits 0-13,
// leading byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45, the
// fixed version 1 in 46-47, swizzle mode in 61-63 (2 = 128-byte swizzle,
// 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFFu) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFFu) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7) << 61;
  return d;
}

// D(tmem) (+)= A(smem) * B(smem)^T, kinds without block scales.
template <int kKind>
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  if constexpr (kKind == kKindF16) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
  }
}

// Block-scaled MMA with scale factors in TMEM.
template <int kKind>
__device__ __forceinline__ void mma_bs(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (kKind == kKindMXF8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  } else if constexpr (kKind == kKindMXF4) {  // E2M1, E8M0 scale per 32 values: two per K = 64
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
  }
}

// Copy 32 rows x 16 bytes of scale factors from shared memory into 4 TMEM
// columns, replicated into all four 32-lane quarters.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Store 4 consecutive 32-bit columns into this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
               "r"(d) : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]) : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Store 16 / 32 consecutive 32-bit columns into this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]) : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]) : "memory");
}

// Store N (4, 8, 16 or 32) consecutive 32-bit columns.
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[N]) {
  static_assert(N == 4 || N == 8 || N == 16 || N == 32, "4, 8, 16 or 32 columns");
  if constexpr (N == 4) tmem_st4(taddr, v[0], v[1], v[2], v[3]);
  else if constexpr (N == 8) tmem_st8(taddr, v);
  else if constexpr (N == 16) tmem_st16(taddr, v);
  else tmem_st32(taddr, v);
}

// Load 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}


// ------------------------------------------------------------------ CTA pairs (cta_group::2)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Relaxed remote arrival, for hand-overs of TMEM whose accesses by the
// arriving side are already complete (tcgen05.wait::st / wait::ld), with no
// memory writes to publish.  A release at cluster scope would make the thread
// wait until all of its earlier memory operations (an epilogue's global
// stores, say) are visible cluster-wide; the relaxed form only delivers the
// arrival.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_shared_remote_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// TMA tile load into this CTA's shared memory that signals an mbarrier in
// either CTA of the pair (given as a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(bar_cluster_addr), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Arrive on the mbarrier at the same offset in every CTA of `mask` once this
// thread's earlier pair MMAs have finished.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)), "h"(mask) : "memory");
}
template <int kKind>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  if constexpr (kKind == kKindF16) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
  }
}

}  // namespace lpq
