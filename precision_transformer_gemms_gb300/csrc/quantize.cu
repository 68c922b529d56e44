// Quantizers of liblpq: per-tensor FP8 (current / delayed), MXFP8, NVFP4 (1D
// with optional random Hadamard transform and stochastic rounding; 2D 16x16),
// sub-channel FP8 (1x128, 128x128) and the bf16 transpose.  HBM-bound work:
// each CTA reads a tile of the bf16 input once with 16-byte loads into
// registers and shared memory; the row-wise copy is produced from registers
// (block max by warp shuffles), the column-wise copy from the shared tile.
//
// The arithmetic of every format follows these pages:
//   FP8 E4M3/E5M2, per-tensor scaling, amax history: "Optimizing Transformer
//     models for low-precision training", technical deep dive.
//   NVFP4 (E2M1, E4M3 per 16 values, FP32 tensor scale): "Accelerate LLM
//     training with NVFP4 on Blackwell", technical deep dive.
//   RHT on Wgrad inputs, SR of gradients, 2D weight blocks, the extra amax
//     pass: "How to optimize Transformer-based models for low-precision
//     training", interpreting real-model results.
//   Current / delayed / sub-channel / MXFP8: "Faster training throughput in
//     FP8 with NVIDIA NeMo", advantages and trade-offs.
// Every float operation is an explicit round-to-nearest intrinsic so that no
// multiply-add is contracted.
#include <cuda_fp16.h>
#include <stdio.h>

#include "lpq_device.cuh"

namespace lpq {

namespace {

// QK_MX: MXFP8 (E4M3 codes, or E5M2 with kE5M2); QK_MX4: MXFP4 (packed E2M1).
enum QKind { QK_FP8 = 0, QK_MX = 1, QK_NV = 2, QK_NV2D = 3, QK_BLK1 = 4, QK_BLK128 = 5, QK_BF16 = 6, QK_MX4 = 7 };

struct QParams {
  const uint16_t* x;
  int64_t R, C;
  // row-wise copy [R, C]
  uint8_t* row_codes;
  uint8_t* row_sf;     // u8 block scales (MX, NV)
  float* row_sfinv;    // FP32 block factors (FP8 block)
  float* row_ts;       // tensor scale out
  int row_gemm;        // scale layout
  int64_t row_kt;      // atoms per 128-row group (GEMM layout)
  // column-wise copy [C, R]
  uint8_t* col_codes;
  uint8_t* col_sf;
  float* col_sfinv;
  float* col_ts;
  int col_gemm;
  int64_t col_kt;
  // scaling inputs
  const float* amax_row;       // global amax feeding the row copy (FP8 current, NV)
  const float* amax_col;       // global amax feeding the column copy (NV: RHT amax)
  const float* delayed_scale;  // FP8 delayed
  float* fused_amax0;          // FP8 delayed: amax measured in this pass
  float* fused_amax1;
  // random
  uint64_t seed, ctr_off;
  uint32_t rht_seed;
  int rht, sr;
};

constexpr int kThreads = 256;
constexpr int kTC = 128;

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float tile_val(const uint16_t* tile_row, int c) {
  return __uint_as_float((uint32_t)tile_row[c] << 16);
}

// Block-wide max of non-negative floats; result valid in every thread.
__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max_xor(v, 32);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
  return m;
}

// NVFP4 block scale (E4M3 code) for block max `bmax` and encode scale s_enc.
__device__ __forceinline__ uint32_t nv_block_scale(float bmax, float s_enc) {
  float d = __fmul_rn(div6_rn(bmax), s_enc);
  return cvt_e4m3x2(d, 0.f) & 0xFFu;
}

// Per-CTA table of the encode factors s_enc / dec(S) for the 128 E4M3 codes S
// a block scale can take (0 for S = 0, whose block is all zeros; the NaN code
// is never produced by the saturating conversion): the per-block division
// becomes a shared-memory lookup with the same values.
__device__ __forceinline__ void nv_factor_table(float* tab, float s_enc, int t) {
  if (t >= 0 && t < 128) {
    const float Sd = t < 127 ? e4m3_value((uint32_t)t) : 0.f;
    tab[t] = Sd == 0.f ? 0.f : __fdiv_rn(s_enc, Sd);
  }
}

// E2M1 codes of 8 values y[i] = v[i] * f packed into 32 bits (nibble i = value
// i).  f == 0 marks a block whose scale decoded to 0: all codes +0.
__device__ __forceinline__ uint32_t nv_codes8(const float v[8], float f, bool sr, uint4 w0, uint4 w1) {
  if (f == 0.f) return 0u;
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(v[i], f);
  uint32_t out = 0;
  if (sr) {
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      out |= cvt_e2m1x2(sr_e2m1_value(y[2 * i], w[2 * i]), sr_e2m1_value(y[2 * i + 1], w[2 * i + 1])) << (8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) out |= cvt_e2m1x2(y[2 * i], y[2 * i + 1]) << (8 * i);
  }
  return out;
}

template <bool kE5M2>
__device__ __forceinline__ uint2 fp8_codes8(const float v[8], float s) {
  uint32_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) b[i] = cvt_fp8x2<kE5M2>(__fmul_rn(v[2 * i], s), __fmul_rn(v[2 * i + 1], s));
  return make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}

// Block exponent of the MX kinds for their element format.
template <int KIND, bool kE5M2>
__device__ __forceinline__ int mx_block_exponent(float m) {
  if constexpr (KIND == QK_MX4) return mx_exponent_e2m1(m);
  else if constexpr (kE5M2) return mx_exponent_e5m2(m);
  else return mx_exponent(m);
}

__device__ __forceinline__ float nv_s_enc(const float* amax) {
  float a = *amax;
  return finite_pos(a) ? __fdiv_rn(2688.0f, a) : 1.0f;
}
__device__ __forceinline__ float nv_ts_dec(const float* amax) {
  float a = *amax;
  return finite_pos(a) ? __fdiv_rn(a, 2688.0f) : 1.0f;
}

// NVO (NVFP4 options, compile-time so that the plain paths carry none of the
// registers of the others): bit 0 stochastic rounding, bit 1 RHT of the
// column-wise copy.
template <int KIND, bool kE5M2, int NVO = 0>
__global__ void __launch_bounds__(kThreads, KIND == QK_NV2D ? 5 : (KIND != QK_NV ? 1 : (NVO == 0 ? 6 : (NVO >= 2 ? 4 : 5)))) quant_tile_kernel(const QParams p) {
  constexpr bool kSR = (NVO & 1) != 0, kRHT = (NVO & 2) != 0;
  constexpr int TR = (KIND == QK_BLK1 || KIND == QK_BLK128) ? 128 : 64;
  __shared__ __align__(16) uint16_t tile[TR][kTC];
  __shared__ float red[kThreads / 32];
  __shared__ float part[2][kTC];
  __shared__ float tile_f[32];
  __shared__ uint32_t tile_s[32];
  __shared__ float fb_tab[2][128];  // NVFP4: s_enc / dec(S) for the row and column copies

  const int t = threadIdx.x;
  const int64_t r0 = (int64_t)blockIdx.y * TR, c0 = (int64_t)blockIdx.x * kTC;
  // The shared tile feeds the column-wise copy and the 2D / 128x128 scales.
  const bool kNeedTile = p.col_codes != nullptr || KIND == QK_NV2D || KIND == QK_BLK128;
  const int64_t R = p.R, C = p.C;
  constexpr float kFmax = kE5M2 ? 57344.0f : 448.0f;

  // ---------------------------------------------------------------- scales
  float scale = 1.0f;  // per-tensor FP8
  if constexpr (KIND == QK_FP8) {
    if (p.delayed_scale) {
      scale = *p.delayed_scale;
    } else {
      float a = *p.amax_row;
      scale = finite_pos(a) ? __fdiv_rn(kFmax, a) : 1.0f;
    }
    if (blockIdx.x == 0 && blockIdx.y == 0 && t == 0) {
      float sinv = __fdiv_rn(1.0f, scale);
      if (p.row_ts) *p.row_ts = sinv;
      if (p.col_ts) *p.col_ts = sinv;
    }
  }
  float s_enc_row = 1.f, s_enc_col = 1.f;
  float sgn[16];
  if constexpr (KIND == QK_NV || KIND == QK_NV2D) {
    if (p.row_codes) s_enc_row = nv_s_enc(p.amax_row);
    if (p.col_codes) s_enc_col = nv_s_enc(p.amax_col);
    if (blockIdx.x == 0 && blockIdx.y == 0 && t == 0) {
      if (p.row_ts) *p.row_ts = nv_ts_dec(p.amax_row);
      if (p.col_ts) *p.col_ts = nv_ts_dec(p.amax_col);
    }
    if constexpr (kRHT) rht_sign_factors(rht_signs(p.rht_seed), sgn);
    nv_factor_table(fb_tab[0], s_enc_row, t);
    nv_factor_table(fb_tab[1], s_enc_col, t - 128);
    __syncthreads();
  }
  const PhiloxKeys keys(kSR ? p.seed : 0);  // dead (and free) without stochastic rounding

  // ---------------------------------------------------------------- load (+ row-wise copy)
  const int lr = t >> 4;        // row within a 16-row slab
  const int lc = (t & 15) * 8;  // first of this thread's 8 columns
  const bool col_ok = c0 + lc < C;
  float local_amax = 0.f;
  // all of this thread's 16-byte loads first, so they are in flight together
  uint4 vbuf[TR / 16];
  if constexpr (KIND == QK_NV) {
    // NVFP4 1D: one thread per 16-value block (8 threads per 128-column row,
    // 32 rows a pass), so each block's scale is computed once, without a
    // shuffle, and the stochastic-rounding words come from four independent
    // Philox blocks.
    const int wr = t >> 3, wc = (t & 7) * 16;
    const bool wcol_ok = c0 + wc < C;  // C is a multiple of 16: whole blocks
#pragma unroll
    for (int it = 0; it < TR / 32; ++it) {
      const int64_t r = r0 + it * 32 + wr;
      const bool ok = wcol_ok && r < R;
      const uint16_t* src = p.x + r * C + c0 + wc;
      vbuf[2 * it] = ok ? ld_stream(src) : make_uint4(0u, 0u, 0u, 0u);
      vbuf[2 * it + 1] = ok ? ld_stream(src + 8) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int it = 0; it < TR / 32; ++it) {
      const int rl = it * 32 + wr;
      const int64_t r = r0 + rl;
      const bool ok = wcol_ok && r < R;
      if (kNeedTile) {
        *reinterpret_cast<uint4*>(&tile[rl][wc]) = vbuf[2 * it];
        *reinterpret_cast<uint4*>(&tile[rl][wc + 8]) = vbuf[2 * it + 1];
      }
      if (!p.row_codes) continue;
      float f[16];
      unpack8(vbuf[2 * it], f);
      unpack8(vbuf[2 * it + 1], f + 8);
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) m = absmax_acc(m, f[i]);
      const uint32_t S = nv_block_scale(m, s_enc_row);
      const float fb = fb_tab[0][S];
      uint4 w[4] = {uint4{}, uint4{}, uint4{}, uint4{}};
      if constexpr (kSR) {
        const uint64_t g = (p.ctr_off + (uint64_t)(r * C + c0 + wc)) >> 2;
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = keys.words(g + j, 0u);
      }
      const uint32_t q0 = nv_codes8(f, fb, kSR, w[0], w[1]);
      const uint32_t q1 = nv_codes8(f + 8, fb, kSR, w[2], w[3]);
      if (ok) {
        *reinterpret_cast<uint2*>(p.row_codes + r * (C >> 1) + ((c0 + wc) >> 1)) = make_uint2(q0, q1);
        const int64_t kb = (c0 + wc) >> 4;
        const int64_t off = p.row_gemm ? sf_gemm_offset(r, kb, p.row_kt) : r * (C >> 4) + kb;
        p.row_sf[off] = (uint8_t)S;
      }
    }
  } else {
#pragma unroll
  for (int it = 0; it < TR / 16; ++it) {
    const int64_t r = r0 + it * 16 + lr;
    vbuf[it] = (col_ok && r < R) ? ld_stream(p.x + r * C + c0 + lc) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int it = 0; it < TR / 16; ++it) {
    const int rl = it * 16 + lr;
    const int64_t r = r0 + rl;
    const bool ok = col_ok && r < R;
    const uint4 v = vbuf[it];
    if (kNeedTile) *reinterpret_cast<uint4*>(&tile[rl][lc]) = v;
    float f[8];
    unpack8(v, f);
    if constexpr (KIND == QK_BLK128 || KIND == QK_FP8) {
#pragma unroll
      for (int i = 0; i < 8; ++i) local_amax = absmax_acc(local_amax, f[i]);
    }
    if (!p.row_codes) continue;
    if constexpr (KIND == QK_FP8) {
      uint2 q = fp8_codes8<kE5M2>(f, scale);
      if (ok) *reinterpret_cast<uint2*>(p.row_codes + r * C + c0 + lc) = q;
    } else if constexpr (KIND == QK_MX || KIND == QK_MX4) {
      // 32-value block = 4 neighbouring threads of the row
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = absmax_acc(m, f[i]);
      m = warp_max_xor(m, 4);
      const int e = mx_block_exponent<KIND, kE5M2>(m);
      const float mult = pow2_exact(-e);
      if (ok) {
        if constexpr (KIND == QK_MX4)
          *reinterpret_cast<uint32_t*>(p.row_codes + r * (C >> 1) + ((c0 + lc) >> 1)) =
              nv_codes8(f, mult, false, uint4{}, uint4{});
        else
          *reinterpret_cast<uint2*>(p.row_codes + r * C + c0 + lc) = fp8_codes8<kE5M2>(f, mult);
        if ((t & 3) == 0) {
          const int64_t kb = (c0 + lc) >> 5;
          const int64_t off = p.row_gemm ? sf_gemm_offset(r, kb, p.row_kt) : r * (C >> 5) + kb;
          p.row_sf[off] = (uint8_t)(e + 127);
        }
      }
    } else if constexpr (KIND == QK_BLK1) {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) m = absmax_acc(m, f[i]);
      m = warp_max_xor(m, 16);
      const float s = finite_pos(m) ? __fdiv_rn(448.0f, m) : 1.0f;
      uint2 q = fp8_codes8<false>(f, s);
      if (ok) {
        *reinterpret_cast<uint2*>(p.row_codes + r * C + c0 + lc) = q;
        if ((t & 15) == 0) {
          const int64_t kb = c0 >> 7;
          const int64_t off = p.row_gemm ? kb * R + r : r * (C >> 7) + kb;
          p.row_sfinv[off] = __fdiv_rn(1.0f, s);
        }
      }
    } else if constexpr (KIND == QK_BF16) {
      if (ok) *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.row_codes) + r * C + c0 + lc) = v;
    }
  }

  }  // load + row-wise copy, other kinds
  if constexpr (KIND == QK_FP8) {
    if (p.fused_amax0) {  // delayed scaling: amax measured in this pass
      float m = block_max(local_amax, red);
      if (t == 0) {
        atomic_max_nonneg(p.fused_amax0, m);
        if (p.fused_amax1) atomic_max_nonneg(p.fused_amax1, m);
      }
    }
  }
  if (!kNeedTile) return;
  __syncthreads();

  // ---------------------------------------------------------------- 2D / 128x128 tiles
  if constexpr (KIND == QK_NV2D) {
    {
      const int tid = t >> 3, sub = t & 7;  // 32 tiles of 16x16, 8 threads each
      const int tr = tid >> 3, tc = tid & 7;
      float m = 0.f;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // 16-byte shared loads of 8 values
          float f[8];
          unpack8(*reinterpret_cast<const uint4*>(&tile[tr * 16 + sub * 2 + rr][tc * 16 + 8 * h]), f);
#pragma unroll
          for (int i = 0; i < 8; ++i) m = absmax_acc(m, f[i]);
        }
      m = warp_max_xor(m, 8);
      if (sub == 0) {
        const float s_enc = p.row_codes ? s_enc_row : s_enc_col;
        const uint32_t S = nv_block_scale(m, s_enc);
        tile_s[tid] = S;
        tile_f[tid] = fb_tab[p.row_codes ? 0 : 1][S];
      }
    }
    __syncthreads();
    if (p.row_codes) {
#pragma unroll
      for (int it = 0; it < TR / 16; ++it) {
        const int rl = it * 16 + lr;
        const int64_t r = r0 + rl;
        if (!(col_ok && r < R)) continue;
        const int tid = (rl >> 4) * 8 + (lc >> 4);
        float f[8];
        unpack8(vbuf[it], f);  // this thread's own loaded values of the row
        const uint32_t q = nv_codes8(f, tile_f[tid], false, uint4{}, uint4{});
        *reinterpret_cast<uint32_t*>(p.row_codes + r * (C >> 1) + ((c0 + lc) >> 1)) = q;
        if ((t & 1) == 0) {
          const int64_t kb = (c0 + lc) >> 4;
          const int64_t off = p.row_gemm ? sf_gemm_offset(r, kb, p.row_kt) : r * (C >> 4) + kb;
          p.row_sf[off] = (uint8_t)tile_s[tid];
        }
      }
    }
    if (p.col_codes) {
      // Two adjacent columns per thread, one 16-row block: each 4-byte shared
      // load gives a row's values of both columns (both in the same 16x16 tile).
      const int cp = t & 63, rq = t >> 6;
      const int cl = 2 * cp;
      const int64_t c = c0 + cl, rr = r0 + rq * 16;
      if (c < C && rr < R) {
        const int tid = rq * 8 + (cl >> 4);
        float f0[16], f1[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t w = *reinterpret_cast<const uint32_t*>(&tile[rq * 16 + i][cl]);
          f0[i] = bf16_lo(w);
          f1[i] = bf16_hi(w);
        }
        const float fb = tile_f[tid];
        const int64_t kb = rr >> 4;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t cc = c + h;
          if (cc >= C) break;
          const float* v = h ? f1 : f0;
          const uint32_t a = nv_codes8(v, fb, false, uint4{}, uint4{});
          const uint32_t b = nv_codes8(v + 8, fb, false, uint4{}, uint4{});
          *reinterpret_cast<uint2*>(p.col_codes + cc * (R >> 1) + (rr >> 1)) = make_uint2(a, b);
          const int64_t off = p.col_gemm ? sf_gemm_offset(cc, kb, p.col_kt) : cc * (R >> 4) + kb;
          p.col_sf[off] = (uint8_t)tile_s[tid];
        }
      }
    }
    return;
  }

  if constexpr (KIND == QK_BLK128) {
    const float m = block_max(local_amax, red);
    const float s = finite_pos(m) ? __fdiv_rn(448.0f, m) : 1.0f;
    const float sinv = __fdiv_rn(1.0f, s);
    const int64_t nrb = (R + 127) >> 7, ncb = C >> 7;
    if (t == 0) {
      if (p.row_codes) p.row_sfinv[(r0 >> 7) * ncb + (c0 >> 7)] = sinv;
      if (p.col_codes) p.col_sfinv[(c0 >> 7) * nrb + (r0 >> 7)] = sinv;
    }
    if (p.row_codes) {
#pragma unroll
      for (int it = 0; it < TR / 16; ++it) {
        const int rl = it * 16 + lr;
        const int64_t r = r0 + rl;
        if (!(col_ok && r < R)) continue;
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = tile_val(tile[rl], lc + i);
        *reinterpret_cast<uint2*>(p.row_codes + r * C + c0 + lc) = fp8_codes8<false>(f, s);
      }
    }
    if (p.col_codes) {
      const int cl = t & 127, rh = t >> 7;
      const int64_t c = c0 + cl, rbase = r0 + rh * 64;
      if (c < C && rbase < R) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float f[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) f[i] = tile_val(tile[rh * 64 + q4 * 16 + i], cl);
          uint2 a = fp8_codes8<false>(f, s), b = fp8_codes8<false>(f + 8, s);
          *reinterpret_cast<uint4*>(p.col_codes + c * R + rbase + q4 * 16) = make_uint4(a.x, a.y, b.x, b.y);
        }
      }
    }
    return;
  }

  if constexpr (KIND == QK_BLK1) {
    if (!p.col_codes) return;
    const int cl = t & 127, rh = t >> 7;
    const int64_t c = c0 + cl, rbase = r0 + rh * 64;
    float m = 0.f;
#pragma unroll 16
    for (int i = 0; i < 64; ++i) m = absmax_acc(m, tile_val(tile[rh * 64 + i], cl));
    part[rh][cl] = m;
    __syncthreads();
    m = fmaxf(part[0][cl], part[1][cl]);
    const float s = finite_pos(m) ? __fdiv_rn(448.0f, m) : 1.0f;
    if (c < C && rbase < R) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float f[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = tile_val(tile[rh * 64 + q4 * 16 + i], cl);
        uint2 a = fp8_codes8<false>(f, s), b = fp8_codes8<false>(f + 8, s);
        *reinterpret_cast<uint4*>(p.col_codes + c * R + rbase + q4 * 16) = make_uint4(a.x, a.y, b.x, b.y);
      }
      if (rh == 0) {
        const int64_t kb = r0 >> 7;
        const int64_t off = p.col_gemm ? kb * C + c : c * (R >> 7) + kb;
        p.col_sfinv[off] = __fdiv_rn(1.0f, s);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- column-wise copy
  if (!p.col_codes) return;
  const int cl = t & 127, rh = t >> 7;
  const int64_t c = c0 + cl, rbase = r0 + rh * 32;
  if (c >= C || rbase >= R) return;
  const int nvalid = (R - rbase) >= 32 ? 32 : 16;  // R is a multiple of 16 here
  if constexpr (KIND == QK_MX4) {
    // R is a multiple of 32 here: the thread's 32 rows are one whole block.
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = tile_val(tile[rh * 32 + i], cl);
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = absmax_acc(m, f[i]);
    const int e = mx_exponent_e2m1(m);
    const float s = pow2_exact(-e);
    uint32_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = nv_codes8(f + 8 * j, s, false, uint4{}, uint4{});
    *reinterpret_cast<uint4*>(p.col_codes + c * (R >> 1) + (rbase >> 1)) = make_uint4(q[0], q[1], q[2], q[3]);
    const int64_t kb = rbase >> 5;
    const int64_t off = p.col_gemm ? sf_gemm_offset(c, kb, p.col_kt) : c * (R >> 5) + kb;
    p.col_sf[off] = (uint8_t)(e + 127);
  } else if constexpr (KIND == QK_FP8 || KIND == QK_MX) {
    float f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) f[i] = tile_val(tile[rh * 32 + i], cl);
    float s = scale;
    int e = 0;
    if constexpr (KIND == QK_MX) {
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) m = absmax_acc(m, f[i]);
      e = mx_block_exponent<KIND, kE5M2>(m);
      s = pow2_exact(-e);
    }
    uint2 q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) q[j] = fp8_codes8<kE5M2>(f + 8 * j, s);
    uint8_t* dst = p.col_codes + c * R + rbase;
    *reinterpret_cast<uint4*>(dst) = make_uint4(q[0].x, q[0].y, q[1].x, q[1].y);
    if (nvalid == 32) *reinterpret_cast<uint4*>(dst + 16) = make_uint4(q[2].x, q[2].y, q[3].x, q[3].y);
    if constexpr (KIND == QK_MX) {
      const int64_t kb = rbase >> 5;
      const int64_t off = p.col_gemm ? sf_gemm_offset(c, kb, p.col_kt) : c * (R >> 5) + kb;
      p.col_sf[off] = (uint8_t)(e + 127);
    }
  } else if constexpr (KIND == QK_NV) {
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      if (hb * 16 >= nvalid) break;
      float f[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) f[i] = tile_val(tile[rh * 32 + hb * 16 + i], cl);
      if constexpr (kRHT) rht16(f, sgn);
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) m = absmax_acc(m, f[i]);
      const uint32_t S = nv_block_scale(m, s_enc_col);
      const float fb = fb_tab[1][S];
      const int64_t rr = rbase + hb * 16;
      uint4 w[4] = {uint4{}, uint4{}, uint4{}, uint4{}};
      if constexpr (kSR) {
        const uint64_t g = (p.ctr_off + (uint64_t)(c * R + rr)) >> 2;
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = keys.words(g + j, 1u);
      }
      const uint32_t a = nv_codes8(f, fb, kSR, w[0], w[1]);
      const uint32_t b = nv_codes8(f + 8, fb, kSR, w[2], w[3]);
      *reinterpret_cast<uint2*>(p.col_codes + c * (R >> 1) + (rr >> 1)) = make_uint2(a, b);
      const int64_t kb = rr >> 4;
      const int64_t off = p.col_gemm ? sf_gemm_offset(c, kb, p.col_kt) : c * (R >> 4) + kb;
      p.col_sf[off] = (uint8_t)S;
    }
  } else if constexpr (KIND == QK_BF16) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      w[i] = (uint32_t)tile[rh * 32 + 2 * i][cl] | ((uint32_t)tile[rh * 32 + 2 * i + 1][cl] << 16);
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.col_codes) + c * R + rbase;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j * 8 < nvalid) *reinterpret_cast<uint4*>(dst + 8 * j) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

// ---------------------------------------------------------------- amax pass
// max |x| over the tensor into up to two targets, and (kRHT) the max |RHT(x)|
// over the column-wise copy (16-runs along rows of each column) into rht_out.
template <bool kRHT>
__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                        float* out0, float* out1, float* rht_out,
                                                        uint32_t rht_seed) {
  __shared__ float red[kThreads / 32];
  __shared__ float red2[kThreads / 32];
  float m = 0.f, mh = 0.f;
  const int64_t chunks = C >> 3;  // 8 columns per 16-byte vector
  if constexpr (!kRHT) {
    const int64_t n = R * chunks;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n; i += (int64_t)gridDim.x * kThreads) {
      uint4 v = ld_stream(x + i * 8);
      float f[8];
      unpack8(v, f);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = absmax_acc(m, f[j]);
    }
  } else {
    float sgn[16];
    rht_sign_factors(rht_signs(rht_seed), sgn);
    const int64_t n = (R >> 4) * chunks;  // units of 16 rows x 8 columns
    for (int64_t u = (int64_t)blockIdx.x * kThreads + threadIdx.x; u < n; u += (int64_t)gridDim.x * kThreads) {
      const int64_t rg = u / chunks, cc = u - rg * chunks;
      uint4 v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = ld_stream(x + (rg * 16 + i) * C + cc * 8);
#pragma unroll
      for (int col = 0; col < 8; ++col) {
        float t[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t w = (&v[i].x)[col >> 1];
          t[i] = (col & 1) ? bf16_hi(w) : bf16_lo(w);
          m = absmax_acc(m, t[i]);
        }
        rht16(t, sgn);
#pragma unroll
        for (int i = 0; i < 16; ++i) mh = absmax_acc(mh, t[i]);
      }
    }
  }
  m = warp_max_xor(m, 32);
  mh = warp_max_xor(mh, 32);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) { red[w] = m; red2[w] = mh; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f, b = 0.f;
    for (int i = 0; i < kThreads / 32; ++i) { a = fmaxf(a, red[i]); b = fmaxf(b, red2[i]); }
    if (out0) atomic_max_nonneg(out0, a);
    if (out1) atomic_max_nonneg(out1, a);
    if (kRHT && rht_out) atomic_max_nonneg(rht_out, b);
  }
}

// ---------------------------------------------------------------- tensor scales of an empty shard
// With a given amax and nothing to quantize, the copies' FP32 tensor scales
// still follow from it: 1 / (fmax / amax) for per-tensor FP8, amax / 2688 for
// NVFP4 (1 when the amax is 0 or not finite).
__global__ void given_amax_scales_kernel(int nvfp4, float fmax, const float* amax_row, const float* amax_col,
                                         float* ts_row, float* ts_col) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  const float* am[2] = {amax_row, amax_col};
  float* ts[2] = {ts_row, ts_col};
  for (int i = 0; i < 2; ++i) {
    if (!ts[i] || !am[i]) continue;
    const float a = *am[i];
    if (nvfp4) {
      *ts[i] = finite_pos(a) ? __fdiv_rn(a, 2688.0f) : 1.0f;
    } else {
      const float scale = finite_pos(a) ? __fdiv_rn(fmax, a) : 1.0f;
      *ts[i] = __fdiv_rn(1.0f, scale);
    }
  }
}

// ---------------------------------------------------------------- delayed-scaling update
__global__ void scale_update_kernel(float* hist, int32_t* pos, float* scale, float* scale_inv, int32_t len,
                                    const float* amax, float fmax) {
  __shared__ float red[32];
  __shared__ int32_t slot;
  const int t = threadIdx.x;
  if (t == 0) {
    slot = *pos;
    hist[slot] = *amax;
    *pos = (slot + 1) % len;
  }
  __syncthreads();
  float m = 0.f;
  for (int i = t; i < len; i += blockDim.x) m = fmaxf(m, hist[i]);
  m = warp_max_xor(m, 32);
  if ((t & 31) == 0) red[t >> 5] = m;
  __syncthreads();
  if (t == 0) {
    float mm = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) mm = fmaxf(mm, red[i]);
    float s = *scale;
    if (finite_pos(mm)) s = __fdiv_rn(fmax, mm);
    *scale = s;
    *scale_inv = __fdiv_rn(1.0f, s);
  }
}

int g_num_sms = 0;

int num_sms() {
  if (g_num_sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (g_num_sms <= 0) g_num_sms = 148;
  }
  return g_num_sms;
}

template <int KIND, bool kE5M2, int NVO = 0>
lpq_status run_tile(const QParams& p, cudaStream_t s) {
  constexpr int TR = (KIND == QK_BLK1 || KIND == QK_BLK128) ? 128 : 64;
  dim3 grid((unsigned)((p.C + kTC - 1) / kTC), (unsigned)((p.R + TR - 1) / TR));
  if (grid.y > 65535u) return set_error(LPQ_ERR_SHAPE, "too many rows (%lld) for one launch", (long long)p.R);
  quant_tile_kernel<KIND, kE5M2, NVO><<<grid, kThreads, 0, s>>>(p);
  return cuda_check(cudaGetLastError(), "quantize kernel launch");
}

lpq_status run_amax(const uint16_t* x, int64_t R, int64_t C, float* o0, float* o1, float* rht_out,
                    uint32_t rht_seed, cudaStream_t s) {
  const int64_t units = rht_out ? (R / 16) * (C / 8) : R * (C / 8);
  int64_t blocks = (units + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (rht_out)
    amax_kernel<true><<<(unsigned)blocks, kThreads, 0, s>>>(x, R, C, o0, o1, rht_out, rht_seed);
  else
    amax_kernel<false><<<(unsigned)blocks, kThreads, 0, s>>>(x, R, C, o0, o1, nullptr, 0);
  return cuda_check(cudaGetLastError(), "amax kernel launch");
}

lpq_status zero_f32(float* p, cudaStream_t s) {
  if (!p) return LPQ_OK;
  return cuda_check(cudaMemsetAsync(p, 0, sizeof(float), s), "cudaMemsetAsync(amax)");
}

}  // namespace

lpq_status launch_quantize(const void* xv, int64_t R, int64_t C, int32_t fmt, int32_t scaling, uint32_t flags,
                           uint64_t seed, uint64_t counter_offset, uint32_t rht_seed,
                           const lpq_delayed_state* state, lpq_qtensor* out, cudaStream_t s) {
  const bool do_row = flags & LPQ_ROWWISE, do_col = flags & LPQ_COLWISE;
  const bool given = flags & LPQ_GIVEN_AMAX;  // the views' amax fields are inputs
  lpq_qview* rv = do_row ? &out->row : nullptr;
  lpq_qview* cv = do_col ? &out->col : nullptr;
  const bool mx = fmt == LPQ_MXFP8 || fmt == LPQ_MXFP8_E5M2 || fmt == LPQ_MXFP4;
  const bool u8_scaled = mx || fmt == LPQ_NVFP4 || fmt == LPQ_NVFP4_2D;  // tensor-core scale layout possible
  QParams p{};
  p.x = static_cast<const uint16_t*>(xv);
  p.R = R;
  p.C = C;
  if (rv) {
    p.row_codes = static_cast<uint8_t*>(rv->codes);
    p.row_sf = static_cast<uint8_t*>(rv->scales);
    p.row_sfinv = static_cast<float*>(rv->scales);
    p.row_ts = rv->tensor_scale;
    p.row_gemm = rv->sf_layout == LPQ_SF_GEMM;
    if (u8_scaled) p.row_kt = sf_kt_atoms(fmt, C);
  }
  if (cv) {
    p.col_codes = static_cast<uint8_t*>(cv->codes);
    p.col_sf = static_cast<uint8_t*>(cv->scales);
    p.col_sfinv = static_cast<float*>(cv->scales);
    p.col_ts = cv->tensor_scale;
    p.col_gemm = cv->sf_layout == LPQ_SF_GEMM;
    if (u8_scaled) p.col_kt = sf_kt_atoms(fmt, R);
  }
  p.seed = seed;
  p.ctr_off = counter_offset;
  p.rht_seed = rht_seed;
  p.rht = (fmt == LPQ_NVFP4) && (flags & LPQ_RHT_COLWISE) && do_col;
  p.sr = (fmt == LPQ_NVFP4) && (flags & LPQ_STOCHASTIC);

  // Zero padding of tensor-core scale layouts so that partial atoms read as 0.
  auto zero_pad = [&](lpq_qview* v) -> lpq_status {
    if (!v || v->sf_layout != LPQ_SF_GEMM) return LPQ_OK;
    if (!u8_scaled) return LPQ_OK;
    const int64_t blk = mx ? 32 : 16;
    const int64_t kt = sf_kt_atoms(fmt, v->cols);
    if (v->rows % 128 == 0 && (v->cols / blk) == kt * 4) return LPQ_OK;
    size_t bytes = (size_t)sf_row_groups(v->rows) * (size_t)kt * 512;
    return cuda_check(cudaMemsetAsync(v->scales, 0, bytes, s), "cudaMemsetAsync(scale padding)");
  };
  lpq_status st;
  if ((st = zero_pad(rv)) != LPQ_OK) return st;
  if ((st = zero_pad(cv)) != LPQ_OK) return st;

  if (R == 0 || C == 0) {
    // Nothing to quantize; scalar outputs take their empty-tensor values.
    if (given) {
      const bool nv = fmt == LPQ_NVFP4 || fmt == LPQ_NVFP4_2D;
      const float* a_row = rv ? rv->amax : nullptr;
      const float* a_col = cv ? cv->amax : nullptr;
      if (!nv && !a_row) a_row = a_col;  // FP8: one amax for both copies
      if (!nv && !a_col) a_col = a_row;
      given_amax_scales_kernel<<<1, 32, 0, s>>>(nv ? 1 : 0, fmt == LPQ_FP8_E5M2 ? 57344.0f : 448.0f, a_row, a_col,
                                                rv ? rv->tensor_scale : nullptr, cv ? cv->tensor_scale : nullptr);
      return cuda_check(cudaGetLastError(), "tensor scales from the given amax");
    }
    if (fmt == LPQ_FP8_E4M3 || fmt == LPQ_FP8_E5M2 || fmt == LPQ_NVFP4 || fmt == LPQ_NVFP4_2D) {
      for (lpq_qview* v : {rv, cv}) {
        if (!v) continue;
        if (v->amax && (st = zero_f32(v->amax, s)) != LPQ_OK) return st;
      }
      if (fmt == LPQ_NVFP4 || fmt == LPQ_NVFP4_2D || scaling == LPQ_SCALING_CURRENT) {
        // tensor scale 1 (amax 0 gives scale 1); written by a 1x1 launch of the tile kernel is
        // unnecessary: copy a host constant.
        static const float one = 1.0f;
        for (lpq_qview* v : {rv, cv})
          if (v && v->tensor_scale &&
              (st = cuda_check(cudaMemcpyAsync(v->tensor_scale, &one, sizeof(float), cudaMemcpyHostToDevice, s),
                               "cudaMemcpyAsync(tensor scale)")) != LPQ_OK)
            return st;
      } else if (state) {
        for (lpq_qview* v : {rv, cv})
          if (v && v->tensor_scale &&
              (st = cuda_check(cudaMemcpyAsync(v->tensor_scale, state->scale_inv, sizeof(float),
                                               cudaMemcpyDeviceToDevice, s), "cudaMemcpyAsync(scale_inv)")) != LPQ_OK)
            return st;
      }
    }
    return LPQ_OK;
  }

  switch (fmt) {
    case LPQ_FP8_E4M3:
    case LPQ_FP8_E5M2: {
      const bool e5 = fmt == LPQ_FP8_E5M2;
      float* a0 = rv ? rv->amax : cv->amax;
      float* a1 = (rv && cv) ? cv->amax : nullptr;
      if (given) {  // current scaling with the amax the caller measured (e.g. over all shards)
        p.amax_row = a0;
        return e5 ? run_tile<QK_FP8, true>(p, s) : run_tile<QK_FP8, false>(p, s);
      }
      if ((st = zero_f32(a0, s)) != LPQ_OK || (st = zero_f32(a1, s)) != LPQ_OK) return st;
      if (scaling == LPQ_SCALING_DELAYED) {
        p.delayed_scale = state->scale;
        p.fused_amax0 = a0;
        p.fused_amax1 = a1;
      } else {
        if ((st = run_amax(p.x, R, C, a0, a1, nullptr, 0, s)) != LPQ_OK) return st;
        p.amax_row = a0;
      }
      return e5 ? run_tile<QK_FP8, true>(p, s) : run_tile<QK_FP8, false>(p, s);
    }
    case LPQ_MXFP8:
    case LPQ_MXFP8_E5M2:
    case LPQ_MXFP4:
      if (rv && rv->amax) {  // optional amax output
        if ((st = zero_f32(rv->amax, s)) != LPQ_OK) return st;
        if ((st = run_amax(p.x, R, C, rv->amax, cv ? cv->amax : nullptr, nullptr, 0, s)) != LPQ_OK) return st;
      }
      if (fmt == LPQ_MXFP4) return run_tile<QK_MX4, false>(p, s);
      return fmt == LPQ_MXFP8_E5M2 ? run_tile<QK_MX, true>(p, s) : run_tile<QK_MX, false>(p, s);
    case LPQ_NVFP4:
    case LPQ_NVFP4_2D: {
      const bool rht = p.rht;
      float* raw0 = rv ? rv->amax : (rht ? nullptr : cv->amax);
      float* raw1 = (rv && cv && !rht) ? cv->amax : nullptr;
      float* rh = rht ? cv->amax : nullptr;
      if (!given) {
        if ((st = zero_f32(raw0, s)) != LPQ_OK || (st = zero_f32(raw1, s)) != LPQ_OK ||
            (st = zero_f32(rh, s)) != LPQ_OK)
          return st;
        if ((st = run_amax(p.x, R, C, raw0, raw1, rh, rht_seed, s)) != LPQ_OK) return st;
      }
      p.amax_row = rv ? rv->amax : nullptr;
      p.amax_col = cv ? cv->amax : nullptr;
      if (fmt == LPQ_NVFP4_2D) return run_tile<QK_NV2D, false>(p, s);
      switch ((p.sr ? 1 : 0) | (p.rht ? 2 : 0)) {
        case 0: return run_tile<QK_NV, false, 0>(p, s);
        case 1: return run_tile<QK_NV, false, 1>(p, s);
        case 2: return run_tile<QK_NV, false, 2>(p, s);
        default: return run_tile<QK_NV, false, 3>(p, s);
      }
    }
    case LPQ_FP8_BLOCK_1x128:
      return run_tile<QK_BLK1, false>(p, s);
    case LPQ_FP8_BLOCK_128x128:
      return run_tile<QK_BLK128, false>(p, s);
    case LPQ_BF16:
      return run_tile<QK_BF16, false>(p, s);
  }
  return set_error(LPQ_ERR_UNSUPPORTED, "format %d", fmt);
}

lpq_status launch_scale_update(const lpq_delayed_state* st, const float* amax, float fmax, cudaStream_t s) {
  scale_update_kernel<<<1, 128, 0, s>>>(st->amax_history, st->pos, st->scale, st->scale_inv, st->len, amax, fmax);
  return cuda_check(cudaGetLastError(), "scale update launch");
}

}  // namespace lpq
