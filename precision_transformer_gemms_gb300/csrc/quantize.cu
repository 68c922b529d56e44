// Quantizers of liblpq: per-tensor FP8 (current / delayed), MXFP8, NVFP4 (1D
// with optional random Hadamard transform and stochastic rounding; 2D 16x16),
// sub-channel FP8 (1x128, 128x128) and the bf16 transpose.  HBM-bound work:
// each CTA reads a tile of the bf16 input once with 16-byte loads into
// registers and shared memory; the row-wise copy is produced from registers
// (block max by warp shuffles), the column-wise copy from the shared tile.
// The 2D NVFP4 kernel needs no shared tile: its 16x16 maxima come from warp
// shuffles and its column copy is a register transpose of the row codes.
// Column-wise NVFP4 codes leave as whole 32-byte column segments staged in
// shared memory.
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
#include <algorithm>
#include <stdio.h>

#include "lpq_device.cuh"

namespace lpq {

namespace {

// QK_MX: MXFP8 (E4M3 codes, or E5M2 with kE5M2); QK_MX4: MXFP4 (packed E2M1).
// NVFP4 with 16x16 tiles has a kernel of its own (nv2d_kernel).
enum QKind { QK_FP8 = 0, QK_MX = 1, QK_NV = 2, QK_BLK1 = 4, QK_BLK128 = 5, QK_BF16 = 6, QK_MX4 = 7 };

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

// fmax / amax-style scale quotient, clamped to the largest finite float when
// it overflows (an amax below about fmax / 3.4e38): an infinite scale would
// turn zero elements into NaN codes and 1 / scale into 0.
__device__ __forceinline__ float scale_quotient(float fmax, float a) {
  return fminf(__fdiv_rn(fmax, a), 3.40282347e38f);
}

// NVFP4 block scale (E4M3 code) for block max `bmax` and encode scale s_enc.
__device__ __forceinline__ uint32_t nv_block_scale(float bmax, float s_enc) {
  float d = __fmul_rn(div6_rn(bmax), s_enc);
  return cvt_e4m3x2(d, 0.f) & 0xFFu;
}

// Per-CTA table of the encode factors s_enc / dec(S) for the 128 E4M3 codes S
// a block scale can take (0 for S = 0, whose block is all zeros; the NaN code
// is never produced by the saturating conversion; clamped to the largest
// finite float like every scale quotient): the per-block division becomes a
// shared-memory lookup with the same values.
__device__ __forceinline__ void nv_factor_table(float* tab, float s_enc, int t) {
  if (t >= 0 && t < 128) {
    const float Sd = t < 127 ? e4m3_value((uint32_t)t) : 0.f;
    tab[t] = Sd == 0.f ? 0.f : scale_quotient(s_enc, Sd);
  }
}

// E2M1 codes of 8 values y[i] = v[i] * f packed into 32 bits (nibble i = value
// i).  f == 0 marks a block whose scale decoded to 0: all codes +0.
__device__ __forceinline__ uint32_t nv_codes8(const float v[8], float f, bool sr, uint4 w0, uint4 w1) {
  if (f == 0.f) return 0u;
  float y[8];
  if (sr) {  // y = v * f and the rounding two values at a time (packed two-wide operations)
    const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 yy = __fmul2_rn(make_float2(v[2 * i], v[2 * i + 1]), make_float2(f, f));
      const float2 r = sr_e2m1_value2(yy, w[2 * i], w[2 * i + 1]);
      y[2 * i] = r.x;
      y[2 * i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // y = v * f two at a time (packed), RNE encode
      const float2 yy = __fmul2_rn(make_float2(v[2 * i], v[2 * i + 1]), make_float2(f, f));
      y[2 * i] = yy.x;
      y[2 * i + 1] = yy.y;
    }
  }
  return cvt_e2m1x8(y);
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
  return finite_pos(a) ? scale_quotient(2688.0f, a) : 1.0f;
}
__device__ __forceinline__ float nv_ts_dec(const float* amax) {
  float a = *amax;
  return finite_pos(a) ? __fdiv_rn(a, 2688.0f) : 1.0f;
}

// Column-wise NVFP4 copy of a 64 x 128 tile staged in shared memory (column
// cl: 32 code bytes for the tile's 64 rows at col_stage + 32 cl, 4 block
// scales at sf_stage + 4 cl): each column's codes leave as two 16-byte
// stores (8-byte pieces when R % 32 != 0 or at a 16-row tail) and its scales
// as one 4-byte store where the layout allows.  R and C are multiples of 16.
__device__ __forceinline__ void store_col_staged(const QParams& p, const uint8_t* col_stage, const uint8_t* sf_stage,
                                                 int64_t c_first, int64_t rt, int t) {
  const int64_t R = p.R, C = p.C;
  {
    const int cl = t >> 1, h = t & 1;  // column, 32-row half
    const int64_t c = c_first + cl, rr = rt + 32 * h;
    if (c < C && rr < R) {
      uint8_t* dst = p.col_codes + c * (R >> 1) + (rr >> 1);
      const uint4 v16 = *reinterpret_cast<const uint4*>(col_stage + cl * 32 + 16 * h);
      if (rr + 32 <= R && (R & 31) == 0) {
        *reinterpret_cast<uint4*>(dst) = v16;  // 16-byte aligned: R / 2 and rr / 2 are multiples of 16
      } else {
        *reinterpret_cast<uint2*>(dst) = make_uint2(v16.x, v16.y);
        if (rr + 16 < R) *reinterpret_cast<uint2*>(dst + 8) = make_uint2(v16.z, v16.w);
      }
    }
  }
  if (t < 128) {
    const int64_t c = c_first + t;
    const int64_t kb0 = rt >> 4, nkb = R >> 4;
    if (c < C) {
      const uint32_t sf4 = *reinterpret_cast<const uint32_t*>(sf_stage + 4 * t);
      const int64_t off0 = p.col_gemm ? sf_gemm_offset(c, kb0, p.col_kt) : c * nkb + kb0;
      if (kb0 + 4 <= nkb && (p.col_gemm || (nkb & 3) == 0)) {
        *reinterpret_cast<uint32_t*>(p.col_sf + off0) = sf4;  // 4 consecutive, 4-byte aligned scales
      } else {
#pragma unroll
        for (int b = 0; b < 4; ++b)
          if (kb0 + b < nkb)
            p.col_sf[p.col_gemm ? sf_gemm_offset(c, kb0 + b, p.col_kt) : c * nkb + kb0 + b] = (uint8_t)(sf4 >> (8 * b));
      }
    }
  }
}

// NVO (NVFP4 options, compile-time so that the plain paths carry none of the
// registers of the others): bit 0 stochastic rounding, bit 1 RHT of the
// column-wise copy.  The NVFP4 kernels run one tile per CTA at high occupancy
// (six CTAs per SM for the plain path at 40 registers, four with stochastic
// rounding at 64, five with the RHT at 47-48); the other kinds are persistent
// with a prefetched next tile (their 62-110 registers allow fewer resident
// CTAs, whose load latency the prefetch covers: FP8 column copy 63 -> 48 us
// at 15872 x 4096).  Persistence made the NVFP4 kernels slower (fewer
// resident CTAs with the prefetch registers).
__host__ __device__ constexpr bool tile_persistent(int kind) { return kind != QK_NV; }
__host__ __device__ constexpr int tile_min_ctas(int kind, int nvo) { return kind != QK_NV ? 1 : (nvo == 0 ? 6 : (nvo == 1 ? 4 : 5)); }

template <int KIND, bool kE5M2, int NVO = 0>
__global__ void __launch_bounds__(kThreads, tile_min_ctas(KIND, NVO)) quant_tile_kernel(const QParams p) {
  constexpr bool kSR = (NVO & 1) != 0, kRHT = (NVO & 2) != 0;
  constexpr int TR = (KIND == QK_BLK1 || KIND == QK_BLK128) ? 128 : 64;
  __shared__ __align__(16) uint16_t tile[TR][kTC];
  __shared__ float red[kThreads / 32];
  __shared__ float part[2][kTC];
  __shared__ float fb_tab[2][128];  // NVFP4: s_enc / dec(S) for the row and column copies
  // NVFP4 column-wise copy staged per column (64 rows: 32 code bytes, 4 scales)
  __shared__ __align__(16) uint8_t col_stage[KIND == QK_NV ? 128 * 32 : 16];
  __shared__ __align__(4) uint8_t sf_stage[KIND == QK_NV ? 128 * 4 : 4];

  const int t = threadIdx.x;
  // The shared tile feeds the column-wise copy and the 2D / 128x128 scales.
  const bool kNeedTile = p.col_codes != nullptr || KIND == QK_BLK128;
  const int64_t R = p.R, C = p.C;
  constexpr float kFmax = kE5M2 ? 57344.0f : 448.0f;

  // ---------------------------------------------------------------- tiles
  // CTA b takes tiles b, b + gridDim.x, ... (row-major over the [R / TR,
  // C / 128] tiles).  Persistent kinds issue the next tile's 16-byte loads
  // before the current tile is processed, so each CTA keeps a tile in flight
  // while it quantizes; NVFP4 launches one CTA per tile.
  const int lr = t >> 4;                     // row within a 16-row slab
  const int lc = (t & 15) * 8;               // first of this thread's 8 columns
  const int wr = t >> 3, wc = (t & 7) * 16;  // NVFP4: one thread per 16-value block, 32 rows a pass
  const int64_t ntx = (C + kTC - 1) / kTC;
  const int64_t ntiles = ntx * ((R + TR - 1) / TR);
  constexpr int NLD = TR / 16;  // 16-byte loads per thread and tile
  constexpr bool kPersist = tile_persistent(KIND);
  // origin of tile tl (persistent kinds) or of this CTA's tile (blockIdx)
  auto tile_origin = [&](int64_t tl, int64_t& r0, int64_t& c0) {
    if constexpr (kPersist) {
      const uint32_t ty = (uint32_t)tl / (uint32_t)ntx;  // fewer than 2^32 tiles (checked at launch)
      r0 = (int64_t)ty * TR;
      c0 = ((int64_t)tl - (int64_t)ty * ntx) * kTC;
    } else {
      r0 = (int64_t)blockIdx.y * TR;
      c0 = (int64_t)blockIdx.x * kTC;
    }
  };
  auto load_tile = [&](int64_t tl, uint4 (&v)[NLD]) {
    int64_t r0, c0;
    tile_origin(tl, r0, c0);
    if constexpr (KIND == QK_NV) {
      const bool wcol_ok = c0 + wc < C;  // C is a multiple of 16: whole blocks
#pragma unroll
      for (int it = 0; it < TR / 32; ++it) {
        const int64_t r = r0 + it * 32 + wr;
        const bool ok = wcol_ok && r < R;
        const uint16_t* src = p.x + r * C + c0 + wc;
        v[2 * it] = ok ? ld_stream(src) : make_uint4(0u, 0u, 0u, 0u);
        v[2 * it + 1] = ok ? ld_stream(src + 8) : make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
      const bool col_ok = c0 + lc < C;
#pragma unroll
      for (int it = 0; it < TR / 16; ++it) {
        const int64_t r = r0 + it * 16 + lr;
        v[it] = (col_ok && r < R) ? ld_stream(p.x + r * C + c0 + lc) : make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  float run_amax = 0.f;  // FP8 delayed scaling: the amax of every element this CTA reads
  // The first tile's loads go out before the scales are set up (the amax read,
  // the factor table, the barrier), so the two memory latencies overlap.
  uint4 nxt[NLD];
  int64_t tl = kPersist ? (int64_t)blockIdx.x : 0;
  const int64_t tl_end = kPersist ? ntiles : 1, tl_step = kPersist ? (int64_t)gridDim.x : 1;
  if (tl < tl_end) load_tile(tl, nxt);

  // ---------------------------------------------------------------- scales
  float scale = 1.0f;  // per-tensor FP8
  if constexpr (KIND == QK_FP8) {
    if (p.delayed_scale) {
      scale = *p.delayed_scale;
    } else {
      float a = *p.amax_row;
      scale = finite_pos(a) ? scale_quotient(kFmax, a) : 1.0f;
    }
    if (blockIdx.x == 0 && blockIdx.y == 0 && t == 0) {
      float sinv = __fdiv_rn(1.0f, scale);
      if (p.row_ts) *p.row_ts = sinv;
      if (p.col_ts) *p.col_ts = sinv;
    }
  }
  float s_enc_row = 1.f, s_enc_col = 1.f;
  uint32_t sgn_mask = 0;  // RHT signs as bits (flips of the sign bit; no registers of factors)
  if constexpr (KIND == QK_NV) {
    if (p.row_codes) s_enc_row = nv_s_enc(p.amax_row);
    if (p.col_codes) s_enc_col = nv_s_enc(p.amax_col);
    if (blockIdx.x == 0 && blockIdx.y == 0 && t == 0) {
      if (p.row_ts) *p.row_ts = nv_ts_dec(p.amax_row);
      if (p.col_ts) *p.col_ts = nv_ts_dec(p.amax_col);
    }
    if constexpr (kRHT) sgn_mask = rht_signs(p.rht_seed);
    nv_factor_table(fb_tab[0], s_enc_row, t);
    nv_factor_table(fb_tab[1], s_enc_col, t - 128);
    __syncthreads();
  }
  const PhiloxKeys keys(kSR ? p.seed : 0);  // dead (and free) without stochastic rounding

  for (; tl < tl_end; tl += tl_step) {
  int64_t r0, c0;
  tile_origin(tl, r0, c0);
  uint4 vbuf[NLD];
  if constexpr (kPersist) {
#pragma unroll
    for (int i = 0; i < NLD; ++i) vbuf[i] = nxt[i];
    if (tl + tl_step < tl_end) load_tile(tl + tl_step, nxt);
    __syncthreads();  // the previous tile's readers of the shared memory are done
  } else {
#pragma unroll
    for (int i = 0; i < NLD; ++i) vbuf[i] = nxt[i];  // this CTA's one tile, loaded at the start
  }
  const bool col_ok = c0 + lc < C;
  float local_amax = 0.f;
  if constexpr (KIND == QK_NV) {
    const bool wcol_ok = c0 + wc < C;
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
      const float s = finite_pos(m) ? scale_quotient(448.0f, m) : 1.0f;
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
  if constexpr (KIND == QK_FP8) run_amax = fmaxf(run_amax, local_amax);
  if (!kNeedTile) continue;
  __syncthreads();

  // ---------------------------------------------------------------- 128x128 tiles
  if constexpr (KIND == QK_BLK128) {
    const float m = block_max(local_amax, red);
    const float s = finite_pos(m) ? scale_quotient(448.0f, m) : 1.0f;
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
    continue;
  }

  if constexpr (KIND == QK_BLK1) {
    if (!p.col_codes) continue;
    const int cl = t & 127, rh = t >> 7;
    const int64_t c = c0 + cl, rbase = r0 + rh * 64;
    float m = 0.f;
#pragma unroll 16
    for (int i = 0; i < 64; ++i) m = absmax_acc(m, tile_val(tile[rh * 64 + i], cl));
    part[rh][cl] = m;
    __syncthreads();
    m = fmaxf(part[0][cl], part[1][cl]);
    const float s = finite_pos(m) ? scale_quotient(448.0f, m) : 1.0f;
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
    continue;
  }

  // ---------------------------------------------------------------- column-wise copy
  if (!p.col_codes) continue;
  if constexpr (KIND == QK_NV) {
    // Two adjacent columns per thread (each 4-byte shared load holds a row's
    // values of both), one 16-row block: RHT, block scale and codes per
    // column; the codes and scales are staged per column and leave as whole
    // 32-byte column segments.  R is a multiple of 16.
    const int cp = t & 63, rq = t >> 6;
    const int64_t c = c0 + 2 * cp, rr = r0 + 16 * rq;
    float f0[16], f1[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t wv = *reinterpret_cast<const uint32_t*>(&tile[16 * rq + i][2 * cp]);
      f0[i] = bf16_lo(wv);
      f1[i] = bf16_hi(wv);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float* f = h ? f1 : f0;
      if constexpr (kRHT) rht16(f, sgn_mask);
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) m = absmax_acc(m, f[i]);
      const uint32_t S = nv_block_scale(m, s_enc_col);
      const float fb = fb_tab[1][S];
      uint4 w[4] = {uint4{}, uint4{}, uint4{}, uint4{}};
      if constexpr (kSR) {
        const uint64_t g = (p.ctr_off + (uint64_t)((c + h) * R + rr)) >> 2;
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = keys.words(g + j, 1u);
      }
      const uint32_t a = nv_codes8(f, fb, kSR, w[0], w[1]);
      const uint32_t b = nv_codes8(f + 8, fb, kSR, w[2], w[3]);
      const int cl = 2 * cp + h;
      *reinterpret_cast<uint2*>(col_stage + cl * 32 + rq * 8) = make_uint2(a, b);
      sf_stage[cl * 4 + rq] = (uint8_t)S;
    }
    __syncthreads();
    store_col_staged(p, col_stage, sf_stage, c0, r0, t);
    continue;
  }
  const int cl = t & 127, rh = t >> 7;
  const int64_t c = c0 + cl, rbase = r0 + rh * 32;
  if (c >= C || rbase >= R) continue;
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
  }  // tiles
  if constexpr (KIND == QK_FP8) {
    if (p.fused_amax0) {  // delayed scaling: amax measured in this pass, one atomic per CTA
      const float m = block_max(run_amax, red);
      if (t == 0) {
        atomic_max_nonneg(p.fused_amax0, m);
        if (p.fused_amax1) atomic_max_nonneg(p.fused_amax1, m);
      }
    }
  }
}


// ---------------------------------------------------------------- NVFP4 2D (16x16 weight tiles)
// One CTA per 64 x 128 tile; warp w owns the 16 x 64 strip at rows
// 16 (w / 2), columns 64 (w % 2): lane l loads 8 columns (8 (l % 8)) of rows
// 4 (l / 8) .. +3, so each load instruction reads four 128-byte row segments.
// A 16 x 16 tile lives in 8 lanes (lane bits 0, 3, 4), whose shuffle max is
// the tile max; nothing goes through shared memory.  The codes are the same
// for both copies (one scale per tile, element-wise encoding), so the
// column-wise copy is the nibble transpose of the row-wise codes: within a
// lane (4 rows x 8 columns) by byte permutes, then across the strip's four
// row groups by shuffles; lane l stores columns 2 (l / 8) and 2 (l / 8) + 1
// of its 8 as two 8-byte words (16 rows), gathered per column in shared memory.
// 48 registers, five CTAs per SM (the column copy is 11% faster than at four).
__device__ __forceinline__ uint32_t nib_lo4(uint32_t x) {  // low nibbles of 4 bytes -> 16 bits
  uint32_t y = x & 0x0F0F0F0Fu;
  y = (y | (y >> 4)) & 0x00FF00FFu;
  return __byte_perm(y, 0u, 0x4420);
}

__global__ void __launch_bounds__(kThreads, 5) nv2d_kernel(const QParams p) {
  __shared__ float fb_tab[128];  // s_enc / dec(S) for the 128 E4M3 codes
  __shared__ __align__(16) uint8_t col_stage[128 * 32];  // column-wise codes: column, 64 rows
  __shared__ __align__(4) uint8_t sf_stage[128 * 4];     // column-wise scales: column, 4 row blocks
  const int t = threadIdx.x, w = t >> 5, l = t & 31;
  const int chunk = l & 7, rsub = l >> 3;
  const int64_t R = p.R, C = p.C;
  const int64_t r0 = (int64_t)blockIdx.y * 64 + 16 * (w >> 1);                // the warp's 16 rows
  const int64_t cw = (int64_t)blockIdx.x * 128 + 64 * (w & 1) + 8 * chunk;  // the lane's first column
  // One weight amax: the tile scales use the row copy's encode scale (the
  // column copy's when only it is requested).
  const bool use_row = p.row_codes != nullptr;
  const float s_enc = nv_s_enc(use_row ? p.amax_row : p.amax_col);
  if (blockIdx.x == 0 && blockIdx.y == 0 && t == 0) {
    if (p.row_ts) *p.row_ts = nv_ts_dec(p.amax_row);
    if (p.col_ts) *p.col_ts = nv_ts_dec(p.amax_col);
  }
  nv_factor_table(fb_tab, s_enc, t);
  __syncthreads();
  // R and C are multiples of 16: a lane's rows and columns are all in range
  // or all out (then it loads zeros and stores nothing).
  const bool ok = cw < C && r0 < R;
  uint4 v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    v[i] = ok ? ld_stream(p.x + (r0 + 4 * rsub + i) * C + cw) : make_uint4(0u, 0u, 0u, 0u);
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float f[8];
    unpack8(v[i], f);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = absmax_acc(m, f[j]);
  }
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 8));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
  const uint32_t S = nv_block_scale(m, s_enc);
  const float fb = fb_tab[S];
  uint32_t q[4];  // codes of row 4 rsub + i: nibble j = column cw + j
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float f[8];
    unpack8(v[i], f);
    q[i] = nv_codes8(f, fb, false, uint4{}, uint4{});
  }
  if (p.row_codes && ok) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = r0 + 4 * rsub + i;
      *reinterpret_cast<uint32_t*>(p.row_codes + r * (C >> 1) + (cw >> 1)) = q[i];
      if ((chunk & 1) == 0) {
        const int64_t kb = cw >> 4;
        p.row_sf[p.row_gemm ? sf_gemm_offset(r, kb, p.row_kt) : r * (C >> 4) + kb] = (uint8_t)S;
      }
    }
  }
  if (!p.col_codes) return;
  // Byte b of q[i] holds columns 2b, 2b+1 of row i.  X[b] = byte b of q[0..3].
  const uint32_t t01l = __byte_perm(q[0], q[1], 0x5140), t01h = __byte_perm(q[0], q[1], 0x7362);
  const uint32_t t23l = __byte_perm(q[2], q[3], 0x5140), t23h = __byte_perm(q[2], q[3], 0x7362);
  const uint32_t X[4] = {__byte_perm(t01l, t23l, 0x5410), __byte_perm(t01l, t23l, 0x7632),
                         __byte_perm(t01h, t23h, 0x5410), __byte_perm(t01h, t23h, 0x7632)};
  // H[k]: columns 2k (low 16 bits) and 2k+1 (high 16 bits), nibble i = row 4 rsub + i.
  uint32_t H[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) H[k] = nib_lo4(X[k]) | (nib_lo4(X[k] >> 4) << 16);
  // This lane stores columns 2 rsub, 2 rsub + 1: gather H[rsub] of the four row groups.
  uint32_t G[4];  // G[g] = H[rsub] of row group g
#pragma unroll
  for (int g = 0; g < 4; ++g) G[g] = 0u;
#pragma unroll
  for (int d = 0; d < 4; ++d) {
    const int k = rsub ^ d;  // what the partner (row group rsub ^ d) needs from this lane
    const uint32_t send = k == 0 ? H[0] : k == 1 ? H[1] : k == 2 ? H[2] : H[3];
    const uint32_t got = d == 0 ? send : __shfl_xor_sync(0xFFFFFFFFu, send, 8 * d);
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (g == k) G[g] = got;
  }
  // The CTA's four row groups write their 8-byte column words and tile
  // scales to shared memory; then each column's 32 code bytes (64 rows) leave
  // as two 16-byte stores and its 4 scales as one 4-byte store where the
  // layout allows (else in pieces).
  const int rb = w >> 1;
  if (ok) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t sel = e ? 0x7632u : 0x5410u;
      const int cl = 64 * (w & 1) + 8 * chunk + 2 * rsub + e;
      *reinterpret_cast<uint2*>(col_stage + cl * 32 + rb * 8) =
          make_uint2(__byte_perm(G[0], G[1], sel), __byte_perm(G[2], G[3], sel));
      sf_stage[cl * 4 + rb] = (uint8_t)S;
    }
  }
  __syncthreads();
  store_col_staged(p, col_stage, sf_stage, (int64_t)blockIdx.x * 128, (int64_t)blockIdx.y * 64, t);
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
      const float scale = finite_pos(a) ? scale_quotient(fmax, a) : 1.0f;
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
    // A position outside [0, len) (a corrupted or foreign checkpoint) is taken
    // modulo len, so the ring write stays inside the history.
    slot = ((*pos % len) + len) % len;
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
    if (finite_pos(mm)) s = scale_quotient(fmax, mm);
    *scale = s;
    *scale_inv = __fdiv_rn(1.0f, s);
  }
}

template <int KIND, bool kE5M2, int NVO = 0>
lpq_status run_tile(const QParams& p, cudaStream_t s) {
  constexpr int TR = (KIND == QK_BLK1 || KIND == QK_BLK128) ? 128 : 64;
  const int64_t tiles = ((p.C + kTC - 1) / kTC) * ((p.R + TR - 1) / TR);
  if (tiles == 0) return LPQ_OK;
  // persistent kinds: as many CTAs as fit on the GPU at once (each loops
  // over tiles); NVFP4: one CTA per tile
  dim3 grid((unsigned)((p.C + kTC - 1) / kTC), (unsigned)((p.R + TR - 1) / TR));
  if (tile_persistent(KIND)) {
    if (tiles >= ((int64_t)1 << 32)) return set_error(LPQ_ERR_SHAPE, "too many tiles (%lld)", (long long)tiles);
    const int per_sm = resident_ctas(reinterpret_cast<const void*>(quant_tile_kernel<KIND, kE5M2, NVO>), kThreads);
    grid = dim3((unsigned)std::min<int64_t>(tiles, (int64_t)device_sms() * per_sm), 1);
  } else if (grid.y > 65535u) {
    return set_error(LPQ_ERR_SHAPE, "too many rows (%lld) for one launch", (long long)p.R);
  }
  quant_tile_kernel<KIND, kE5M2, NVO><<<grid, kThreads, 0, s>>>(p);
  return cuda_check(cudaGetLastError(), "quantize kernel launch");
}

lpq_status run_nv2d(const QParams& p, cudaStream_t s) {
  dim3 grid((unsigned)((p.C + kTC - 1) / kTC), (unsigned)((p.R + 63) / 64));
  if (grid.y > 65535u) return set_error(LPQ_ERR_SHAPE, "too many rows (%lld) for one launch", (long long)p.R);
  nv2d_kernel<<<grid, kThreads, 0, s>>>(p);
  return cuda_check(cudaGetLastError(), "NVFP4 2D kernel launch");
}

lpq_status run_amax(const uint16_t* x, int64_t R, int64_t C, float* o0, float* o1, float* rht_out,
                    uint32_t rht_seed, cudaStream_t s) {
  const int64_t units = rht_out ? (R / 16) * (C / 8) : R * (C / 8);
  int64_t blocks = (units + kThreads - 1) / kThreads;
  const int64_t cap = (int64_t)device_sms() * 8;
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
      {  // optional amax outputs: whichever views ask for one get max |x|
        float* a0 = rv ? rv->amax : nullptr;
        float* a1 = cv ? cv->amax : nullptr;
        if (!a0) { a0 = a1; a1 = nullptr; }
        if (a0) {
          if ((st = zero_f32(a0, s)) != LPQ_OK || (st = zero_f32(a1, s)) != LPQ_OK) return st;
          if ((st = run_amax(p.x, R, C, a0, a1, nullptr, 0, s)) != LPQ_OK) return st;
        }
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
      if (fmt == LPQ_NVFP4_2D) return run_nv2d(p, s);
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

// ---------------------------------------------------------------- arithmetic self-checks
// Device helpers of the quantizers against their definitions, for the test
// suite (lpq_selftest_arith).  out[0] counts mismatches, out[1] keeps the
// smallest mismatching index.
namespace {

__global__ void selftest_init_kernel(unsigned long long* out) {
  out[0] = 0ull;
  out[1] = ~0ull;
}

// Stochastic E2M1 rounding stated directly: adjacent grid magnitudes
// lo <= |y| < hi, frac = (|y| - lo) / (hi - lo) in double (exact: the spacing
// is a power of two), round up iff float(r >> 8) < frac * 2^24; |y| >= 6 and
// NaN give 6; the sign of y is kept.
__device__ float sr_e2m1_definition(float y, uint32_t r) {
  if (y != y) return 6.0f;
  const float a = fabsf(y);
  float v;
  if (a >= 6.0f) {
    v = 6.0f;
  } else {
    const float g[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
    int j = 0;
    while (j < 6 && g[j + 1] <= a) ++j;
    const double lo = g[j], hi = g[j + 1];
    const double thr = ((double)a - lo) / (hi - lo) * 16777216.0;
    v = (double)(r >> 8) < thr ? (float)hi : (float)lo;
  }
  return copysignf(v, y);
}

__device__ __forceinline__ void selftest_record(unsigned long long* out, uint64_t i) {
  atomicAdd(&out[0], 1ull);
  atomicMin(&out[1], (unsigned long long)i);
}

// which 0: x = the float with bits i (i <= 0x7F800000: every non-negative
//   float and +inf): div6_rn(x) against the IEEE quotient x / 6.
// which 1: |y| = the float with bits i >> 3, r = the (i & 7)-th probe word
//   (r >> 8 = 0, 1, 2^23 - 2, 2^23, 2^24 - 3, 2^24 - 2, 2^24 - 1, low bytes
//   0x00 or 0xFF); y and -y as one pair through sr_e2m1_value2.
// which 2: y = the float with bits `param`, r = i << 8 | (low byte i * 37),
//   i < 2^24: every threshold word for one y, pairs (y, -y).
__global__ void selftest_arith_kernel(int which, uint64_t begin, uint64_t count, uint32_t param,
                                      unsigned long long* out) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t k = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; k < count; k += stride) {
    const uint64_t i = begin + k;
    if (which == 0) {
      const float x = __uint_as_float((uint32_t)i);
      if (__float_as_uint(div6_rn(x)) != __float_as_uint(__fdiv_rn(x, 6.0f))) selftest_record(out, i);
    } else {
      float y;
      uint32_t r;
      if (which == 1) {
        y = __uint_as_float((uint32_t)(i >> 3));
        const uint32_t probes[8] = {0x00000000u, 0x000001FFu, 0x7FFFFE00u, 0x800000FFu,
                                    0xFFFFFD00u, 0xFFFFFEFFu, 0xFFFFFF00u, 0xFFFFFFFFu};
        r = probes[i & 7];
      } else {
        y = __uint_as_float(param);
        r = ((uint32_t)i << 8) | ((uint32_t)(i * 37u) & 0xFFu);
      }
      const float2 got = sr_e2m1_value2(make_float2(y, -y), r, r);
      if (__float_as_uint(got.x) != __float_as_uint(sr_e2m1_definition(y, r)) ||
          __float_as_uint(got.y) != __float_as_uint(sr_e2m1_definition(-y, r)))
        selftest_record(out, i);
    }
  }
}

}  // namespace

lpq_status launch_selftest_arith(int32_t which, uint64_t begin, uint64_t count, uint32_t param, int64_t* out,
                                 cudaStream_t s) {
  auto* o = reinterpret_cast<unsigned long long*>(out);
  selftest_init_kernel<<<1, 1, 0, s>>>(o);
  selftest_arith_kernel<<<device_sms() * 8, 256, 0, s>>>(which, begin, count, param, o);
  return cuda_check(cudaGetLastError(), "arithmetic self-check launch");
}

lpq_status launch_amax(const void* x, int64_t R, int64_t C, bool rht, uint32_t rht_seed, float* amax, float* rht_amax,
                       cudaStream_t s) {
  float* rh = rht ? rht_amax : nullptr;
  lpq_status st;
  if ((st = zero_f32(amax, s)) != LPQ_OK || (st = zero_f32(rh, s)) != LPQ_OK) return st;
  if (R == 0 || C == 0) return LPQ_OK;
  return run_amax(static_cast<const uint16_t*>(x), R, C, amax, nullptr, rh, rht_seed, s);
}

lpq_status launch_scale_update(const lpq_delayed_state* st, const float* amax, float fmax, cudaStream_t s) {
  scale_update_kernel<<<1, 128, 0, s>>>(st->amax_history, st->pos, st->scale, st->scale_inv, st->len, amax, fmax);
  return cuda_check(cudaGetLastError(), "scale update launch");
}

}  // namespace lpq
