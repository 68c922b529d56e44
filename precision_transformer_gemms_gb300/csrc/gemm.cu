// Tensor-core GEMMs of liblpq on sm_103a: C[m, n] = sum_k A[m, k] B[n, k]
// with both operands contiguous along k ("TN"), as every Fprop, Dgrad and
// Wgrad of a linear layer is posed ("How to optimize Transformer-based models
// for low-precision training", autocast vs pre-quantize: the 12 GEMMs of a
// layer, benchmarked separately per pass).
//
// Persistent, warp-specialized kernels.  Warp 0 (one lane) streams A/B tiles
// into a shared-memory ring with TMA (128-byte swizzle) and the block scale
// factors with bulk or TMA copies; warp 1 (one lane) issues the tcgen05.mma
// instructions, accumulating in FP32 in TMEM; for the block-scaled kinds four
// scale warps write each stage's scale factors into a TMEM slot with
// tcgen05.st (or, with lpq_gemm_opts.scale_copies, the MMA thread copies them
// with tcgen05.cp); eight epilogue warps read the accumulator back with
// tcgen05.ld, apply the per-tensor scale product and store bf16 or FP32.  The
// default for M >= 256 is a CTA pair (cta_group::2) per 256 x 256 tile.
//
// Kinds: kind::f16 (bf16 x bf16), kind::f8f6f4 (per-tensor E4M3/E5M2),
// kind::mxf8f6f4.block_scale (MXFP8: E4M3 or E5M2 with an E8M0 scale per 32
// values, "Faster training throughput in FP8 with NVIDIA NeMo", MXFP8),
// kind::mxf4nvf4.block_scale.scale_vec::4X (NVFP4: E2M1 with an E4M3 scale per
// 16 values and an FP32 tensor scale, "Accelerate LLM training with NVFP4 on
// Blackwell") and scale_vec::2X (MXFP4: E2M1 with an E8M0 scale per 32).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "lpq_device.cuh"

namespace lpq {

// Device error word: set when a bounded wait inside a kernel of this library
// gives up; read and cleared by lpq_device_status.
__device__ int g_device_error = 0;

namespace {

constexpr int kBM = 128;
constexpr int kKBytes = 128;  // bytes of K per pipeline stage (one 128-byte swizzle row)

// Scale atoms (512 bytes: 4 scales of each of 128 rows) per k-step of
// kKBytes: 128 FP8 values = 4 MX blocks (one atom); 256 FP4 values = 8 MX
// blocks (two) or 16 NVFP4 blocks (four).
constexpr int sf_atoms_per_step(int kind) {
  return kind == kKindNVF4 ? 4 : kind == kKindMXF4 ? 2 : kind == kKindMXF8 ? 1 : 0;
}
// Instruction-descriptor scale selectors of MMA j (K = 32 or 64) of a k-step:
// MXFP8 (one scale per MMA) takes byte j of the atom's 32-bit column, MXFP4
// (two per MMA) bytes 2 (j % 2) and 2 (j % 2) + 1 of atom j / 2, NVFP4 (four
// per MMA) the whole column of atom j.
template <int KIND>
__device__ __forceinline__ uint32_t sf_select(int j) {
  const uint32_t id = KIND == kKindMXF8 ? (uint32_t)j : KIND == kKindMXF4 ? (uint32_t)(j & 1) * 2u : 0u;
  return (id << 4) | (id << 29);
}

template <int KIND, int BN, int NACC, bool SFST = false>
struct Cfg {
  static constexpr int kSfAtoms = sf_atoms_per_step(KIND);  // per 128 rows
  static constexpr int kA = kBM * kKBytes;
  static constexpr int kB = BN * kKBytes;
  static constexpr int kSfa = kSfAtoms * 512;
  static constexpr int kSfb = kSfAtoms * 512 * (BN / 128);
  static constexpr int kStage = kA + kB + kSfa + kSfb;
  static constexpr int kStages = (220 * 1024) / kStage > 8 ? 8 : (220 * 1024) / kStage;
  static constexpr int kSmem = kStages * kStage + 1024 /*align slack*/ + 512 /*barriers*/;
  static constexpr int kSfaCols = kSfAtoms * 4;
  static constexpr int kSfbCols = kSfAtoms * 4 * (BN / 128);
  // SFST: one TMEM scale slot per stage, written by the scale warps
  static constexpr int kSlots = SFST ? kStages : 1;
  static constexpr int kCols = NACC * BN + kSlots * (kSfaCols + kSfbCols);
  static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static_assert(kCols <= 512, "TMEM holds 512 columns");
  static_assert(BN % 128 == 0 || kSfAtoms == 0, "scale atoms cover 128 rows");
};

constexpr int kGroupM = 16;  // tiles along M that share a band of B tiles (L2 reuse)
constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, each owning half of the tile's columns
constexpr int kThreadsGemm = 64 + 32 * kEpiWarps;
constexpr int kSfWarps = 4;  // scale-store warps of the block-scaled kernels, one per TMEM lane quarter

struct GemmArgs {
  const uint8_t* sfa;  // tensor-core scale layout of A (block-scaled kinds)
  const uint8_t* sfb;
  int64_t sfa_kt, sfb_kt;  // atoms per 128-row group
  int64_t sfb_groups;      // 128-row groups of B
  void* c;
  int64_t M, N, K;
  int c_fp32;
  int c_tma;             // bf16 C written by TMA tile stores (pair kernel; N % 8 == 0)
  const float* alpha_a;  // per-tensor factors (may be NULL)
  const float* alpha_b;
  uint32_t idesc;
  uint32_t idesc_half;  // CTA-pair kernel: the same with N = 128 (half tiles)
  int num_k;  // k-tiles of kKBytes
  int tiles_m, tiles_n;
  int full_tiles, items;  // CTA-pair kernel: work items (whole tiles, then half tiles)
};

// Tile t of the persistent schedule -> (m tile, n tile): consecutive tiles
// walk down a band of kGroupM m-tiles before moving to the next n-tile.
__device__ __forceinline__ void tile_coords(int t, int tiles_m, int tiles_n, int& mt, int& nt) {
  const int per_group = kGroupM * tiles_n;
  const int group = t / per_group;
  const int first_m = group * kGroupM;
  const int gsize = min(kGroupM, tiles_m - first_m);
  const int r = t - group * per_group;
  mt = first_m + r % gsize;
  nt = r / gsize;
}

// Work item w of the CTA-pair kernel's persistent schedule -> (m tile, n tile,
// part): the first g.full_tiles items are whole 256 x 256 tiles in tile_coords
// order; each item after them is one 256 x 128 half (part 0 or 1) of the
// remaining tiles, two items per tile.  part = -1 for a whole tile.
__device__ __forceinline__ void work_coords(int w, int full_tiles, int tiles_m, int tiles_n, int& mt, int& nt,
                                            int& part) {
  if (w < full_tiles) {
    tile_coords(w, tiles_m, tiles_n, mt, nt);
    part = -1;
    return;
  }
  const int h = w - full_tiles;
  tile_coords(full_tiles + (h >> 1), tiles_m, tiles_n, mt, nt);
  part = h & 1;
}

// After an abort: wait (bounded, whatever the abort flag says) until the loads
// issued for ring uses [from, to) have landed, so that none is in flight when
// the CTA exits.  Use k of a ring of `n` entries completes phase k / n of
// barrier k % n.
__device__ __forceinline__ void drain_stages(uint64_t* bars, int n, uint32_t from, uint32_t to) {
  volatile int no_abort = 0;
  for (uint32_t k = from; k < to; ++k) mbar_wait_bounded(&bars[k % n], (k / n) & 1u, &no_abort, &g_device_error);
}

// Persistent warp-specialized GEMM.  Warp 0: TMA producer; warp 1: TMEM
// allocator and MMA issuer; warps 2..5: epilogue (warp w reads TMEM lanes
// 32 * (w % 4) ..).  The shared-memory ring runs continuously across the
// CTA's tiles; NACC accumulators in TMEM let the epilogue of one tile overlap
// the main loop of the next.
template <int KIND, int BN, int NACC, bool SFST>
__global__ void __launch_bounds__(kThreadsGemm + (SFST ? 32 * kSfWarps : 0))
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmArgs g) {
  using CF = Cfg<KIND, BN, NACC, SFST>;
  constexpr int S = CF::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * CF::kA;
  uint8_t* sSfa = sB + S * CF::kB;
  uint8_t* sSfb = sSfa + S * CF::kSfa;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSfb + S * CF::kSfb);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* sfd = acc_empty + NACC;         // [S] (SFST): the stage's scale atoms landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfd + S);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = g.tiles_m * g.tiles_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // SFST: the stage is full once its A/B landed and the four scale warps
      // have written its scale slot; the MMA commit alone empties it (the
      // scale warps have read the stage's scale atoms before they arrive).
      mbar_init(&full[s], SFST ? 1 + kSfWarps : 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sfd[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kEpiWarps);  // one arrive per epilogue warp
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, CF::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t tmem_sfa = tmem_base + NACC * BN;
  const uint32_t tmem_sfb = tmem_sfa + CF::kSfaCols;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      const int elem_per_kt = KIND == kKindF16 ? kKBytes / 2 : kKBytes;  // TMA x unit: elements (bf16) or bytes
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int mt, nt;
        tile_coords(t, g.tiles_m, g.tiles_n, mt, nt);
        const int32_t m0 = mt * kBM, n0 = nt * BN;
        for (int kt = 0; kt < g.num_k; ++kt, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!(ok = mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag, &g_device_error))) break;
          // Scale atoms first; with scale warps they land on a barrier of their
          // own, so the warps move them into TMEM while A and B still arrive.
          uint64_t* sbar = SFST ? &sfd[s] : &full[s];
          if constexpr (SFST) mbar_arrive_expect_tx(&sfd[s], CF::kSfa + CF::kSfb);
          mbar_arrive_expect_tx(&full[s], SFST ? CF::kA + CF::kB : CF::kStage);
          if constexpr (CF::kSfAtoms > 0) {
            bulk_load(sSfa + s * CF::kSfa, g.sfa + ((int64_t)mt * g.sfa_kt + (int64_t)kt * CF::kSfAtoms) * 512,
                      CF::kSfa, sbar);
#pragma unroll
            for (int i = 0; i < BN / 128; ++i) {
              int64_t gb = (int64_t)n0 / 128 + i;
              if (gb >= g.sfb_groups) gb = g.sfb_groups - 1;
              bulk_load(sSfb + s * CF::kSfb + i * CF::kSfAtoms * 512,
                        g.sfb + (gb * g.sfb_kt + (int64_t)kt * CF::kSfAtoms) * 512, CF::kSfAtoms * 512, sbar);
            }
          }
          tma_load_2d(sA + s * CF::kA, &tmA, kt * elem_per_kt, m0, &full[s]);
          tma_load_2d(sB + s * CF::kB, &tmB, kt * elem_per_kt, n0, &full[s]);
        }
      }
      // After an abort, let the loads still in flight land before the CTA exits.
      if (!ok) drain_stages(full, S, it > (uint32_t)S ? it - S : 0u, it);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      // Descriptors are precomputed: only the low word (start address >> 4)
      // changes between stages and K steps.  Each MMA's scale-factor copies
      // are issued right before it, so they overlap the previous MMA.
      const uint32_t kHiSw = (uint32_t)(smem_desc(0, 16, 1024, 2) >> 32);
      const uint32_t kLoSw = (uint32_t)smem_desc(0, 16, 1024, 2);
      const uint32_t kHiSf = (uint32_t)(smem_desc(0, 0, 128, 0) >> 32);
      const uint32_t a0 = kLoSw | (smem_u32(sA) >> 4), b0 = kLoSw | (smem_u32(sB) >> 4);
      const uint32_t fa0 = smem_u32(sSfa) >> 4, fb0 = smem_u32(sSfb) >> 4;
      uint32_t s = 0, ph = 0, lt = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++lt) {
        const uint32_t a = lt % NACC, aph = (lt / NACC) & 1u;
        if (!(ok = mbar_wait_bounded(&acc_empty[a], aph ^ 1u, abort_flag, &g_device_error))) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + a * BN;
        for (int kt = 0; kt < g.num_k; ++kt) {
          if (!(ok = mbar_wait_bounded(&full[s], ph, abort_flag, &g_device_error))) break;
          tc_fence_after();
          const uint32_t alo = a0 + s * (CF::kA >> 4), blo = b0 + s * (CF::kB >> 4);
          const uint32_t falo = fa0 + s * (CF::kSfa >> 4), fblo = fb0 + s * (CF::kSfb >> 4);
          if constexpr (KIND == kKindMXF8 && !SFST) {
            tmem_cp_sf(tmem_sfa, ((uint64_t)kHiSf << 32) | falo);
#pragma unroll
            for (int i = 0; i < BN / 128; ++i) tmem_cp_sf(tmem_sfb + 4 * i, ((uint64_t)kHiSf << 32) | (fblo + i * 32));
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t ad = ((uint64_t)kHiSw << 32) | (alo + 2 * j);
            const uint64_t bd = ((uint64_t)kHiSw << 32) | (blo + 2 * j);
            const uint32_t acc = (kt > 0 || j > 0) ? 1u : 0u;
            if constexpr (KIND == kKindF16 || KIND == kKindF8F6F4) {
              mma_ss<KIND>(tmem_d, ad, bd, g.idesc, acc);
            } else if constexpr (KIND == kKindMXF8 && !SFST) {
              mma_bs<KIND>(tmem_d, ad, bd, g.idesc | ((uint32_t)j << 4) | ((uint32_t)j << 29), tmem_sfa, tmem_sfb, acc);
            } else if constexpr (SFST) {
              const int at = j * CF::kSfAtoms / 4;  // the MMA's scale atom
              const uint32_t base = tmem_sfa + s * (CF::kSfaCols + CF::kSfbCols);  // the stage's slot
              mma_bs<KIND>(tmem_d, ad, bd, g.idesc | sf_select<KIND>(j), base + 4 * at,
                           base + CF::kSfaCols + 4 * (BN / 128) * at, acc);
            } else {
              const int at = j * CF::kSfAtoms / 4;
              if ((j * CF::kSfAtoms) % 4 == 0) {  // first MMA of the atom: copy it
                tmem_cp_sf(tmem_sfa + 4 * at, ((uint64_t)kHiSf << 32) | (falo + at * 32));
#pragma unroll
                for (int i = 0; i < BN / 128; ++i)
                  tmem_cp_sf(tmem_sfb + 4 * (BN / 128) * at + 4 * i,
                             ((uint64_t)kHiSf << 32) | (fblo + (i * CF::kSfAtoms + at) * 32));
              }
              mma_bs<KIND>(tmem_d, ad, bd, g.idesc | sf_select<KIND>(j), tmem_sfa + 4 * at,
                           tmem_sfb + 4 * (BN / 128) * at, acc);
            }
          }
          tc_commit(&empty[s]);
          if (++s == (uint32_t)S) { s = 0; ph ^= 1u; }
        }
        if (ok) tc_commit(&acc_full[a]);
      }
    }
  } else if (SFST && warp >= 2 + kEpiWarps) {
    if constexpr (SFST) {  // only kernels with scale warps carry this code
      // ------------------------------------------------------------ scale warps (block-scaled kinds)
      // Per k-step: once the stage's previous MMAs are done (its TMEM scale slot
      // is free), this warp's lane quarter of the step's scale atoms (per 128
      // rows: 1 MXFP8, 2 MXFP4, 4 NVFP4) goes from shared memory into the slot
      // with tcgen05.st (replicated in every quarter), and the warp arrives on
      // the stage's full barrier.
      const int q = warp & 3;
      const uint32_t lanes = (uint32_t)(q * 32) << 16;
      uint32_t s = 0, ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        for (int kt = 0; kt < g.num_k; ++kt) {
          if (!(ok = mbar_wait_bounded(&sfd[s], ph, abort_flag, &g_device_error))) break;
          if (!(ok = mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag, &g_device_error))) break;  // slot free
          __syncwarp();
          tc_fence_after();
          constexpr int NA = CF::kSfAtoms, G = BN / 128;
          const uint4* fa = reinterpret_cast<const uint4*>(sSfa + s * CF::kSfa) + lane;  // atom j line `lane`
          const uint4* fb = reinterpret_cast<const uint4*>(sSfb + s * CF::kSfb) + lane;
          uint32_t va[4 * NA], vb[4 * NA * G];
#pragma unroll
          for (int j = 0; j < NA; ++j) {
            const uint4 x = fa[j * 32];
            va[4 * j] = x.x; va[4 * j + 1] = x.y; va[4 * j + 2] = x.z; va[4 * j + 3] = x.w;
#pragma unroll
            for (int i = 0; i < G; ++i) {
              const uint4 y = fb[(i * NA + j) * 32];
              const int c = 4 * G * j + 4 * i;
              vb[c] = y.x; vb[c + 1] = y.y; vb[c + 2] = y.z; vb[c + 3] = y.w;
            }
          }
          const uint32_t base = tmem_base + NACC * BN + s * (CF::kSfaCols + CF::kSfbCols) + lanes;
          tmem_st_cols(base, va);
          tmem_st_cols(base + CF::kSfaCols, vb);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[s]);
          if (++s == (uint32_t)S) { s = 0; ph ^= 1u; }
        }
      }
    }  // SFST
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lanes 32 * (w % 4) .. of columns [half * BN/2, +BN/2).
    constexpr int HALF = BN / 2;
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    float alpha = 1.0f;
    if (g.alpha_a) alpha = *g.alpha_a;
    if (g.alpha_b) alpha = __fmul_rn(alpha, *g.alpha_b);
    const bool vec_ok = g.c_fp32 ? (g.N % 4 == 0) : (g.N % 8 == 0);
    uint32_t lt = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
      int mt, nt;
      tile_coords(t, g.tiles_m, g.tiles_n, mt, nt);
      const uint32_t a = lt % NACC, aph = (lt / NACC) & 1u;
      if (!mbar_wait_bounded(&acc_full[a], aph, abort_flag, &g_device_error)) break;
      __syncwarp();
      tc_fence_after();
      const int64_t row = (int64_t)mt * kBM + q * 32 + lane;
      const int64_t c0 = (int64_t)nt * BN + half * HALF;
      const int64_t ncols = g.N - c0;
      const uint32_t tbase = tmem_base + a * BN + half * HALF + ((uint32_t)(q * 32) << 16);
      if (!g.c_fp32) {
        // bf16: the warp's whole column range into registers as packed pairs,
        // TMEM handed back, then the stores.
        uint32_t pk[HALF / 2];
#pragma unroll
        for (int cc = 0; cc < HALF / 32; ++cc) {
          uint32_t v[32];
          tmem_ld32(tbase + (uint32_t)(cc * 32), v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            // one packed two-wide multiply (each half rounded like __fmul_rn), one packed convert
            const float2 y = __fmul2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                        make_float2(alpha, alpha));
            __nv_bfloat162 h = __floats2bfloat162_rn(y.x, y.y);
            pk[cc * 16 + i] = *reinterpret_cast<uint32_t*>(&h);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[a]);
        if (row < g.M && ncols > 0) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(g.c) + row * g.N + c0;
          if (vec_ok && ncols >= HALF) {
#pragma unroll
            for (int i = 0; i < HALF / 8; ++i)
              reinterpret_cast<uint4*>(out)[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          } else {
#pragma unroll
            for (int i = 0; i < HALF / 2; ++i) {
              if (2 * i < ncols) out[2 * i] = __ushort_as_bfloat16((unsigned short)(pk[i] & 0xFFFFu));
              if (2 * i + 1 < ncols) out[2 * i + 1] = __ushort_as_bfloat16((unsigned short)(pk[i] >> 16));
            }
          }
        }
        continue;
      }
#pragma unroll 1
      for (int cc = 0; cc < HALF / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)(cc * 32), v);
        if (cc == HALF / 32 - 1) {  // accumulator columns fully read: hand them back
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[a]);
        }
        const int64_t col0 = c0 + cc * 32;
        if (row >= g.M || col0 >= g.N) continue;
        float* out = static_cast<float*>(g.c) + row * g.N + col0;
        if (vec_ok && col0 + 32 <= g.N) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(out)[i] = make_float4(
                __fmul_rn(__uint_as_float(v[4 * i]), alpha), __fmul_rn(__uint_as_float(v[4 * i + 1]), alpha),
                __fmul_rn(__uint_as_float(v[4 * i + 2]), alpha), __fmul_rn(__uint_as_float(v[4 * i + 3]), alpha));
        } else {
          for (int i = 0; i < 32 && col0 + i < g.N; ++i) out[i] = __fmul_rn(__uint_as_float(v[i]), alpha);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, CF::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2D map over a row-major [rows, inner] matrix whose rows are `row_bytes`
// apart; box = box_inner x box_rows, 128-byte swizzle, zero fill outside.
lpq_status make_map(CUtensorMap* map, const void* base, bool bf16, int64_t inner, int64_t rows, int64_t row_bytes,
                    uint32_t box_inner, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(LPQ_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(LPQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return LPQ_OK;
}

// Instruction descriptors (tcgen05): D format F32 in bits 4-5 (dense kinds),
// A/B formats in 7-9 / 10-12, K-major A and B (bits 15, 16 clear), N >> 3 in
// 17-22, M >> 4 in 24-28; block-scaled kinds put the scale type in bit 23
// (1 = E8M0, 0 = E4M3) and the scale-factor selectors in 4-5 (B) and 29-30 (A).
uint32_t idesc_dense(uint32_t afmt, uint32_t bfmt, int n) {
  return (1u << 4) | (afmt << 7) | (bfmt << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}
uint32_t idesc_block_scaled(uint32_t afmt, uint32_t bfmt, uint32_t e8m0, int n) {
  return (afmt << 7) | (bfmt << 10) | ((uint32_t)(n >> 3) << 17) | (e8m0 << 23) | ((uint32_t)(kBM >> 4) << 24);
}

template <int KIND, int BN, int NACC, bool SFST = false>
lpq_status run(const CUtensorMap& ta, const CUtensorMap& tb, GemmArgs g, cudaStream_t s) {
  using CF = Cfg<KIND, BN, NACC, SFST>;
  lpq_status st = set_smem_attr(reinterpret_cast<const void*>(gemm_kernel<KIND, BN, NACC, SFST>), CF::kSmem);
  if (st != LPQ_OK) return st;
  const int sms = device_sms();
  const int64_t tm = (g.M + kBM - 1) / kBM, tn = (g.N + BN - 1) / BN;
  if (tm * tn > (int64_t)1 << 30) return set_error(LPQ_ERR_SHAPE, "too many output tiles");
  g.tiles_m = (int)tm;
  g.tiles_n = (int)tn;
  const int grid = (int)std::min<int64_t>(tm * tn, sms);
  gemm_kernel<KIND, BN, NACC, SFST><<<grid, kThreadsGemm + (SFST ? 32 * kSfWarps : 0), CF::kSmem, s>>>(ta, tb, g);
  return cuda_check(cudaGetLastError(), "gemm kernel launch");
}


// CTA-pair GEMM (cta_group::2).  A cluster of two CTAs on two SMs computes a
// 256 x 256 output tile: each CTA loads its own 128 rows of A and its own 128
// rows of B (each SM streams half the B bytes of the single-CTA kernel), the
// even CTA issues the pair MMAs, and each CTA's TMEM holds the accumulator
// rows of its half.  A short last round runs its tiles as 256 x 128 halves
// (64 B rows per CTA, N = 128 MMAs; work_coords).  Every A/B load is a TMA tile load that signals the even
// CTA's full barrier; MMA completion is multicast to both CTAs.  For the
// block-scaled kinds each CTA also loads the scale atoms of its A rows and of
// all 256 B rows of the tile (each CTA's accumulator spans every column, so
// each TMEM needs every column's scales: with only its own 128 B rows' scales
// in each CTA the results fail the parity tests).  With scale warps
// (SFST, the default) each CTA's four scale warps write them into the
// stage's TMEM slot with tcgen05.st and report to the even CTA's full
// barrier; otherwise the pair copies (tcgen05.cp.cta_group::2) move them.
constexpr int kPairBN = 256;

template <int KIND, bool SFST = false>
struct PairCfg {
  static constexpr int kSfAtoms = sf_atoms_per_step(KIND);
  static constexpr int kA = kBM * kKBytes;
  static constexpr int kB = (kPairBN / 2) * kKBytes;
  static constexpr int kSfbGroups = 2;  // B scale atoms of both 128-row halves of the tile
  static constexpr int kSfa = kSfAtoms * 512;
  static constexpr int kSfb = kSfAtoms * 512 * kSfbGroups;
  static constexpr int kStage = kA + kB + kSfa + kSfb;
  // Epilogue staging for TMA stores: per epilogue warp one 32 x 64 bf16 tile
  // (128-byte rows, 128-byte swizzle).  The stage ring takes what is left of
  // the 227 KB a CTA can have.
  static constexpr int kStgWarp = 32 * 128;
  static constexpr int kStg = kEpiWarps * kStgWarp;
  static constexpr int kRing = 232448 - 1024 /*align*/ - 512 /*barriers*/ - kStg - 1024 /*staging align*/;
  static constexpr int kStages = kRing / kStage > 8 ? 8 : kRing / kStage;
  static constexpr int kSmem = kStages * kStage + 1024 + 512 + kStg + 1024;
  static constexpr int kNacc = kSfAtoms == 0 ? 2 : 1;
  static constexpr int kSfaCols = kSfAtoms * 4;
  static constexpr int kSfbCols = kSfAtoms * 4 * kSfbGroups;
  static constexpr int kSlots = SFST ? kStages : 1;  // one TMEM scale slot per stage
  static_assert(kNacc * kPairBN + kSlots * (kSfaCols + kSfbCols) <= 512, "TMEM holds 512 columns");
};

template <int KIND>
__device__ __forceinline__ void mma_pair_bs(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  if constexpr (KIND == kKindMXF8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate) : "memory");
  } else if constexpr (KIND == kKindMXF4) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate) : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate) : "memory");
  }
}
__device__ __forceinline__ void tmem_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <int KIND, bool SFST>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsGemm + (SFST ? 32 * kSfWarps : 0))
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmSfa,
                     const __grid_constant__ CUtensorMap tmSfb, const __grid_constant__ CUtensorMap tmC,
                     const GemmArgs g) {
  using PC = PairCfg<KIND, SFST>;
  constexpr int S = PC::kStages, NACC = PC::kNacc;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * PC::kA;
  uint8_t* sSfa = sB + S * PC::kB;
  uint8_t* sSfb = sSfa + S * PC::kSfa;
  uint8_t* stage_c = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(sSfb + S * PC::kSfb) + 1023) & ~uintptr_t(1023));  // epilogue staging
  uint64_t* full = reinterpret_cast<uint64_t*>(stage_c + PC::kStg);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + NACC;
  uint64_t* sfd = acc_empty + NACC;      // [S] (SFST): this CTA's scale atoms landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfd + S);
  uint32_t* peer_base = tmem_slot + 1;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int total = g.items;  // work items: whole tiles, then half tiles

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // SFST: full once the pair's A/B landed and the scale warps of both CTAs
      // have written the stage's scale slot; the MMA commit alone empties it.
      mbar_init(&full[s], SFST ? 1 + 2 * kSfWarps : 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 2 * kEpiWarps);  // the epilogue warps of both CTAs
    }
    for (int s = 0; s < S; ++s) mbar_init(&sfd[s], 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (g.full_tiles < g.items) prefetch_tmap(&tmBh);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Both CTAs must see the same TMEM address; otherwise stop cleanly.
  if (threadIdx.x == 0) st_shared_remote_u32(mapa_shared(smem_u32(peer_base), rank ^ 1u), tmem_base);
  cluster_sync_all();
  if (*peer_base != tmem_base) {
    if (threadIdx.x == 0) atomicCAS(&g_device_error, 0, (int)LPQ_ERR_UNSUPPORTED);
    *abort_flag = 1;
  }
  const bool run = *abort_flag == 0;
  const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
  const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
  const uint32_t tmem_sfa = tmem_base + NACC * kPairBN;
  const uint32_t tmem_sfb = tmem_sfa + PC::kSfaCols;

  if (run && warp == 0) {
    if (lane == 0) {
      const int elem_per_kt = KIND == kKindF16 ? kKBytes / 2 : kKBytes;
      uint32_t s = 0, ph = 0, it = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        int mt, nt, part;
        work_coords(t, g.full_tiles, g.tiles_m, g.tiles_n, mt, nt, part);
        // A half tile (part >= 0) has 128 B rows, 64 in each CTA, and the scale
        // atoms of their one 128-row group (in the first group slot)
        const bool hf = part >= 0;
        const int32_t arow = mt * 256 + (int32_t)rank * 128;
        const int32_t brow = hf ? nt * kPairBN + part * 128 + (int32_t)rank * 64 : nt * kPairBN + (int32_t)rank * 128;
        const uint32_t kb = hf ? PC::kB / 2 : PC::kB;
        const int ngb = hf ? 1 : PC::kSfbGroups;
        const uint32_t ksfb = (uint32_t)ngb * PC::kSfAtoms * 512;
        for (int kt = 0; kt < g.num_k; ++kt) {
          if (!(ok = mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag, &g_device_error))) break;
          if (leader) mbar_arrive_expect_tx(&full[s], SFST ? 2 * (PC::kA + kb) : 2 * (PC::kA + kb + PC::kSfa + ksfb));
          const uint32_t fb = full_leader + 8 * s;
          if constexpr (PC::kSfAtoms > 0) {
            // scale atoms: rows of a 2D map are 512-byte atoms (128 x u32).  With
            // scale warps they land on this CTA's own barrier (its scale warps
            // read them); otherwise on the even CTA's full barrier (pair copies).
            const int32_t ga = mt * 2 + (int32_t)rank;
            if constexpr (SFST) mbar_arrive_expect_tx(&sfd[s], PC::kSfa + ksfb);
            const int32_t ya = (int32_t)(ga * g.sfa_kt + kt * PC::kSfAtoms);
            if constexpr (SFST) tma_load_2d(sSfa + s * PC::kSfa, &tmSfa, 0, ya, &sfd[s]);
            else tma_load_2d_pair(sSfa + s * PC::kSfa, &tmSfa, 0, ya, fb);
#pragma unroll
            for (int i = 0; i < PC::kSfbGroups; ++i) {
              if (i >= ngb) break;
              int64_t gb = hf ? (int64_t)nt * 2 + part : (int64_t)nt * 2 + i;
              if (gb >= g.sfb_groups) gb = g.sfb_groups - 1;
              const int32_t yb = (int32_t)(gb * g.sfb_kt + kt * PC::kSfAtoms);
              if constexpr (SFST) tma_load_2d(sSfb + s * PC::kSfb + i * PC::kSfAtoms * 512, &tmSfb, 0, yb, &sfd[s]);
              else tma_load_2d_pair(sSfb + s * PC::kSfb + i * PC::kSfAtoms * 512, &tmSfb, 0, yb, fb);
            }
          }
          tma_load_2d_pair(sA + s * PC::kA, &tmA, kt * elem_per_kt, arow, fb);
          tma_load_2d_pair(sB + s * PC::kB, hf ? &tmBh : &tmB, kt * elem_per_kt, brow, fb);
          ++it;
          if (++s == (uint32_t)S) { s = 0; ph ^= 1u; }
        }
      }
      // After an abort, the even CTA lets the pair's loads in flight land
      // (they all signal its full barriers) before either CTA exits.
      if (!ok && leader) drain_stages(full, S, it > (uint32_t)S ? it - S : 0u, it);
    }
  } else if (run && warp == 1) {
    if (lane == 0 && leader) {
      const uint32_t kHiSw = (uint32_t)(smem_desc(0, 16, 1024, 2) >> 32);
      const uint32_t kHiSf = (uint32_t)(smem_desc(0, 0, 128, 0) >> 32);
      const uint32_t a0 = (uint32_t)smem_desc(smem_u32(sA), 16, 1024, 2);
      const uint32_t b0 = (uint32_t)smem_desc(smem_u32(sB), 16, 1024, 2);
      const uint32_t fa0 = smem_u32(sSfa) >> 4, fb0 = smem_u32(sSfb) >> 4;
      uint32_t s = 0, ph = 0, lt = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs, ++lt) {
        const uint32_t a = lt % NACC, aph = (lt / NACC) & 1u;
        const uint32_t idesc = t < g.full_tiles ? g.idesc : g.idesc_half;  // N = 256 or 128
        if (!(ok = mbar_wait_bounded(&acc_empty[a], aph ^ 1u, abort_flag, &g_device_error))) break;
        tc_fence_after();
        const uint32_t tmem_d = tmem_base + a * kPairBN;
        for (int kt = 0; kt < g.num_k; ++kt) {
          if (!(ok = mbar_wait_bounded(&full[s], ph, abort_flag, &g_device_error))) break;
          tc_fence_after();
          const uint32_t alo = a0 + s * (PC::kA >> 4), blo = b0 + s * (PC::kB >> 4);
          const uint32_t falo = fa0 + s * (PC::kSfa >> 4), fblo = fb0 + s * (PC::kSfb >> 4);
          if constexpr (KIND == kKindMXF8 && !SFST) {
            tmem_cp_sf_pair(tmem_sfa, ((uint64_t)kHiSf << 32) | falo);
#pragma unroll
            for (int i = 0; i < PC::kSfbGroups; ++i)
              tmem_cp_sf_pair(tmem_sfb + 4 * i, ((uint64_t)kHiSf << 32) | (fblo + i * 32));
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t ad = ((uint64_t)kHiSw << 32) | (alo + 2 * j);
            const uint64_t bd = ((uint64_t)kHiSw << 32) | (blo + 2 * j);
            const uint32_t acc = (kt > 0 || j > 0) ? 1u : 0u;
            if constexpr (KIND == kKindF16 || KIND == kKindF8F6F4) {
              mma_pair<KIND>(tmem_d, ad, bd, idesc, acc);
            } else if constexpr (KIND == kKindMXF8 && !SFST) {
              mma_pair_bs<KIND>(tmem_d, ad, bd, idesc | ((uint32_t)j << 4) | ((uint32_t)j << 29), tmem_sfa, tmem_sfb,
                                acc);
            } else if constexpr (SFST) {
              const int at = j * PC::kSfAtoms / 4;  // the MMA's scale atom
              const uint32_t base = tmem_sfa + s * (PC::kSfaCols + PC::kSfbCols);  // the stage's slot
              mma_pair_bs<KIND>(tmem_d, ad, bd, idesc | sf_select<KIND>(j), base + 4 * at,
                                base + PC::kSfaCols + 4 * PC::kSfbGroups * at, acc);
            } else {
              const int at = j * PC::kSfAtoms / 4;
              if ((j * PC::kSfAtoms) % 4 == 0) {  // first MMA of the atom: copy it
                tmem_cp_sf_pair(tmem_sfa + 4 * at, ((uint64_t)kHiSf << 32) | (falo + at * 32));
#pragma unroll
                for (int i = 0; i < PC::kSfbGroups; ++i)
                  tmem_cp_sf_pair(tmem_sfb + 4 * PC::kSfbGroups * at + 4 * i,
                                  ((uint64_t)kHiSf << 32) | (fblo + (i * PC::kSfAtoms + at) * 32));
              }
              mma_pair_bs<KIND>(tmem_d, ad, bd, idesc | sf_select<KIND>(j), tmem_sfa + 4 * at,
                                tmem_sfb + 4 * PC::kSfbGroups * at, acc);
            }
          }
          tc_commit_pair(&empty[s], 0x3);
          if (++s == (uint32_t)S) { s = 0; ph ^= 1u; }
        }
        if (ok) tc_commit_pair(&acc_full[a], 0x3);
      }
    }
  } else if (run && SFST && warp >= 2 + kEpiWarps) {
    if constexpr (SFST) {  // only kernels with scale warps carry this code
      // scale warps: this CTA's lane quarter of the step's scale atoms (its own A
      // rows, all 256 B rows) from shared memory into the TMEM slot; both CTAs'
      // scale warps report to the even CTA's slot barrier
      const int q = warp & 3;
      const uint32_t lanes = (uint32_t)(q * 32) << 16;
      uint32_t s = 0, ph = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        for (int kt = 0; kt < g.num_k; ++kt) {
          if (!(ok = mbar_wait_bounded(&sfd[s], ph, abort_flag, &g_device_error))) break;  // own scale atoms
          if (!(ok = mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag, &g_device_error))) break;  // slot free
          __syncwarp();
          tc_fence_after();
          constexpr int NA = PC::kSfAtoms, G = PC::kSfbGroups;
          const uint4* fa = reinterpret_cast<const uint4*>(sSfa + s * PC::kSfa) + lane;
          const uint4* fb = reinterpret_cast<const uint4*>(sSfb + s * PC::kSfb) + lane;
          uint32_t va[4 * NA], vb[4 * NA * G];
#pragma unroll
          for (int j = 0; j < NA; ++j) {
            const uint4 x = fa[j * 32];
            va[4 * j] = x.x; va[4 * j + 1] = x.y; va[4 * j + 2] = x.z; va[4 * j + 3] = x.w;
#pragma unroll
            for (int i = 0; i < G; ++i) {
              const uint4 y = fb[(i * NA + j) * 32];
              const int c = 4 * G * j + 4 * i;
              vb[c] = y.x; vb[c + 1] = y.y; vb[c + 2] = y.z; vb[c + 3] = y.w;
            }
          }
          const uint32_t base = tmem_sfa + s * (PC::kSfaCols + PC::kSfbCols) + lanes;
          tmem_st_cols(base, va);
          tmem_st_cols(base + PC::kSfaCols, vb);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(&full[s]); else mbar_arrive_remote_relaxed(full_leader + 8 * s);
          }
          if (++s == (uint32_t)S) { s = 0; ph ^= 1u; }
        }
      }
    }  // SFST
  } else if (run && warp >= 2) {
    constexpr int HALF = kPairBN / 2;
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    float alpha = 1.0f;
    if (g.alpha_a) alpha = *g.alpha_a;
    if (g.alpha_b) alpha = __fmul_rn(alpha, *g.alpha_b);
    const bool vec_ok = g.c_fp32 ? (g.N % 4 == 0) : (g.N % 8 == 0);
    uint32_t lt = 0;
    for (int t = pair; t < total; t += npairs, ++lt) {
      int mt, nt, part;
      work_coords(t, g.full_tiles, g.tiles_m, g.tiles_n, mt, nt, part);
      // columns of this warp: 128 of a whole tile, 64 of a half tile (part >= 0)
      const int width = part >= 0 ? HALF / 2 : HALF;
      const uint32_t a = lt % NACC, aph = (lt / NACC) & 1u;
      if (!mbar_wait_bounded(&acc_full[a], aph, abort_flag, &g_device_error)) break;
      __syncwarp();
      tc_fence_after();
      const int64_t row = (int64_t)mt * 256 + rank * 128 + q * 32 + lane;
      const int64_t c0 = (int64_t)nt * kPairBN + (part >= 0 ? part * 128 : 0) + half * width;
      const int64_t ncols = g.N - c0;
      const uint32_t tbase = tmem_base + a * kPairBN + half * width + ((uint32_t)(q * 32) << 16);
      if (!g.c_fp32) {
        uint32_t pk[HALF / 2];
#pragma unroll
        for (int cc = 0; cc < HALF / 32; ++cc) {
          if (cc * 32 >= width) break;
          uint32_t v[32];
          tmem_ld32(tbase + (uint32_t)(cc * 32), v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            // one packed two-wide multiply (each half rounded like __fmul_rn), one packed convert
            const float2 y = __fmul2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                        make_float2(alpha, alpha));
            __nv_bfloat162 h = __floats2bfloat162_rn(y.x, y.y);
            pk[cc * 16 + i] = *reinterpret_cast<uint32_t*>(&h);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&acc_empty[a]); else mbar_arrive_remote_relaxed(acc_empty_leader + 8 * a);
        }
        if (g.c_tma) {
          // The warp's 32 rows x 128 columns (64 of a half tile) leave as TMA
          // stores of 32 x 64 tiles staged in shared memory (128-byte swizzle:
          // 16-byte chunk i of row r at chunk position i ^ (r & 7)); the
          // stores clip at M and N.
          uint8_t* stg = stage_c + (warp - 2) * PC::kStgWarp;
          const int32_t y = mt * 256 + (int32_t)rank * 128 + q * 32;
#pragma unroll
          for (int ch = 0; ch < 2; ++ch) {
            if (ch * 64 >= width) break;
            if (lane == 0) bulk_wait_group_read0();  // the previous store has read the buffer
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(stg + lane * 128 + ((i ^ (lane & 7)) << 4)) =
                  make_uint4(pk[32 * ch + 4 * i], pk[32 * ch + 4 * i + 1], pk[32 * ch + 4 * i + 2],
                             pk[32 * ch + 4 * i + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, stg, (int32_t)(c0 + ch * 64), y);
              bulk_commit_group();
            }
          }
          continue;
        }
        if (row < g.M && ncols > 0) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(g.c) + row * g.N + c0;
          const int64_t nc = ncols < width ? ncols : width;
          if (vec_ok && nc == width) {
#pragma unroll
            for (int i = 0; i < HALF / 8; ++i) {
              if (i * 8 >= width) break;
              reinterpret_cast<uint4*>(out)[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < HALF / 2; ++i) {
              if (2 * i < nc) out[2 * i] = __ushort_as_bfloat16((unsigned short)(pk[i] & 0xFFFFu));
              if (2 * i + 1 < nc) out[2 * i + 1] = __ushort_as_bfloat16((unsigned short)(pk[i] >> 16));
            }
          }
        }
        continue;
      }
#pragma unroll 1
      for (int cc = 0; cc < width / 32; ++cc) {
        uint32_t v[32];
        tmem_ld32(tbase + (uint32_t)(cc * 32), v);
        if (cc == width / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (leader) mbar_arrive(&acc_empty[a]); else mbar_arrive_remote_relaxed(acc_empty_leader + 8 * a);
          }
        }
        const int64_t col0 = c0 + cc * 32;
        if (row >= g.M || col0 >= g.N) continue;
        float* out = static_cast<float*>(g.c) + row * g.N + col0;
        if (vec_ok && col0 + 32 <= g.N) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(out)[i] = make_float4(
                __fmul_rn(__uint_as_float(v[4 * i]), alpha), __fmul_rn(__uint_as_float(v[4 * i + 1]), alpha),
                __fmul_rn(__uint_as_float(v[4 * i + 2]), alpha), __fmul_rn(__uint_as_float(v[4 * i + 3]), alpha));
        } else {
          for (int i = 0; i < 32 && col0 + i < g.N; ++i) out[i] = __fmul_rn(__uint_as_float(v[i]), alpha);
        }
      }
    }
    if (lane == 0) bulk_wait_group0();  // this warp's TMA stores complete before the CTA exits
    __syncwarp();
  }
  tc_fence_before();
  cluster_sync_all();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// 2D map over a scale array in the tensor-core layout: rows are 512-byte
// atoms (128 x u32), a box is `atoms` consecutive atoms.
lpq_status make_sf_map(CUtensorMap* map, const void* base, int64_t total_atoms, uint32_t atoms) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return set_error(LPQ_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
  cuuint64_t dims[2] = {128, (cuuint64_t)(total_atoms > 0 ? total_atoms : 1)};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, atoms};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(LPQ_ERR_CUDA, "cuTensorMapEncodeTiled (scales) failed (%d)", (int)r);
  return LPQ_OK;
}

template <int KIND, bool SFST = false>
lpq_status run_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tbh, const CUtensorMap& tsa,
                    const CUtensorMap& tsb, GemmArgs g, bool direct_store, bool whole_tiles, cudaStream_t s) {
  using PC = PairCfg<KIND, SFST>;
  lpq_status st = set_smem_attr(reinterpret_cast<const void*>(gemm_pair_kernel<KIND, SFST>), PC::kSmem);
  if (st != LPQ_OK) return st;
  const int sms = device_sms();
  const int64_t tm = (g.M + 255) / 256, tn = (g.N + kPairBN - 1) / kPairBN;
  if (tm * tn > (int64_t)1 << 29) return set_error(LPQ_ERR_SHAPE, "too many output tiles");
  g.tiles_m = (int)tm;
  g.tiles_n = (int)tn;
  // Persistent schedule over work items: whole tiles, and, when the tiles of
  // the last round fill at most half of the pairs, those tiles as two
  // 256 x 128 halves each (the round then takes half as long).
  const int64_t total = tm * tn, P = std::max(1, sms / 2);
  const int64_t rem = total - ((total - 1) / P) * P;  // tiles in the last round, 1 .. P
  const bool split = !whole_tiles && 2 * rem <= P;
  g.full_tiles = (int)(split ? total - rem : total);
  g.items = (int)(split ? total + rem : total);
  g.idesc_half = (g.idesc & ~(63u << 17)) | ((uint32_t)(128 >> 3) << 17);
  const int pairs = (int)std::min<int64_t>(g.items, P);
  // bf16 C leaves through TMA tile stores (32 x 64 boxes) when its row pitch
  // allows a tensor map (N % 8 == 0); otherwise the epilogue stores directly.
  CUtensorMap tc = ta;
  g.c_tma = 0;
  if (!g.c_fp32 && g.N % 8 == 0 && !direct_store) {
    if ((st = make_map(&tc, g.c, true, g.N, g.M, g.N * 2, 64, 32)) != LPQ_OK) return st;
    g.c_tma = 1;
  }
  gemm_pair_kernel<KIND, SFST>
      <<<2 * pairs, kThreadsGemm + (SFST ? 32 * kSfWarps : 0), PC::kSmem, s>>>(ta, tb, tbh, tsa, tsb, tc, g);
  return cuda_check(cudaGetLastError(), "pair gemm launch");
}

// Sub-channel FP8 GEMM ("Faster training throughput in FP8 with NVIDIA NeMo",
// sub-channel scaling: 1x128 activation and 128x128 weight blocks with FP32
// factors).  Every 128-deep K slice is one pipeline stage: the MMA warp
// computes the slice's partial product sum_{k in slice} qa * qb with
// kind::f8f6f4 into one of four TMEM buffers; the epilogue warps read it and
// accumulate partial * sa[m, slice] * sb[n, slice] in FP32 registers (the
// tensor cores have no FP32 block scales), while the next slice runs.
struct BlockArgs {
  const float* sa;  // A factors: 1x128 -> [K/128][M]; 128x128 -> [ceil(M/128)][K/128]
  const float* sb;  // B factors, same convention with N
  int a_rows, b_rows;  // block rows: 1 or 128
  void* c;
  int64_t M, N, K;
  int c_fp32;
  uint32_t idesc;
  int num_k;
  int tiles_m, tiles_n;
};

constexpr int kBlkBN = 128;
constexpr int kBlkStages = 6;
constexpr int kBlkBufs = 4;   // TMEM partial buffers (4 x 128 columns): the MMA warp runs up to 3 slices ahead
constexpr int kBlkStage = kBM * kKBytes + kBlkBN * kKBytes;
constexpr int kBlkEpiWarps = 8;  // two per TMEM lane quarter, 64 columns each
// Shared-memory ring of the block factors of the slices in flight, filled by
// the factor warp: per slice the tile's 128 A factors (one per row) and 128 B
// factors (one per column).
constexpr int kBlkFacSlots = 8;
constexpr int kBlkFacSlot = 2 * 128;
constexpr int kBlkSmem = kBlkStages * kBlkStage + 1024 + 512 + kBlkFacSlots * kBlkFacSlot * 4;
constexpr int kBlkFacWarp = 2 + kBlkEpiWarps;  // the last warp
constexpr int kBlkThreads = 32 * (kBlkFacWarp + 1);

__global__ void __launch_bounds__(kBlkThreads, 1)
    block_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const BlockArgs g) {
  constexpr int S = kBlkStages, BN = kBlkBN, HALF = BN / 2, NB = kBlkBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * kBM * kKBytes;
  float* s_fac = reinterpret_cast<float*>(sB + S * BN * kKBytes);  // [kBlkFacSlots][128 A, 128 B factors]
  uint64_t* full = reinterpret_cast<uint64_t*>(s_fac + kBlkFacSlots * kBlkFacSlot);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;   // [NB]
  uint64_t* acc_empty = acc_full + NB;
  uint64_t* fac_full = acc_empty + NB;  // [kBlkFacSlots]: the slot's factor copies landed
  uint64_t* fac_empty = fac_full + kBlkFacSlots;  // the epilogue warps are done with the slot
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fac_empty + kBlkFacSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = g.tiles_m * g.tiles_n;
  const int64_t KB = g.K / 128;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < NB; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kBlkEpiWarps);
    }
    for (int f = 0; f < kBlkFacSlots; ++f) {
      mbar_init(&fac_full[f], 32);  // one arrival per lane of the factor warp, when its copies land
      mbar_init(&fac_empty[f], kBlkEpiWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, NB * BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int mt, nt;
        tile_coords(t, g.tiles_m, g.tiles_n, mt, nt);
        for (int kt = 0; kt < g.num_k; ++kt, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1u;
          if (!(ok = mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag, &g_device_error))) break;
          mbar_arrive_expect_tx(&full[s], kBlkStage);
          tma_load_2d(sA + s * kBM * kKBytes, &tmA, kt * kKBytes, mt * kBM, &full[s]);
          tma_load_2d(sB + s * BN * kKBytes, &tmB, kt * kKBytes, nt * BN, &full[s]);
        }
      }
      // After an abort, let the loads still in flight land before the CTA exits.
      if (!ok) drain_stages(full, S, it > (uint32_t)S ? it - S : 0u, it);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t kHiSw = (uint32_t)(smem_desc(0, 16, 1024, 2) >> 32);
      const uint32_t a0 = (uint32_t)smem_desc(smem_u32(sA), 16, 1024, 2);
      const uint32_t b0 = (uint32_t)smem_desc(smem_u32(sB), 16, 1024, 2);
      uint32_t s = 0, ph = 0, slice = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        for (int kt = 0; kt < g.num_k; ++kt, ++slice) {
          const uint32_t a = slice % NB, aph = (slice / NB) & 1u;
          if (!(ok = mbar_wait_bounded(&acc_empty[a], aph ^ 1u, abort_flag, &g_device_error))) break;
          if (!(ok = mbar_wait_bounded(&full[s], ph, abort_flag, &g_device_error))) break;
          tc_fence_after();
          const uint32_t alo = a0 + s * (kBM * kKBytes >> 4), blo = b0 + s * (BN * kKBytes >> 4);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mma_ss<kKindF8F6F4>(tmem_base + a * BN, ((uint64_t)kHiSw << 32) | (alo + 2 * j),
                                ((uint64_t)kHiSw << 32) | (blo + 2 * j), g.idesc, j > 0 ? 1u : 0u);
          tc_commit(&empty[s]);
          tc_commit(&acc_full[a]);
          if (++s == (uint32_t)S) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp == kBlkFacWarp) {
    // Factor warp: for every slice, the tile's 128 A factors (1x128: its rows';
    // 128x128: the block's, repeated) and 128 B factors (1x128: its columns';
    // 128x128: the block's, repeated) into the slice's ring slot with cp.async,
    // zeros past the matrix.  Each lane's copies arrive on the slot's full
    // barrier when they land, so the warp never waits for a load; it runs up to
    // kBlkFacSlots slices ahead of the epilogue.
    uint32_t slice = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      int mt, nt;
      tile_coords(t, g.tiles_m, g.tiles_n, mt, nt);
      for (int kt = 0; kt < g.num_k; ++kt, ++slice) {
        const uint32_t f = slice % kBlkFacSlots, fph = (slice / kBlkFacSlots) & 1u;
        if (!(ok = mbar_wait_bounded(&fac_empty[f], fph ^ 1u, abort_flag, &g_device_error))) break;
        float* slot = s_fac + f * kBlkFacSlot;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = 4 * lane + i;
          const int64_t row = (int64_t)mt * kBM + j, col = (int64_t)nt * BN + j;
          const bool va = g.a_rows != 1 || row < g.M, vb = g.b_rows != 1 || col < g.N;
          const float* pa = g.a_rows == 1 ? g.sa + (va ? (int64_t)kt * g.M + row : 0) : g.sa + (int64_t)mt * KB + kt;
          const float* pb = g.b_rows == 1 ? g.sb + (vb ? (int64_t)kt * g.N + col : 0)
                                          : g.sb + (int64_t)(nt * BN / 128) * KB + kt;
          cp_async4(slot + j, pa, va);
          cp_async4(slot + 128 + j, pb, vb);
        }
        cp_async_arrive_noinc(&fac_full[f]);
      }
    }
    cp_async_wait_all();  // no copy is still in flight when the CTA exits
  } else {
    // Epilogue: per 128-deep slice, acc += partial * fa[row] * fb[col] in FP32
    // registers, with the slice's factors from the factor warp's ring slot.
    const int ew = warp - 2;          // 0..7
    const int q = warp & 3;           // TMEM lane quarter
    const int half = ew >> 2;         // column half of the tile
    const bool vec_ok = g.c_fp32 ? (g.N % 4 == 0) : (g.N % 8 == 0);
    uint32_t slice = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      int mt, nt;
      tile_coords(t, g.tiles_m, g.tiles_n, mt, nt);
      const int64_t row = (int64_t)mt * kBM + q * 32 + lane;
      const int64_t n0 = (int64_t)nt * BN;
      float2 acc[HALF / 2];  // column pairs: the promotion runs as packed two-wide FMAs
#pragma unroll
      for (int i = 0; i < HALF / 2; ++i) acc[i] = make_float2(0.f, 0.f);
      for (int kt = 0; kt < g.num_k; ++kt, ++slice) {
        const uint32_t a = slice % NB, aph = (slice / NB) & 1u;
        const uint32_t f = slice % kBlkFacSlots, fph = (slice / kBlkFacSlots) & 1u;
        if (!(ok = mbar_wait_bounded(&fac_full[f], fph, abort_flag, &g_device_error))) break;
        const float* slot = s_fac + f * kBlkFacSlot;
        const float fa = slot[q * 32 + lane];          // this thread's row
        const float* sbs = slot + 128 + half * HALF;   // the warp's 64 columns (128x128: all equal)
        if (!(ok = mbar_wait_bounded(&acc_full[a], aph, abort_flag, &g_device_error))) break;
        __syncwarp();
        tc_fence_after();
        const uint32_t tb = tmem_base + a * BN + half * HALF + ((uint32_t)(q * 32) << 16);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t v[32];
          tmem_ld32(tb + 32 * cc, v);
          if (cc == 1) {  // slice fully read: the MMA warp may reuse this buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[a]);
          }
          if (g.b_rows == 1) {
#pragma unroll
            for (int i4 = 0; i4 < 8; ++i4) {
              const float4 f4 = *reinterpret_cast<const float4*>(sbs + 32 * cc + 4 * i4);  // broadcast
              // row factor x the four columns' factors, then acc += partial x factor (packed)
              const float2 w01 = __fmul2_rn(make_float2(fa, fa), make_float2(f4.x, f4.y));
              const float2 w23 = __fmul2_rn(make_float2(fa, fa), make_float2(f4.z, f4.w));
              const int i = 4 * i4;
              float2& a01 = acc[16 * cc + 2 * i4];
              float2& a23 = acc[16 * cc + 2 * i4 + 1];
              a01 = __ffma2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), w01, a01);
              a23 = __ffma2_rn(make_float2(__uint_as_float(v[i + 2]), __uint_as_float(v[i + 3])), w23, a23);
            }
          } else {
            const float f = fa * sbs[0];
            const float2 w = make_float2(f, f);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              acc[16 * cc + i] = __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), w,
                                            acc[16 * cc + i]);
          }
        }
        __syncwarp();  // every lane is done with the slot
        if (lane == 0) mbar_arrive(&fac_empty[f]);
      }
      if (!ok || row >= g.M) continue;
      const int64_t c0 = n0 + half * HALF;
      const int64_t ncols = g.N - c0;
      if (ncols <= 0) continue;
      if (g.c_fp32) {
        float* out = static_cast<float*>(g.c) + row * g.N + c0;
        if (vec_ok && ncols >= HALF) {
#pragma unroll
          for (int i = 0; i < HALF / 4; ++i)
            reinterpret_cast<float4*>(out)[i] = make_float4(acc[2 * i].x, acc[2 * i].y, acc[2 * i + 1].x, acc[2 * i + 1].y);
        } else {
#pragma unroll
          for (int i = 0; i < HALF / 2; ++i) {
            if (2 * i < ncols) out[2 * i] = acc[i].x;
            if (2 * i + 1 < ncols) out[2 * i + 1] = acc[i].y;
          }
        }
      } else {
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(g.c) + row * g.N + c0;
        if (vec_ok && ncols >= HALF) {
#pragma unroll
          for (int i = 0; i < HALF / 8; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              __nv_bfloat162 h = __floats2bfloat162_rn(acc[4 * i + j].x, acc[4 * i + j].y);
              w[j] = *reinterpret_cast<uint32_t*>(&h);
            }
            reinterpret_cast<uint4*>(out)[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < HALF / 2; ++i) {
            if (2 * i < ncols) out[2 * i] = __float2bfloat16_rn(acc[i].x);
            if (2 * i + 1 < ncols) out[2 * i + 1] = __float2bfloat16_rn(acc[i].y);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, NB * BN);
  }
}

lpq_status run_block_gemm(const CUtensorMap& ta, const CUtensorMap& tb, BlockArgs g, cudaStream_t s) {
  lpq_status st = set_smem_attr(reinterpret_cast<const void*>(block_gemm_kernel), kBlkSmem);
  if (st != LPQ_OK) return st;
  const int sms = device_sms();
  const int64_t tm = (g.M + kBM - 1) / kBM, tn = (g.N + kBlkBN - 1) / kBlkBN;
  g.tiles_m = (int)tm;
  g.tiles_n = (int)tn;
  const int grid = (int)std::min<int64_t>(tm * tn, sms);
  block_gemm_kernel<<<grid, kBlkThreads, kBlkSmem, s>>>(ta, tb, g);
  return cuda_check(cudaGetLastError(), "block gemm launch");
}

}  // namespace

lpq_status launch_gemm(const lpq_qview* a, const lpq_qview* b, void* c, int32_t c_is_fp32, int64_t m, int64_t n,
                       int64_t k, const lpq_gemm_opts* opts, cudaStream_t s) {
  if (m == 0 || n == 0) return LPQ_OK;
  const int32_t fa = a->fmt, fb = b->fmt;
  GemmArgs g{};
  g.c = c;
  g.M = m;
  g.N = n;
  g.K = k;
  g.c_fp32 = c_is_fp32;
  if (k == 0) {
    // Empty reduction: C = 0.
    size_t bytes = (size_t)m * (size_t)n * (c_is_fp32 ? 4 : 2);
    return cuda_check(cudaMemsetAsync(c, 0, bytes, s), "cudaMemsetAsync(C)");
  }
  CUtensorMap ta, tb;
  lpq_status st;
  constexpr int BN = 256;
  // Kernel path (lpq_gemm_opts; NULL = the defaults): CTA pairs per 256 x 256
  // tile whenever M >= 256, else one CTA per 128 x 256 tile; block-scaled
  // scales written into TMEM by the scale warps; bf16 C through TMA stores.
  const bool pair_ok = !(opts && opts->single_cta) && m >= 256;
  const int nv_bn = (opts && opts->tile_n == 128) ? 128 : 256;
  const bool cp = opts && opts->scale_copies;
  const bool direct = opts && opts->direct_store;
  const bool whole = opts && opts->whole_tiles;
  CUtensorMap tbh;  // CTA-pair kernel: B boxes of 64 rows for the half tiles
  if (fa == LPQ_BF16) {
    g.num_k = (int)((k * 2 + kKBytes - 1) / kKBytes);
    if ((st = make_map(&ta, a->codes, true, k, m, k * 2, 64, kBM)) != LPQ_OK) return st;
    if ((st = make_map(&tb, b->codes, true, k, n, k * 2, 64, BN)) != LPQ_OK) return st;
    g.idesc = idesc_dense(1, 1, BN);  // BF16 x BF16 -> F32
    if (pair_ok) {
      if ((st = make_map(&ta, a->codes, true, k, m, k * 2, 64, kBM)) != LPQ_OK) return st;
      if ((st = make_map(&tb, b->codes, true, k, n, k * 2, 64, kPairBN / 2)) != LPQ_OK) return st;
      if ((st = make_map(&tbh, b->codes, true, k, n, k * 2, 64, kPairBN / 4)) != LPQ_OK) return st;
      g.idesc = idesc_dense(1, 1, kPairBN) & ~(31u << 24) | (16u << 24);  // M = 256
      return run_pair<kKindF16>(ta, tb, tbh, ta, tb, g, direct, whole, s);
    }
    return run<kKindF16, BN, 2>(ta, tb, g, s);
  }
  if (fa == LPQ_FP8_E4M3 || fa == LPQ_FP8_E5M2) {
    g.num_k = (int)((k + kKBytes - 1) / kKBytes);
    if ((st = make_map(&ta, a->codes, false, k, m, k, 128, kBM)) != LPQ_OK) return st;
    if ((st = make_map(&tb, b->codes, false, k, n, k, 128, BN)) != LPQ_OK) return st;
    g.idesc = idesc_dense(fa == LPQ_FP8_E5M2 ? 1 : 0, fb == LPQ_FP8_E5M2 ? 1 : 0, BN);
    g.alpha_a = a->tensor_scale;
    g.alpha_b = b->tensor_scale;
    if (pair_ok) {
      if ((st = make_map(&tb, b->codes, false, k, n, k, 128, kPairBN / 2)) != LPQ_OK) return st;
      if ((st = make_map(&tbh, b->codes, false, k, n, k, 128, kPairBN / 4)) != LPQ_OK) return st;
      g.idesc = (g.idesc & ~(31u << 24)) | (16u << 24);  // M = 256
      return run_pair<kKindF8F6F4>(ta, tb, tbh, ta, tb, g, direct, whole, s);
    }
    return run<kKindF8F6F4, BN, 2>(ta, tb, g, s);
  }
  if (fa == LPQ_MXFP8 || fa == LPQ_MXFP8_E5M2) {
    // E4M3 (format 0) or E5M2 (format 1) elements on either side, E8M0 scales
    const uint32_t af = fa == LPQ_MXFP8_E5M2 ? 1 : 0, bf = fb == LPQ_MXFP8_E5M2 ? 1 : 0;
    g.num_k = (int)((k + kKBytes - 1) / kKBytes);
    if ((st = make_map(&ta, a->codes, false, k, m, k, 128, kBM)) != LPQ_OK) return st;
    if ((st = make_map(&tb, b->codes, false, k, n, k, 128, BN)) != LPQ_OK) return st;
    g.idesc = idesc_block_scaled(af, bf, 1, BN);
    g.sfa = static_cast<const uint8_t*>(a->scales);
    g.sfb = static_cast<const uint8_t*>(b->scales);
    g.sfa_kt = sf_kt_atoms(LPQ_MXFP8, k);
    g.sfb_kt = g.sfa_kt;
    g.sfb_groups = sf_row_groups(n);
    // scale atoms into TMEM by the scale warps (tcgen05.st), or (scale_copies)
    // tcgen05.cp by the MMA thread
    if (pair_ok) {
      CUtensorMap tsa, tsb;
      if ((st = make_map(&tb, b->codes, false, k, n, k, 128, kPairBN / 2)) != LPQ_OK) return st;
      if ((st = make_map(&tbh, b->codes, false, k, n, k, 128, kPairBN / 4)) != LPQ_OK) return st;
      if ((st = make_sf_map(&tsa, g.sfa, sf_row_groups(m) * g.sfa_kt, 1)) != LPQ_OK) return st;
      if ((st = make_sf_map(&tsb, g.sfb, g.sfb_groups * g.sfb_kt, 1)) != LPQ_OK) return st;
      g.idesc = (g.idesc & ~(31u << 24)) | (16u << 24);
      if (cp) return run_pair<kKindMXF8>(ta, tb, tbh, tsa, tsb, g, direct, whole, s);
      return run_pair<kKindMXF8, true>(ta, tb, tbh, tsa, tsb, g, direct, whole, s);
    }
    if (nv_bn == 128) {
      if ((st = make_map(&tb, b->codes, false, k, n, k, 128, 128)) != LPQ_OK) return st;
      g.idesc = idesc_block_scaled(af, bf, 1, 128);
      if (cp) return run<kKindMXF8, 128, 2>(ta, tb, g, s);
      return run<kKindMXF8, 128, 2, true>(ta, tb, g, s);
    }
    if (cp) return run<kKindMXF8, BN, 1>(ta, tb, g, s);
    return run<kKindMXF8, BN, 1, true>(ta, tb, g, s);
  }
  if (fa == LPQ_MXFP4) {
    // packed E2M1 (format 1) with an E8M0 scale per 32 values: two scales per
    // K = 64 MMA, two atoms per 256-value k-step; the scale warps write them
    // into TMEM as for NVFP4 (scale_copies: tcgen05.cp by the MMA thread)
    g.num_k = (int)((k / 2 + kKBytes - 1) / kKBytes);
    if ((st = make_map(&ta, a->codes, false, k / 2, m, k / 2, 128, kBM)) != LPQ_OK) return st;
    if ((st = make_map(&tb, b->codes, false, k / 2, n, k / 2, 128, BN)) != LPQ_OK) return st;
    g.idesc = idesc_block_scaled(1, 1, 1, BN);
    g.sfa = static_cast<const uint8_t*>(a->scales);
    g.sfb = static_cast<const uint8_t*>(b->scales);
    g.sfa_kt = sf_kt_atoms(LPQ_MXFP4, k);
    g.sfb_kt = g.sfa_kt;
    g.sfb_groups = sf_row_groups(n);
    if (pair_ok) {
      CUtensorMap tsa, tsb;
      if ((st = make_map(&tb, b->codes, false, k / 2, n, k / 2, 128, kPairBN / 2)) != LPQ_OK) return st;
      if ((st = make_map(&tbh, b->codes, false, k / 2, n, k / 2, 128, kPairBN / 4)) != LPQ_OK) return st;
      if ((st = make_sf_map(&tsa, g.sfa, sf_row_groups(m) * g.sfa_kt, 2)) != LPQ_OK) return st;
      if ((st = make_sf_map(&tsb, g.sfb, g.sfb_groups * g.sfb_kt, 2)) != LPQ_OK) return st;
      g.idesc = (g.idesc & ~(31u << 24)) | (16u << 24);
      if (cp) return run_pair<kKindMXF4>(ta, tb, tbh, tsa, tsb, g, direct, whole, s);
      return run_pair<kKindMXF4, true>(ta, tb, tbh, tsa, tsb, g, direct, whole, s);
    }
    if (nv_bn == 128) {
      if ((st = make_map(&tb, b->codes, false, k / 2, n, k / 2, 128, 128)) != LPQ_OK) return st;
      g.idesc = idesc_block_scaled(1, 1, 1, 128);
      if (cp) return run<kKindMXF4, 128, 2>(ta, tb, g, s);
      return run<kKindMXF4, 128, 2, true>(ta, tb, g, s);
    }
    if (cp) return run<kKindMXF4, BN, 1>(ta, tb, g, s);
    return run<kKindMXF4, BN, 1, true>(ta, tb, g, s);
  }
  if (fa == LPQ_NVFP4 || fa == LPQ_NVFP4_2D) {
    g.num_k = (int)((k / 2 + kKBytes - 1) / kKBytes);
    if ((st = make_map(&ta, a->codes, false, k / 2, m, k / 2, 128, kBM)) != LPQ_OK) return st;
    if ((st = make_map(&tb, b->codes, false, k / 2, n, k / 2, 128, BN)) != LPQ_OK) return st;
    g.idesc = idesc_block_scaled(1, 1, 0, BN);  // E2M1 x E2M1, E4M3 scales
    g.sfa = static_cast<const uint8_t*>(a->scales);
    g.sfb = static_cast<const uint8_t*>(b->scales);
    g.sfa_kt = sf_kt_atoms(LPQ_NVFP4, k);
    g.sfb_kt = g.sfa_kt;
    g.sfb_groups = sf_row_groups(n);
    g.alpha_a = a->tensor_scale;
    g.alpha_b = b->tensor_scale;
    if (pair_ok) {
      CUtensorMap tsa, tsb;
      if ((st = make_map(&tb, b->codes, false, k / 2, n, k / 2, 128, kPairBN / 2)) != LPQ_OK) return st;
      if ((st = make_map(&tbh, b->codes, false, k / 2, n, k / 2, 128, kPairBN / 4)) != LPQ_OK) return st;
      if ((st = make_sf_map(&tsa, g.sfa, sf_row_groups(m) * g.sfa_kt, 4)) != LPQ_OK) return st;
      if ((st = make_sf_map(&tsb, g.sfb, g.sfb_groups * g.sfb_kt, 4)) != LPQ_OK) return st;
      g.idesc = (g.idesc & ~(31u << 24)) | (16u << 24);
      if (cp) return run_pair<kKindNVF4>(ta, tb, tbh, tsa, tsb, g, direct, whole, s);
      return run_pair<kKindNVF4, true>(ta, tb, tbh, tsa, tsb, g, direct, whole, s);
    }
    if (nv_bn == 128) {
      if ((st = make_map(&tb, b->codes, false, k / 2, n, k / 2, 128, 128)) != LPQ_OK) return st;
      g.idesc = idesc_block_scaled(1, 1, 0, 128);
      if (cp) return run<kKindNVF4, 128, 2>(ta, tb, g, s);
      return run<kKindNVF4, 128, 2, true>(ta, tb, g, s);
    }
    if (cp) return run<kKindNVF4, BN, 1>(ta, tb, g, s);
    return run<kKindNVF4, BN, 1, true>(ta, tb, g, s);
  }
  if (fa == LPQ_FP8_BLOCK_1x128 || fa == LPQ_FP8_BLOCK_128x128) {
    BlockArgs bg{};
    bg.c = c;
    bg.M = m;
    bg.N = n;
    bg.K = k;
    bg.c_fp32 = c_is_fp32;
    bg.num_k = (int)(k / 128);
    bg.sa = static_cast<const float*>(a->scales);
    bg.sb = static_cast<const float*>(b->scales);
    bg.a_rows = fa == LPQ_FP8_BLOCK_1x128 ? 1 : 128;
    bg.b_rows = fb == LPQ_FP8_BLOCK_1x128 ? 1 : 128;
    if ((st = make_map(&ta, a->codes, false, k, m, k, 128, kBM)) != LPQ_OK) return st;
    if ((st = make_map(&tb, b->codes, false, k, n, k, 128, kBlkBN)) != LPQ_OK) return st;
    bg.idesc = idesc_dense(0, 0, kBlkBN);
    return run_block_gemm(ta, tb, bg, s);
  }
  return set_error(LPQ_ERR_UNSUPPORTED, "no GEMM kernel for format %d", fa);
}

// Tensor-core rate measurement: every CTA issues `iters` k-steps of four
// 128 x 256 MMAs on operand tiles resident in shared memory (no global
// traffic), optionally with the per-step scale-factor copies of the
// block-scaled kinds.  Operands are zero; the FLOP count is what is timed.
template <int KIND, int MODE>
__global__ void __launch_bounds__(256, 1) mma_peak_kernel(int iters, uint32_t idesc) {
  constexpr int with_sf = MODE;
  constexpr int BN = 256;
  using CF = Cfg<KIND, BN, 1>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + CF::kA;
  uint8_t* sSf = sB + CF::kB;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sSf + CF::kSfa + CF::kSfb);  // [2]: MMAs, other-warp copies
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (CF::kA + CF::kB + CF::kSfa + CF::kSfb) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 1, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 1) tmem_alloc(tmem_slot, CF::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  // with_sf: 0 none, 1 all copies of a step before its MMAs, 2 the same into
  // two alternating TMEM regions, 3 each MMA's copies right before it,
  // 4 (NVFP4) the scale columns rewritten with tcgen05.st by warps 4..7 while
  // the MMAs run, 5 (NVFP4) the step's 12 copies issued by warp 4 while the
  // MMAs run.  Modes 4 and 5 are unsynchronised with the MMAs: a rate probe.
  const uint32_t region = CF::kSfaCols + CF::kSfbCols;
  if (MODE >= 4 && warp >= 4) {
    const uint32_t tsfa = tbase + BN, tsfb = tsfa + CF::kSfaCols;
    if constexpr (MODE == 4) {
      uint32_t z16[16], z32[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) z16[i] = 0x38383838u;
#pragma unroll
      for (int i = 0; i < 32; ++i) z32[i] = 0x38383838u;
      const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
      for (int it = 0; it < iters; ++it) {
        tmem_st16(tsfa + lanes, z16);
        tmem_st32(tsfb + lanes, z32);
        tmem_wait_st();
      }
    } else if (MODE == 5 && warp == 4 && (threadIdx.x & 31) == 0) {
      const uint32_t kHiSf = (uint32_t)(smem_desc(0, 0, 128, 0) >> 32);
      const uint32_t flo = smem_u32(sSf) >> 4;
      for (int it = 0; it < iters; ++it)
        for (int j = 0; j < 4; ++j) {
          tmem_cp_sf(tsfa + 4 * j, ((uint64_t)kHiSf << 32) | (flo + j * 32));
          tmem_cp_sf(tsfb + 8 * j, ((uint64_t)kHiSf << 32) | (flo + 128 + j * 32));
          tmem_cp_sf(tsfb + 8 * j + 4, ((uint64_t)kHiSf << 32) | (flo + 256 + j * 32));
        }
      tc_commit(bar + 1);
      mbar_wait_bounded(bar + 1, 0, abort_flag, &g_device_error);
    }
  }
  if (threadIdx.x == 0) {
    const uint32_t kHiSw = (uint32_t)(smem_desc(0, 16, 1024, 2) >> 32);
    const uint32_t kHiSf = (uint32_t)(smem_desc(0, 0, 128, 0) >> 32);
    const uint32_t alo = (uint32_t)smem_desc(smem_u32(sA), 16, 1024, 2), blo = (uint32_t)smem_desc(smem_u32(sB), 16, 1024, 2);
    const uint32_t flo = smem_u32(sSf) >> 4;
    constexpr bool cps_first = with_sf == 1 || with_sf == 2, cps_inter = with_sf == 3;
    for (int it = 0; it < iters; ++it) {
      const uint32_t tsfa = tbase + BN + (with_sf == 2 ? (it & 1) * region : 0), tsfb = tsfa + CF::kSfaCols;
      if constexpr (KIND == kKindMXF8 && with_sf) {
        tmem_cp_sf(tsfa, ((uint64_t)kHiSf << 32) | flo);
        tmem_cp_sf(tsfb, ((uint64_t)kHiSf << 32) | (flo + 32));
        tmem_cp_sf(tsfb + 4, ((uint64_t)kHiSf << 32) | (flo + 64));
      } else if constexpr (KIND == kKindNVF4 && cps_first) {
        for (int j = 0; j < 4; ++j) {
          tmem_cp_sf(tsfa + 4 * j, ((uint64_t)kHiSf << 32) | (flo + j * 32));
          tmem_cp_sf(tsfb + 8 * j, ((uint64_t)kHiSf << 32) | (flo + 128 + j * 32));
          tmem_cp_sf(tsfb + 8 * j + 4, ((uint64_t)kHiSf << 32) | (flo + 256 + j * 32));
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t ad = ((uint64_t)kHiSw << 32) | (alo + 2 * j);
        const uint64_t bd = ((uint64_t)kHiSw << 32) | (blo + 2 * j);
        const uint32_t acc = (it > 0 || j > 0) ? 1u : 0u;
        if constexpr (KIND == kKindF16 || KIND == kKindF8F6F4) {
          mma_ss<KIND>(tbase, ad, bd, idesc, acc);
        } else if constexpr (KIND == kKindMXF8) {
          mma_bs<KIND>(tbase, ad, bd, idesc | ((uint32_t)j << 4) | ((uint32_t)j << 29), tsfa, tsfb, acc);
        } else {
          if constexpr (cps_inter) {
            tmem_cp_sf(tsfa + 4 * j, ((uint64_t)kHiSf << 32) | (flo + j * 32));
            tmem_cp_sf(tsfb + 8 * j, ((uint64_t)kHiSf << 32) | (flo + 128 + j * 32));
            tmem_cp_sf(tsfb + 8 * j + 4, ((uint64_t)kHiSf << 32) | (flo + 256 + j * 32));
          }
          mma_bs<KIND>(tbase, ad, bd, idesc, tsfa + 4 * j, tsfb + 8 * j, acc);
        }
      }
    }
    tc_commit(bar);
    mbar_wait_bounded(bar, 0, abort_flag, &g_device_error);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, CF::kTmemCols);
  }
}

// The same rate measurement on CTA pairs (cta_group::2), the shape the
// product GEMM issues: each cluster of two CTAs runs `iters` k-steps of four
// 256 x 256 pair MMAs (each SM holds 128 rows of A and 128 rows of B in shared
// memory, as in gemm_pair_kernel).  MODE 7 (block-scaled kinds) has four warps
// per CTA rewrite the scale columns with tcgen05.st while the MMAs run
// (unsynchronised; a rate probe).
template <int KIND, int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1) mma_peak_pair_kernel(int iters, uint32_t idesc) {
  // MODE 8: each k-step's four 256 x 256 MMAs issued as eight 256 x 128 MMAs
  // (two column halves, each half's B rows 64 per CTA) into two TMEM regions.
  constexpr bool kHalves = MODE == 8;
  using PC = PairCfg<KIND, false>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + PC::kA;
  uint8_t* sSf = sB + PC::kB;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sSf + PC::kSfa + PC::kSfb);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  const bool leader = cluster_ctarank() == 0;
  for (int i = threadIdx.x; i < (PC::kA + PC::kB + PC::kSfa + PC::kSfb) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  if (warp == 1) tmem_alloc_pair(tmem_slot, 512);
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tsfa = tbase + kPairBN, tsfb = tsfa + PC::kSfaCols;
  if (MODE == 7 && warp >= 4) {
    if constexpr (MODE == 7 && PC::kSfAtoms > 0) {
      uint32_t va[PC::kSfaCols], vb[PC::kSfbCols];
#pragma unroll
      for (int i = 0; i < PC::kSfaCols; ++i) va[i] = 0x38383838u;
#pragma unroll
      for (int i = 0; i < PC::kSfbCols; ++i) vb[i] = 0x38383838u;
      const uint32_t lanes = (uint32_t)((warp & 3) * 32) << 16;
      for (int it = 0; it < iters; ++it) {
        tmem_st_cols(tsfa + lanes, va);
        tmem_st_cols(tsfb + lanes, vb);
        tmem_wait_st();
      }
    }
  }
  if (threadIdx.x == 0) {
    if (leader) {
      const uint32_t kHiSw = (uint32_t)(smem_desc(0, 16, 1024, 2) >> 32);
      const uint32_t alo = (uint32_t)smem_desc(smem_u32(sA), 16, 1024, 2);
      const uint32_t blo = (uint32_t)smem_desc(smem_u32(sB), 16, 1024, 2);
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t ad = ((uint64_t)kHiSw << 32) | (alo + 2 * j);
          const uint32_t acc = (it > 0 || j > 0) ? 1u : 0u;
#pragma unroll
          for (int h = 0; h < (kHalves ? 2 : 1); ++h) {
            // half h: this CTA's B rows 64 h .. 64 h + 63 (8 KB into the swizzled tile)
            const uint64_t bd = ((uint64_t)kHiSw << 32) | (blo + 2 * j + (kHalves ? h * (8192 >> 4) : 0));
            const uint32_t d = tbase + (kHalves ? h * 128 : 0);
            if constexpr (KIND == kKindF16 || KIND == kKindF8F6F4) {
              mma_pair<KIND>(d, ad, bd, idesc, acc);
            } else {
              const int at = j * PC::kSfAtoms / 4;
              mma_pair_bs<KIND>(d, ad, bd, idesc | sf_select<KIND>(j), tsfa + 4 * at, tsfb + 8 * at + (kHalves ? 4 * h : 0),
                                acc);
            }
          }
        }
      }
      tc_commit_pair(bar, 0x3);
    }
    mbar_wait_bounded(bar, 0, abort_flag, &g_device_error);
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tbase, 512);
  }
}

template <int KIND, int MODE>
lpq_status run_peak_pair(int iters, uint32_t idesc, cudaStream_t s) {
  using PC = PairCfg<KIND, false>;
  const int smem = PC::kA + PC::kB + PC::kSfa + PC::kSfb + 1024 + 256;
  lpq_status st = set_smem_attr(reinterpret_cast<const void*>(mma_peak_pair_kernel<KIND, MODE>), smem);
  if (st != LPQ_OK) return st;
  const int sms = device_sms();
  uint32_t id = (idesc & ~(31u << 24)) | (16u << 24);                   // M = 256
  if (MODE == 8) id = (id & ~(63u << 17)) | ((uint32_t)(128 >> 3) << 17);  // N = 128
  mma_peak_pair_kernel<KIND, MODE><<<sms & ~1, 256, smem, s>>>(iters, id);
  return cuda_check(cudaGetLastError(), "pair peak kernel launch");
}

template <int KIND, int MODE>
lpq_status run_peak(int iters, uint32_t idesc, cudaStream_t s) {
  using CF = Cfg<KIND, 256, 1>;
  const int smem = CF::kA + CF::kB + CF::kSfa + CF::kSfb + 1024 + 256;
  lpq_status st = set_smem_attr(reinterpret_cast<const void*>(mma_peak_kernel<KIND, MODE>), smem);
  if (st != LPQ_OK) return st;
  const int sms = device_sms();
  mma_peak_kernel<KIND, MODE><<<sms, MODE >= 4 ? 256 : 128, smem, s>>>(iters, idesc);
  return cuda_check(cudaGetLastError(), "peak kernel launch");
}

lpq_status launch_mma_peak(int32_t kind, int32_t iters, int32_t with_sf, cudaStream_t s) {
  const uint32_t mx = idesc_block_scaled(0, 0, 1, 256), nv = idesc_block_scaled(1, 1, 0, 256);
  if (with_sf == 6) {  // CTA pairs, no scale traffic
    switch (kind) {
      case kKindF16: return run_peak_pair<kKindF16, 6>(iters, idesc_dense(1, 1, 256), s);
      case kKindF8F6F4: return run_peak_pair<kKindF8F6F4, 6>(iters, idesc_dense(0, 0, 256), s);
      case kKindMXF8: return run_peak_pair<kKindMXF8, 6>(iters, mx, s);
      case kKindNVF4: return run_peak_pair<kKindNVF4, 6>(iters, nv, s);
    }
    return set_error(LPQ_ERR_INVALID_ARG, "kind %d", kind);
  }
  if (with_sf == 8) {  // CTA pairs, 256 x 128 MMAs (two column halves per k-step)
    switch (kind) {
      case kKindF16: return run_peak_pair<kKindF16, 8>(iters, idesc_dense(1, 1, 256), s);
      case kKindF8F6F4: return run_peak_pair<kKindF8F6F4, 8>(iters, idesc_dense(0, 0, 256), s);
      case kKindMXF8: return run_peak_pair<kKindMXF8, 8>(iters, mx, s);
      case kKindNVF4: return run_peak_pair<kKindNVF4, 8>(iters, nv, s);
    }
    return set_error(LPQ_ERR_INVALID_ARG, "kind %d", kind);
  }
  if (with_sf == 7) {  // CTA pairs, scale columns rewritten by four warps per CTA
    if (kind == kKindMXF8) return run_peak_pair<kKindMXF8, 7>(iters, mx, s);
    if (kind == kKindNVF4) return run_peak_pair<kKindNVF4, 7>(iters, nv, s);
    return set_error(LPQ_ERR_INVALID_ARG, "mode 7 is for the block-scaled kinds");
  }
  switch (kind) {
    case kKindF16: return run_peak<kKindF16, 0>(iters, idesc_dense(1, 1, 256), s);
    case kKindF8F6F4: return run_peak<kKindF8F6F4, 0>(iters, idesc_dense(0, 0, 256), s);
    case kKindMXF8: return with_sf ? run_peak<kKindMXF8, 1>(iters, mx, s) : run_peak<kKindMXF8, 0>(iters, mx, s);
    case kKindNVF4:
      switch (with_sf) {
        case 0: return run_peak<kKindNVF4, 0>(iters, nv, s);
        case 1: return run_peak<kKindNVF4, 1>(iters, nv, s);
        case 2: return run_peak<kKindNVF4, 2>(iters, nv, s);
        case 3: return run_peak<kKindNVF4, 3>(iters, nv, s);
        case 4: return run_peak<kKindNVF4, 4>(iters, nv, s);
        case 5: return run_peak<kKindNVF4, 5>(iters, nv, s);
        default: return set_error(LPQ_ERR_INVALID_ARG, "with_scale_copies %d", with_sf);
      }
  }
  return set_error(LPQ_ERR_INVALID_ARG, "kind %d", kind);
}

// One CTA waits with the bounded wait on a barrier that nothing completes;
// used to check that a wait that runs out reports LPQ_ERR_TIMEOUT and leaves
// the context usable.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, &abort_flag, &g_device_error, limit_ns);
}

lpq_status launch_selftest_wait(uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cuda_check(cudaGetLastError(), "selftest kernel launch");
}

lpq_status read_and_clear_device_error(cudaStream_t s, int32_t* code) {
  lpq_status st = cuda_check(cudaStreamSynchronize(s), "cudaStreamSynchronize");
  if (st != LPQ_OK) return st;
  int v = 0;
  if ((st = cuda_check(cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)), "read device error word")) != LPQ_OK)
    return st;
  const int zero = 0;
  if ((st = cuda_check(cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)), "clear device error word")) != LPQ_OK)
    return st;
  *code = v;
  return LPQ_OK;
}

}  // namespace lpq
