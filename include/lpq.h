/*
 * lpq — block-scaled low-precision quantize-then-GEMM for transformer linear
 * layers on GB300 (sm_103a).  C ABI of liblpq.so.
 *
 * What the library computes is defined by these pages:
 *   [FP8]   "Optimizing Transformer models for low-precision training"
 *           (setupai.cc summary), "technical deep dive": E4M3 (1/4/3 bits,
 *           forward activations and weights) and E5M2 (1/5/2, gradients);
 *           per-tensor dynamic scaling from the amax; amax history.
 *   [NVFP4] "Accelerate LLM training with NVFP4 on Blackwell" (setupai.cc
 *           summary), "technical deep dive": E2M1 values (range about +-6), an
 *           E4M3 scale per 16-value micro-block plus an FP32 tensor scale;
 *           MXFP4, the format it refines, shares one scale per 32 values.
 *   [TE]    "How to optimize Transformer-based models for low-precision
 *           training" (developer.nvidia.cn): config -> 12 GEMM shapes
 *           ("model configuration and training input", "autocast vs
 *           pre-quantize"), Fprop/Dgrad/Wgrad benchmarked separately,
 *           pre-quantize mode, the NVFP4 extra costs (random Hadamard
 *           transform on Wgrad inputs, stochastic rounding of gradients, 2D
 *           weight blocks, extra amax pass) and silent fallbacks to avoid
 *           ("interpreting real-model results").
 *   [NeMo]  "Faster training throughput in FP8 with NVIDIA NeMo", "advantages
 *           and trade-offs": delayed, current, sub-channel (1x128 / 128x128)
 *           and MXFP8 (32-value blocks, E8M0 power-of-two scales).
 *
 * Conventions for every entry point:
 *   - Device pointers are owned by the caller; the library allocates no device
 *     memory (TMEM inside kernels is allocated and released per launch).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronising.
 *   - Every call returns an lpq_status; nothing throws across the ABI.  A
 *     non-OK status leaves a message readable with lpq_last_error() on the
 *     calling thread.  A call that returns non-OK has enqueued nothing unless
 *     the status is LPQ_ERR_CUDA.
 *   - No call ever falls back to another format, precision or a CPU path
 *     ([TE] warns of silent fallbacks): an unsupported combination is an error.
 *   - Matrices are row-major and contiguous along their last dimension.
 */
#ifndef LPQ_H_
#define LPQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *lpq_stream_t; /* same type as cudaStream_t */

typedef enum {
  LPQ_OK = 0,
  LPQ_ERR_INVALID_ARG = 1, /* NULL pointer, bad enum or flag */
  LPQ_ERR_SHAPE = 2,       /* a dimension is not a multiple of the block / tile rule */
  LPQ_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  LPQ_ERR_UNSUPPORTED = 4, /* format / layout / operand pairing not provided */
  LPQ_ERR_ARCH = 5,        /* current device is not compute capability 10.3 */
  LPQ_ERR_CUDA = 6,        /* a CUDA runtime call failed */
  LPQ_ERR_TIMEOUT = 7      /* a device-side wait gave up (see lpq_device_status) */
} lpq_status;

typedef enum {
  LPQ_BF16 = 0,               /* unquantized bf16 (the speed-up baseline) */
  LPQ_FP8_E4M3 = 1,           /* per-tensor scaled E4M3 [FP8] */
  LPQ_FP8_E5M2 = 2,           /* per-tensor scaled E5M2 [FP8] */
  LPQ_MXFP8 = 3,              /* E4M3 codes, one E8M0 scale per 32 values [NeMo] */
  LPQ_NVFP4 = 4,              /* E2M1 codes, E4M3 scale per 16 + FP32 tensor scale [NVFP4] */
  LPQ_NVFP4_2D = 5,           /* NVFP4 with one scale per 16x16 tile (weights) [TE] */
  LPQ_FP8_BLOCK_1x128 = 6,    /* E4M3, FP32 scale per 1x128 block (activations) [NeMo] */
  LPQ_FP8_BLOCK_128x128 = 7,  /* E4M3, FP32 scale per 128x128 block (weights) [NeMo] */
  LPQ_MXFP8_E5M2 = 8,         /* E5M2 codes, one E8M0 scale per 32 values (gradients) [NeMo], [FP8] */
  LPQ_MXFP4 = 9               /* packed E2M1 codes, one E8M0 scale per 32 values [NVFP4] */
} lpq_format;

/* Per-tensor FP8 scaling.  Every scale that is a quotient of a format maximum
 * by an amax (fmax / amax, NVFP4's 2688 / amax and s_enc / dec(S), the
 * sub-channel 448 / block max) is clamped to the largest finite float when it
 * overflows (an amax below about fmax / 3.4e38), so zeros stay +0 and every
 * dequantization factor stays positive. */
typedef enum { LPQ_SCALING_CURRENT = 0, LPQ_SCALING_DELAYED = 1 } lpq_scaling;

/* lpq_quantize flags */
enum {
  LPQ_ROWWISE = 1,     /* emit the row-wise copy [rows, cols] */
  LPQ_COLWISE = 2,     /* emit the column-wise copy [cols, rows] (re-blocked along rows) */
  LPQ_RHT_COLWISE = 4, /* NVFP4: 16-point random-sign Hadamard on the column-wise copy */
  LPQ_STOCHASTIC = 8,  /* NVFP4: stochastic rounding of the E2M1 codes (both copies) */
  LPQ_GIVEN_AMAX = 16  /* per-tensor FP8 (current scaling) and NVFP4: the views' amax fields
                          already hold the amax to scale with (e.g. the MAX over all shards of a
                          token-sharded tensor); no amax pass is run and they are left as given */
};

/* Scale-factor layouts of a copy. */
enum {
  LPQ_SF_PLAIN = 0, /* [rows, cols / block] row-major (FP8 block: FP32 [rows / br, cols / 128]) */
  LPQ_SF_GEMM = 1   /* tensor-core layout read by lpq_gemm (see lpq_copy_bytes) */
};

/* One quantized copy of a matrix.  All pointers are device pointers.
 *   codes        [rows, cols] bytes (FP8 formats), [rows, cols / 2] packed
 *                E2M1 (NVFP4, MXFP4: low nibble = even column), or bf16
 *                [rows, cols].
 *   scales       block scales: u8 E8M0 (MXFP8, MXFP8_E5M2, MXFP4), u8 E4M3
 *                (NVFP4), FP32 scale_inv (FP8 block); NULL for per-tensor FP8
 *                and bf16.  An E8M0 scale s stands for 2^(s - 127), where the
 *                block exponent is the smallest e with fmax * 2^e >= the
 *                block's max |value| (fmax 448 E4M3, 57344 E5M2, 6 E2M1), so
 *                that no code saturates.
 *   tensor_scale one FP32 dequantization factor: scale_inv for per-tensor
 *                FP8, the FP32 tensor scale for NVFP4; NULL otherwise.
 *   amax         one FP32: max |value| of this copy's input values (after the
 *                Hadamard transform for an RHT copy).  Required for per-tensor
 *                FP8 and NVFP4 (lpq_quantize writes it), optional for the MX
 *                formats (written when non-NULL), unused by the others.
 *   rows, cols   dimensions of this copy (the column-wise copy of an
 *                [R, C] tensor is [C, R]).
 *   colwise      1 for a column-wise copy, 0 for a row-wise copy.        */
typedef struct {
  void *codes;
  void *scales;
  float *tensor_scale;
  float *amax;
  int64_t rows, cols;
  int32_t fmt;       /* lpq_format */
  int32_t sf_layout; /* LPQ_SF_PLAIN or LPQ_SF_GEMM */
  int32_t colwise;
  int32_t reserved;
} lpq_qview;

typedef struct {
  lpq_qview row, col;
} lpq_qtensor;

/* Delayed-scaling state of one tensor role ([FP8] amax history; [NeMo]
 * per-tensor delayed scaling).  Device pointers.  Initial state: history all
 * 0, pos 0, scale 1, scale_inv 1.  The state is raw FP32/INT32 arrays, so a
 * checkpoint is a copy of them. */
typedef struct {
  float *amax_history; /* [len] */
  int32_t *pos;        /* next slot of the ring */
  float *scale;        /* scale used by the next quantize */
  float *scale_inv;
  int32_t len;         /* 1..1024; the workloads use 16 */
} lpq_delayed_state;

/* Bytes of one copy's codes and scales for format `fmt`, a copy of `rows` x
 * `cols` and scale layout `sf_layout`.  Host-only, needs no GPU.
 * LPQ_SF_GEMM layout for the MX formats and NVFP4: 128-row groups x KT atoms of 512
 * bytes; atom (g, t) starts at (g * KT + t) * 512 and holds, for row
 * r = 128 g + 32 j + i (i < 32, j < 4), its 4 scales of column-blocks
 * 4t .. 4t+3 at bytes 16 i + 4 j + 0..3.  KT = ceil(cols / 128) for MXFP8
 * and MXFP8_E5M2, 2 * ceil(cols / 256) for MXFP4 and 4 * ceil(cols / 256) for
 * NVFP4; entries beyond the matrix read as 0.
 * LPQ_SF_GEMM for FP8_BLOCK_1x128 is FP32 [cols / 128, rows] (rows fastest);
 * for FP8_BLOCK_128x128 it equals the plain layout. */
lpq_status lpq_copy_bytes(int32_t fmt, int64_t rows, int64_t cols, int32_t sf_layout,
                          size_t *codes_bytes, size_t *scale_bytes);

/* Quantizes x [rows, cols] bf16 (device) into the copies `flags` selects.
 *   fmt            LPQ_FP8_E4M3/E5M2 (with `scaling`), LPQ_MXFP8,
 *                  LPQ_MXFP8_E5M2, LPQ_MXFP4, LPQ_NVFP4, LPQ_NVFP4_2D,
 *                  LPQ_FP8_BLOCK_*, or LPQ_BF16 (row-wise = copy,
 *                  column-wise = transpose).
 *   scaling        per-tensor FP8 only.  CURRENT: scale = fmax / amax(x)
 *                  from an extra amax pass.  DELAYED: scale = *state->scale
 *                  from earlier steps; amax(x) is measured in the same pass
 *                  and written to out->row.amax (or col.amax); the state is
 *                  NOT advanced — call lpq_scale_update with that amax.
 *   seed, counter_offset   stochastic rounding: Philox-4x32-10 key = seed,
 *                  element j of a copy (row-major index + counter_offset)
 *                  uses word j mod 4 of counter (j / 4, copy id, 0).
 *                  counter_offset must be a multiple of 4.
 *   rht_seed       the 16 Hadamard signs: bits of word 0 of
 *                  Philox(key = (rht_seed, 0), counter = (0, 0, 2, 0)).
 *   out            views to fill; out->row used if LPQ_ROWWISE, out->col if
 *                  LPQ_COLWISE.  Each view's rows/cols/fmt must match.
 *                  With LPQ_GIVEN_AMAX the amax of each requested view is an
 *                  input (NVFP4: the row view's the raw amax, the column
 *                  view's the amax of its own values, after the RHT when
 *                  LPQ_RHT_COLWISE is set; FP8: the row view's, else the
 *                  column view's, for both copies).  Quantizing the shards of
 *                  a tensor with the MAX of their amaxes gives exactly the
 *                  codes and scales of the whole tensor (for the row-wise
 *                  copy with stochastic rounding, pass counter_offset =
 *                  first row * cols).
 * Shape rules: cols a multiple of the row-wise block (16 NVFP4, 32 MX formats, 128
 * FP8 block, 16 NVFP4_2D), rows a multiple of the column-wise block when
 * LPQ_COLWISE is set (same numbers; 128x128 needs neither rows nor cols beyond
 * cols % 128 == 0 and rows % 128 == 0 for its column copy), and every row of
 * every output 16-byte aligned.  A 0 x n or n x 0 input is valid and enqueues
 * nothing but the scalar outputs. */
lpq_status lpq_quantize(const void *x, int64_t rows, int64_t cols, int32_t fmt, int32_t scaling,
                        uint32_t flags, uint64_t seed, uint64_t counter_offset, uint32_t rht_seed,
                        const lpq_delayed_state *state, lpq_qtensor *out, lpq_stream_t stream);

/* The global amax pass ([TE] "interpreting real-model results": the extra
 * memory pass for the per-tensor amax; [FP8] per-tensor scaling from the
 * tensor's amax): *amax = max |x| over x [rows, cols] bf16 (NaN ignored,
 * infinities counted), overwritten (not accumulated).  With LPQ_RHT_COLWISE
 * in flags, *rht_amax gets max |RHT16(v)| over the column-wise copy (each
 * column's 16-runs of rows transformed with the signs of rht_seed, as in
 * lpq_quantize), the amax an NVFP4 RHT column copy is scaled with; rows must
 * then be a multiple of 16.  amax and rht_amax are device FP32 pointers;
 * either may be NULL, not both (rht_amax is ignored without the flag).  cols
 * must be a multiple of 16 and x 16-byte aligned; an empty x gives 0.  This is
 * the pass lpq_quantize runs before current-scaled FP8 and NVFP4 copies: a
 * token-sharded caller runs it on its own shard, combines the shards' values
 * with a MAX all-reduce and quantizes with LPQ_GIVEN_AMAX.  flags other than
 * LPQ_RHT_COLWISE give LPQ_ERR_INVALID_ARG. */
lpq_status lpq_amax(const void *x, int64_t rows, int64_t cols, uint32_t flags, uint32_t rht_seed, float *amax,
                    float *rht_amax, lpq_stream_t stream);

/* Delayed-scaling update (one CTA): history[pos] = *amax; pos = (pos+1) % len;
 * m = max(history); scale = fmax / m if m > 0 and finite (else unchanged),
 * clamped to the largest finite float if the quotient overflows;
 * scale_inv = 1 / scale.  fmax is 448 (E4M3) or 57344 (E5M2).  pos should be
 * in [0, len); a value outside is taken modulo len (no write leaves the
 * history). */
lpq_status lpq_scale_update(const lpq_delayed_state *state, const float *amax, float fmax,
                            lpq_stream_t stream);

/* Which copies a GEMM of a linear layer reads ([TE]: Fprop, Dgrad and Wgrad
 * are separate GEMMs).  X [M, K] activations, W [N, K] weights, dY [M, N]:
 *   LPQ_FPROP  Y  = X W^T   : a = X row-wise,   b = W row-wise   -> C [M, N]
 *   LPQ_DGRAD  dX = dY W    : a = dY row-wise,  b = W col-wise   -> C [M, K]
 *   LPQ_WGRAD  dW = dY^T X  : a = dY col-wise,  b = X col-wise   -> C [N, K]
 * The layout only states which copies are expected (checked against the
 * views' `colwise` flags); the arithmetic is the same. */
typedef enum { LPQ_FPROP = 0, LPQ_DGRAD = 1, LPQ_WGRAD = 2 } lpq_layout;

/* C[m, n] = sum_k deq(a)[m, k] * deq(b)[n, k], FP32 accumulation on the
 * tensor cores (tcgen05), output bf16 (c_is_fp32 = 0) or FP32, row-major with
 * leading dimension n.  a is [m, k], b is [n, k], both contiguous along k.
 * Legal pairings: BF16 x BF16; {E4M3, E5M2} x {E4M3, E5M2} (per-tensor,
 * scale_inv product applied in the epilogue); {MXFP8, MXFP8_E5M2} x {MXFP8,
 * MXFP8_E5M2} (E5M2 gradients against E4M3 activations or weights);
 * MXFP4 x MXFP4; {NVFP4,
 * NVFP4_2D} x {NVFP4, NVFP4_2D} (tensor scales in the epilogue); FP8 block
 * (1x128 or 128x128) x FP8 block (FP32 block scales applied per 128-deep
 * slice).  Block-scaled operands must use LPQ_SF_GEMM.  k must be a multiple
 * of 32 (128 for FP8 block); m and n are arbitrary (>= 0).  Anything else
 * returns LPQ_ERR_UNSUPPORTED or LPQ_ERR_SHAPE; nothing falls back. */
lpq_status lpq_gemm(int32_t layout, const lpq_qview *a, const lpq_qview *b, void *c, int32_t c_is_fp32,
                    int64_t m, int64_t n, int64_t k, lpq_stream_t stream);

/* Kernel-path options of lpq_gemm_ex.  They choose between kernels that
 * compute the same result (every path passes the same parity tests); they
 * never change the format, the precision or the arithmetic, and nothing else
 * (no environment variable, no global setting) selects a path.  All-zero is
 * the default path that lpq_gemm takes.
 *   single_cta    0: CTA pairs (cta_group::2, 256 x 256 output tiles) when
 *                 m >= 256, one CTA per 128 x 256 tile otherwise; 1: always
 *                 one CTA per tile.
 *   tile_n        single-CTA block-scaled kinds: 0 or 256 (128 x 256 tiles,
 *                 one TMEM accumulator) or 128 (128 x 128 tiles, two
 *                 accumulators).  Ignored elsewhere.
 *   scale_copies  block-scaled kinds: 0 = the scale factors are written into
 *                 TMEM by four scale warps (tcgen05.st); 1 = copied by the
 *                 MMA-issuing thread (tcgen05.cp).
 *   direct_store  CTA-pair kernel, bf16 output: 0 = TMA tile stores through
 *                 shared memory (when n % 8 == 0); 1 = stores from registers.
 *   whole_tiles   CTA-pair kernel: 0 = when the tiles left for the last round
 *                 of the persistent schedule fill at most half of the CTA
 *                 pairs, each of them runs as two 256 x 128 halves (N = 128
 *                 MMAs) on two pairs, so that the last round takes half as
 *                 long; 1 = whole 256 x 256 tiles only.
 *   reserved      must be 0.
 * Values outside these sets give LPQ_ERR_INVALID_ARG. */
typedef struct {
  int32_t single_cta;
  int32_t tile_n;
  int32_t scale_copies;
  int32_t direct_store;
  int32_t whole_tiles;
  int32_t reserved[3];
} lpq_gemm_opts;

/* lpq_gemm with explicit kernel-path options (NULL = all defaults). */
lpq_status lpq_gemm_ex(int32_t layout, const lpq_qview *a, const lpq_qview *b, void *c, int32_t c_is_fp32,
                       int64_t m, int64_t n, int64_t k, const lpq_gemm_opts *opts, lpq_stream_t stream);

/* Transformer configuration ([TE] "model configuration and training input"). */
typedef struct {
  int64_t hidden, intermediate, heads, layers, micro_batch, seq;
} lpq_transformer_cfg;

typedef struct {
  char name[24];   /* e.g. "qkv_fprop" */
  int32_t layout;  /* lpq_layout */
  int64_t m, k, n; /* C [m, n] = sum over k */
} lpq_gemm_shape;

/* The 12 GEMMs of one layer: M = micro_batch * seq; QKV (K = hidden,
 * N = 3 hidden), attention out (hidden, hidden), MLP up (hidden,
 * intermediate), MLP down (intermediate, hidden), each as Fprop (M, K, N),
 * Dgrad (M, N, K) and Wgrad (N, M, K).  `heads` and `layers` do not change
 * the linear shapes.  Host-only. */
lpq_status lpq_layer_shapes(const lpq_transformer_cfg *cfg, lpq_gemm_shape out[12], int32_t *count);

/* Text of the last non-OK status on this thread ("" if none). */
const char *lpq_last_error(void);

/* Synchronises `stream`, then reads and clears the device error word that
 * kernels set when a bounded wait gives up (0 = none, else an lpq_status). */
lpq_status lpq_device_status(lpq_stream_t stream, int32_t *code);

/* Failure-detection check: launches one CTA whose bounded wait (the same
 * helper the GEMM pipeline uses) waits on a barrier that nothing completes.
 * After limit_ns (0 < limit_ns <= 1 s) the wait gives up and records
 * LPQ_ERR_TIMEOUT in the device error word, which lpq_device_status then
 * returns; the CUDA context stays usable.  No fault, trap or hang is involved. */
lpq_status lpq_selftest_wait(uint64_t limit_ns, lpq_stream_t stream);

/* Arithmetic self-check of the quantizers' device helpers against their
 * definitions, for the test suite.  Counts mismatches over indices i in
 * [begin, begin + count):
 *   which 0: x = the float with bits i (i <= 0x7F800000: every non-negative
 *            float and +inf): the block-max division by 6 (a product with
 *            RN(1/6) corrected by one fused multiply-add of the exact
 *            residual) against the IEEE quotient x / 6;
 *   which 1: |y| = the float with bits i >> 3 and the (i & 7)-th of eight
 *            probe words r (r >> 8 = 0, 1, 2^23 - 2, 2^23, 2^24 - 3,
 *            2^24 - 2, 2^24 - 1, 2^24 - 1, low bytes 0x00 or 0xFF): the
 *            stochastic E2M1 rounding of y and -y against the definition
 *            (round up to the next grid magnitude iff float(r >> 8) <
 *            frac * 2^24; 6 at and beyond 6 and for NaN);
 *   which 2: y = the float with bits `param` and r = i << 8 | (i * 37 mod
 *            256), i < 2^24 (every threshold value for one y), y and -y.
 * result (device, two int64, 8-byte aligned) receives the mismatch count and
 * the smallest mismatching index (-1 if none); the call returns at once, read
 * result after synchronising `stream`.  Ranges beyond the mode's index limit
 * give LPQ_ERR_INVALID_ARG. */
lpq_status lpq_selftest_arith(int32_t which, uint64_t begin, uint64_t count, uint32_t param, int64_t *result,
                              lpq_stream_t stream);

/* Tensor-core rate measurement (the dense peaks the roofline divides by):
 * one CTA per SM issues `iters` k-steps of four 128 x 256 tcgen05.mma on
 * zero operands resident in shared memory; kind 0 = kind::f16 (bf16, K 16),
 * 1 = kind::f8f6f4 (E4M3, K 32), 2 = MXFP8 block-scaled (K 32), 3 = NVFP4
 * block-scaled (K 64).  with_scale_copies adds the per-step tcgen05.cp of the
 * scale factors (kinds 2, 3): 1 = all of a step's copies before its MMAs,
 * 2 = the same into two alternating TMEM regions, 3 = each MMA's copies
 * right before it, 4 = the scale columns rewritten by four other warps with
 * tcgen05.st while the MMAs run, 5 = the step's copies issued by a thread of
 * another warp while the MMAs run (4 and 5: NVFP4 only, unsynchronised with
 * the MMAs, throughput only), 6 = CTA pairs (cta_group::2: clusters of two
 * CTAs, each pair issuing four 256 x 256 MMAs per k-step, each SM holding
 * 128 rows of A and of B, the shape of the product GEMM; any kind), 7 = CTA
 * pairs with the scale columns rewritten by four warps per CTA with
 * tcgen05.st while the MMAs run (kinds 2, 3), 8 = CTA pairs issuing each
 * k-step as eight 256 x 128 MMAs (two column halves into two TMEM regions;
 * any kind).  Other values give LPQ_ERR_INVALID_ARG.  Modes 6 to 8 launch SMs
 * rounded down to even CTAs.
 * FLOPs = CTAs * iters * 4 * 2 * 128 * 256 * K;
 * the caller times the launch with events on `stream`. */
lpq_status lpq_mma_peak(int32_t kind, int32_t iters, int32_t with_scale_copies, lpq_stream_t stream);

/* Library version (major * 10000 + minor * 100 + patch). */
int32_t lpq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LPQ_H_ */
