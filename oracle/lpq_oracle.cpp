// lpq CPU oracle — TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, obviously-correct CPU statement of what the low-precision
// quantize-then-GEMM path computes.  Only the test suite, the smoke check and
// the benchmark's CPU-baseline leg load this library; the product path never
// does.  It shares no source with the CUDA library: every codec, scale rule,
// random-number generator and transform below is written out again here from
// the format definitions.
//
// Sources (pages on low-precision training of transformer linear layers):
//   [FP8]   "Optimizing Transformer models for low-precision training"
//           (setupai.cc summary), section "technical deep dive": FP8 comes as
//           E4M3 (1 sign, 4 exponent, 3 mantissa bits; forward activations and
//           weights) and E5M2 (1/5/2; backward gradients); per-tensor scaling
//           from the tensor's amax; a rolling amax history for delayed scaling.
//   [NVFP4] "Accelerate LLM training with NVFP4 on Blackwell" (setupai.cc
//           summary), section "technical deep dive": E2M1 values (1/2/1 bits,
//           range about +-6), one E4M3 scale per 16-value micro-block and a
//           second FP32 scale per tensor, about 4.5 bits per value.
//   [TE]    "How to optimize Transformer-based models for low-precision
//           training" (developer.nvidia.cn), sections "autocast vs pre-quantize"
//           and "interpreting real-model results": the 12 GEMMs of a layer,
//           Fprop/Dgrad/Wgrad, and the NVFP4 extra costs (random Hadamard
//           transform on Wgrad inputs, stochastic rounding of gradients, 2D
//           block scaling of weights, an extra pass for the per-tensor amax).
//   [NeMo]  "Faster training throughput in FP8 with NVIDIA NeMo", section
//           "advantages and trade-offs of FP8 scaling methods": delayed,
//           current, sub-channel (1x128 activation / 128x128 weight blocks)
//           and MXFP8 (32-value blocks, power-of-two E8M0 scales).
//   [Philox] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
//           1, 2, 3", SC'11, section 4 (Philox-4x32 round function and key
//           schedule).
//
// Where the pages leave a step open the plainest reading is taken; every such
// reading is listed in the design notes of the repository and repeated at the
// function that makes it.
//
// Arithmetic: IEEE binary32/binary64 with round-to-nearest-even, built with
// -ffp-contract=off (no fused multiply-add) and without fast-math, so each
// float expression below rounds exactly once per operation.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- threading
int g_threads = 0;

int num_threads() {
  if (g_threads > 0) return g_threads;
  const char* env = std::getenv("LPQ_ORACLE_THREADS");
  int n = env ? std::atoi(env) : 0;
  if (n <= 0) n = (int)std::thread::hardware_concurrency();
  if (n <= 0) n = 1;
  g_threads = n;
  return n;
}

// Runs fn(lo, hi) over static chunks of [0, n) on all threads; small ranges
// (fewer than `serial_below` items) run on the calling thread.
void parallel_for(int64_t n, const std::function<void(int64_t, int64_t)>& fn,
                  int64_t serial_below = 64) {
  int t = num_threads();
  if (n < serial_below || t == 1) {
    fn(0, n);
    return;
  }
  if (t > n) t = (int)n;
  std::vector<std::thread> pool;
  int64_t chunk = (n + t - 1) / t;
  for (int i = 0; i < t; ++i) {
    int64_t lo = i * chunk, hi = std::min<int64_t>(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([&fn, lo, hi] { fn(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

// ---------------------------------------------------------------- bf16
float bf16_value(uint16_t bits) {
  uint32_t u = uint32_t(bits) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// ---------------------------------------------------------------- codecs
// Format ids shared with the Python side of the oracle.
enum { E4M3 = 0, E5M2 = 1, E2M1 = 2 };

// Decodes one code from its bit fields [FP8] technical deep dive (E4M3 =
// 1/4/3, E5M2 = 1/5/2) and [NVFP4] technical deep dive (E2M1 = 1/2/1).
// Exponent biases 7 / 15 / 1 and the special values are the usual reading of
// those bit splits: E4M3 has no infinity and one NaN mantissa (S.1111.111), so
// its largest finite value is 448; E5M2 keeps IEEE infinities and NaNs, so its
// largest finite value is 57344; E2M1 has no special values, largest 6 (the
// "about +-6" range of [NVFP4]).
double decode(int fmt, uint8_t c) {
  int s, e, m;
  double v;
  if (fmt == E4M3) {
    s = c >> 7; e = (c >> 3) & 15; m = c & 7;
    if (e == 15 && m == 7) return std::nan("");
    v = (e == 0) ? (m / 8.0) * std::ldexp(1.0, -6) : (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);
  } else if (fmt == E5M2) {
    s = c >> 7; e = (c >> 2) & 31; m = c & 3;
    if (e == 31) return m == 0 ? (s ? -INFINITY : INFINITY) : std::nan("");
    v = (e == 0) ? (m / 4.0) * std::ldexp(1.0, -14) : (1.0 + m / 4.0) * std::ldexp(1.0, e - 15);
  } else {
    s = (c >> 3) & 1; e = (c >> 1) & 3; m = c & 1;
    v = (e == 0) ? m * 0.5 : (1.0 + m / 2.0) * std::ldexp(1.0, e - 1);
  }
  return s ? -v : v;
}

int max_code(int fmt) { return fmt == E4M3 ? 0x7E : fmt == E5M2 ? 0x7B : 0x7; }
uint8_t sign_bit(int fmt) { return fmt == E2M1 ? 0x8 : 0x80; }
uint8_t nan_code(int fmt) { return fmt == E2M1 ? 0x7 : 0x7F; }

// Encodes y by round-to-nearest-even with saturation.  The positive codes
// 0..max_code are monotone in value, so the encoder finds the two neighbours
// of |y| among them, keeps the nearer, and on an exact tie keeps the one whose
// mantissa LSB (= code LSB) is 0.  |y| at or above the largest finite value,
// infinities included, saturates to it.  The sign bit is always copied, so a
// negative value that rounds to zero gives the negative-zero code.  NaN gives
// 0x7F for the FP8 formats and +6 (0x7) for E2M1, which has no NaN.
uint8_t encode(int fmt, float y) {
  if (std::isnan(y)) return nan_code(fmt);
  uint8_t s = std::signbit(y) ? sign_bit(fmt) : 0;
  double a = std::fabs((double)y);
  int top = max_code(fmt);
  if (a >= decode(fmt, (uint8_t)top)) return s | (uint8_t)top;
  int lo = 0, hi = top;  // invariant: value(lo) <= a < value(hi)
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (decode(fmt, (uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  double dlo = a - decode(fmt, (uint8_t)lo), dhi = decode(fmt, (uint8_t)hi) - a;
  int pick = dlo < dhi ? lo : dhi < dlo ? hi : ((lo & 1) == 0 ? lo : hi);
  return s | (uint8_t)pick;
}

// The eight E2M1 magnitudes in code order (code = index).
const float kE2M1[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};

// ---------------------------------------------------------------- Philox
// Philox-4x32 with 10 rounds [Philox] section 4: each round multiplies the
// even words by the two published multipliers, takes the 64-bit product's
// high and low halves, and mixes them with the odd words and the round key;
// the key is bumped by the two Weyl constants between rounds.
void philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { k0 += W0; k1 += W1; }
    uint64_t p0 = (uint64_t)M0 * x0;
    uint64_t p1 = (uint64_t)M1 * x2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t y0 = hi1 ^ x1 ^ k0, y1 = lo1, y2 = hi0 ^ x3 ^ k1, y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

// Random 32-bit word for element j of a copy (stochastic rounding).  Reading
// of "stochastic rounding of gradients" [TE] (the pages name no generator):
// key = (seed low 32 bits, seed high 32 bits), counter = (g low, g high,
// copy id, 0) with g = j / 4, and the word used is output word j mod 4, where
// j = counter_offset + the element's row-major index inside the copy.
uint32_t sr_word(uint64_t seed, uint64_t j, uint32_t copy_id) {
  uint64_t g = j >> 2;
  uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), copy_id, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return out[j & 3];
}

// The 16 signs of the random Hadamard transform: bit j of word 0 of
// Philox(key = (rht_seed, 0), counter = (0, 0, 2, 0)); a set bit means -1.
uint32_t rht_sign_mask(uint32_t rht_seed) {
  uint32_t ctr[4] = {0u, 0u, 2u, 0u};
  uint32_t key[2] = {rht_seed, 0u};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return out[0] & 0xFFFFu;
}

// 16-point random-sign Hadamard transform of one run (the "random Hadamard
// transform on Wgrad inputs" of [TE], interpreting section).  Reading: flip
// signs, then a Sylvester butterfly in fp32 with stages h = 1, 2, 4, 8, each
// pair (t_i, t_{i+h}) with bit h of i clear becoming (t_i + t_{i+h},
// t_i - t_{i+h}), then a scale by 1/4 so the transform is orthonormal.
void rht16(const float* x, uint32_t signs, float* v) {
  float t[16];
  for (int j = 0; j < 16; ++j) t[j] = ((signs >> j) & 1u) ? -x[j] : x[j];
  for (int h = 1; h < 16; h <<= 1)
    for (int i = 0; i < 16; ++i)
      if ((i & h) == 0) {
        float a = t[i], b = t[i + h];
        t[i] = a + b;
        t[i + h] = a - b;
      }
  for (int j = 0; j < 16; ++j) v[j] = 0.25f * t[j];
}

// Stochastic E2M1 rounding of y with random word r.  Reading: for |y| < 6
// between adjacent magnitudes lo <= |y| <= hi, round up to hi exactly when
// float(r >> 8) < frac * 2^24 with frac = (|y| - lo) / (hi - lo); both steps
// are exact in fp32 (Sterbenz subtraction, division by a power of two).
// |y| >= 6 gives 6; NaN gives +6; the sign is copied.
uint8_t sr_encode_e2m1(float y, uint32_t r) {
  if (std::isnan(y)) return 0x7;
  uint8_t s = std::signbit(y) ? 0x8 : 0;
  float a = std::fabs(y);
  if (a >= 6.0f) return s | 0x7;
  int lo = 0;
  while (lo < 7 && kE2M1[lo + 1] <= a) ++lo;
  float frac = (a - kE2M1[lo]) / (kE2M1[lo + 1] - kE2M1[lo]);
  float r24 = (float)(r >> 8);
  bool up = r24 < frac * 16777216.0f;
  return s | (uint8_t)(up ? lo + 1 : lo);
}

// max |v| ignoring NaN (IEEE maxNum); infinities count.
float absmax(const float* v, int64_t n, int64_t stride) {
  float m = 0.f;
  for (int64_t i = 0; i < n; ++i) {
    float a = std::fabs(v[i * stride]);
    if (a > m) m = a;
  }
  return m;
}

float amax_bf16(const uint16_t* x, int64_t n) {
  int t = num_threads();
  std::vector<float> part(t, 0.f);
  int64_t chunk = (n + t - 1) / t;
  parallel_for(t, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) {
      float m = 0.f;
      int64_t a = i * chunk, b = std::min<int64_t>(n, a + chunk);
      for (int64_t k = a; k < b; ++k) {
        float v = std::fabs(bf16_value(x[k]));
        if (v > m) m = v;
      }
      part[i] = m;
    }
  }, n < (1 << 16) ? t + 1 : 1);
  float m = 0.f;
  for (float p : part) m = std::max(m, p);
  return m;
}

float fmt_max(int fmt) { return (float)decode(fmt, (uint8_t)max_code(fmt)); }

// Value 2^k as a float for k in [-127, 127] (2^-127 is a subnormal).
float pow2f(int k) { return (float)std::ldexp(1.0, k); }

// A scale that is the quotient of a format maximum by an amax (fmax / amax,
// 2688 / A, 448 / block max) overflows the float range when the amax is below
// about fmax / 3.4e38 (bf16 holds such values).  Reading: the quotient is then
// clamped to the largest finite float.  The pages give no rule for this case;
// an infinite scale would turn zero elements into NaN codes and the
// dequantization factor 1 / scale into 0.
float finite_scale(float q) { return q > 3.40282347e38f ? 3.40282347e38f : q; }

// MXFP8 block exponent for block amax a ([NeMo] MXFP8: power-of-two E8M0
// scale per 32 values).  Reading: the smallest e with 448 * 2^e >= a, i.e.
// ceil(log2(a / 448)), so no element of the block saturates; taken from the
// exact decomposition a = m * 2^E, m in [1, 2): e = E - 8 + (m > 1.75).
// a = 0 gives -127; a non-finite amax gives 127; e is clamped to [-127, 127].
int mx_exponent(float a) {
  if (a == 0.f) return -127;
  if (!std::isfinite(a)) return 127;
  int ex;
  double f = std::frexp((double)a, &ex);  // a = f * 2^ex, f in [0.5, 1)
  double m = 2.0 * f;
  int E = ex - 1;
  int e = E - 8 + (m > 1.75 ? 1 : 0);
  return std::max(-127, std::min(127, e));
}

// The same rule for an MX element format of largest value fmax = mf * 2^Ef
// (mf in [1, 2)): the smallest e with fmax * 2^e >= a is Ea - Ef + (ma > mf)
// for a = ma * 2^Ea.  E4M3 (448 = 1.75 * 2^8) gives mx_exponent; E5M2 (57344 =
// 1.75 * 2^15) the MXFP8 gradient variant; E2M1 (6 = 1.5 * 2^2) MXFP4 ([NVFP4]:
// NVFP4 narrows MXFP4's 32-value blocks to 16).
int mx_exponent_fmt(float a, int fmt) {
  if (a == 0.f) return -127;
  if (!std::isfinite(a)) return 127;
  int ea, ef;
  double ma = 2.0 * std::frexp((double)a, &ea);
  double mf = 2.0 * std::frexp((double)fmt_max(fmt), &ef);
  int e = (ea - 1) - (ef - 1) + (ma > mf ? 1 : 0);
  return std::max(-127, std::min(127, e));
}

}  // namespace

// ======================================================================= C API
extern "C" {

int orc_num_threads() { return num_threads(); }
void orc_set_threads(int n) { g_threads = n; }

double orc_decode(int fmt, uint8_t c) { return decode(fmt, c); }
uint8_t orc_encode(int fmt, float y) { return encode(fmt, y); }

void orc_encode_array(int fmt, const float* y, int64_t n, uint8_t* out) {
  parallel_for(n, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) out[i] = encode(fmt, y[i]);
  });
}

void orc_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}
uint32_t orc_sr_word(uint64_t seed, uint64_t j, uint32_t copy_id) { return sr_word(seed, j, copy_id); }
uint32_t orc_rht_sign_mask(uint32_t rht_seed) { return rht_sign_mask(rht_seed); }
void orc_rht16(const float* x, uint32_t signs, float* v) { rht16(x, signs, v); }
uint8_t orc_sr_encode_e2m1(float y, uint32_t r) { return sr_encode_e2m1(y, r); }
int orc_mx_exponent(float a) { return mx_exponent(a); }

float orc_amax_bf16(const uint16_t* x, int64_t n) { return amax_bf16(x, n); }

// ---------------------------------------------------------------- per-tensor FP8
// Current scaling ([FP8] per-tensor dynamic scaling; [NeMo] current scaling):
// scale = fmax / amax (fp32, RN; clamped to the largest finite float if it
// overflows), or 1 when amax is 0 or not finite; codes =
// RNE-saturated encode of x * scale; scale_inv = 1 / scale.  Reading: no
// margin and no power-of-two rounding of the scale (the pages state neither).
// The column-wise copy ([C, R]) is the transpose of the same codes.
// `scale_in` != NULL selects delayed scaling: that scale is used instead and
// amax is only measured ([FP8] amax history: the scale comes from earlier
// iterations).  Returns the number of elements with |x * scale| > fmax.
int64_t orc_fp8_pertensor(const uint16_t* x, int64_t R, int64_t C, int fmt, const float* scale_in,
                          uint8_t* row, uint8_t* col, float* scale_out, float* scale_inv_out,
                          float* amax_out) {
  float fmax = fmt_max(fmt);
  float amax = amax_bf16(x, R * C);
  float scale;
  if (scale_in) scale = *scale_in;
  else scale = (amax > 0.f && std::isfinite(amax)) ? finite_scale(fmax / amax) : 1.0f;
  std::atomic<int64_t> sat{0};
  parallel_for(R, [&](int64_t lo, int64_t hi) {
    int64_t local = 0;
    for (int64_t r = lo; r < hi; ++r)
      for (int64_t c = 0; c < C; ++c) {
        float y = bf16_value(x[r * C + c]) * scale;
        if (std::fabs(y) > fmax) ++local;
        uint8_t q = encode(fmt, y);
        if (row) row[r * C + c] = q;
        if (col) col[c * R + r] = q;
      }
    sat += local;
  });
  if (scale_out) *scale_out = scale;
  if (scale_inv_out) *scale_inv_out = 1.0f / scale;
  if (amax_out) *amax_out = amax;
  return sat.load();
}

// Delayed-scaling state update ([FP8] amax history; [NeMo] per-tensor delayed
// scaling).  Reading: the amax of this step goes into a ring of `len` entries
// at `pos`; pos advances modulo len; the next scale is fmax / max(ring)
// (clamped to the largest finite float) when that max is positive and finite,
// else the scale is kept; scale_inv = 1/scale.
void orc_scale_update(float* hist, int32_t len, int32_t* pos, float* scale, float* scale_inv,
                      float amax, float fmax) {
  int32_t slot = ((*pos % len) + len) % len;  // a position outside [0, len) is taken modulo len
  hist[slot] = amax;
  *pos = (slot + 1) % len;
  float m = 0.f;
  for (int i = 0; i < len; ++i) m = std::max(m, hist[i]);
  if (m > 0.f && std::isfinite(m)) *scale = finite_scale(fmax / m);
  *scale_inv = 1.0f / *scale;
}

// ---------------------------------------------------------------- MXFP8
// One copy: values v [rows, cols] (float), blocks of 32 along cols.
static void mxfp8_copy(const std::function<float(int64_t, int64_t)>& v, int64_t rows, int64_t cols,
                       uint8_t* codes, uint8_t* sf) {
  int64_t nb = cols / 32;
  parallel_for(rows, [&](int64_t lo, int64_t hi) {
    float blk[32];
    for (int64_t r = lo; r < hi; ++r)
      for (int64_t b = 0; b < nb; ++b) {
        for (int i = 0; i < 32; ++i) blk[i] = v(r, b * 32 + i);
        int e = mx_exponent(absmax(blk, 32, 1));
        float mult = pow2f(-e);
        for (int i = 0; i < 32; ++i) codes[r * cols + b * 32 + i] = encode(E4M3, blk[i] * mult);
        sf[r * nb + b] = (uint8_t)(e + 127);
      }
  });
}

// MX copy of any element format: blocks of 32 along cols, E8M0 exponent from
// mx_exponent_fmt, codes = RNE encode of v * 2^-e (nothing saturates).  E2M1
// codes are packed two per byte, the low nibble holding the even column.
static void mx_copy(const std::function<float(int64_t, int64_t)>& v, int64_t rows, int64_t cols, int fmt,
                    uint8_t* codes, uint8_t* sf) {
  int64_t nb = cols / 32;
  parallel_for(rows, [&](int64_t lo, int64_t hi) {
    float blk[32];
    for (int64_t r = lo; r < hi; ++r)
      for (int64_t b = 0; b < nb; ++b) {
        for (int i = 0; i < 32; ++i) blk[i] = v(r, b * 32 + i);
        int e = mx_exponent_fmt(absmax(blk, 32, 1), fmt);
        float mult = pow2f(-e);
        for (int i = 0; i < 32; ++i) {
          uint8_t q = encode(fmt, blk[i] * mult);
          if (fmt == E2M1) {
            uint8_t& byte = codes[r * (cols / 2) + (b * 32 + i) / 2];
            byte = (i & 1) ? (uint8_t)((byte & 0x0F) | (q << 4)) : (uint8_t)((byte & 0xF0) | q);
          } else {
            codes[r * cols + b * 32 + i] = q;
          }
        }
        sf[r * nb + b] = (uint8_t)(e + 127);
      }
  });
}

// MXFP8 ([NeMo] MXFP8: fixed 32-value blocks, E8M0 power-of-two scales).
// Row-wise copy: codes [R, C] + E8M0 [R, C/32].  Column-wise copy: the
// transpose re-blocked along R ([NeMo] sub-channel: transposes need
// recomputation): codes [C, R] + E8M0 [C, R/32].  All tensors use E4M3.
void orc_mxfp8(const uint16_t* x, int64_t R, int64_t C, uint8_t* row_codes, uint8_t* row_sf,
               uint8_t* col_codes, uint8_t* col_sf) {
  if (row_codes)
    mxfp8_copy([&](int64_t r, int64_t c) { return bf16_value(x[r * C + c]); }, R, C, row_codes, row_sf);
  if (col_codes)
    mxfp8_copy([&](int64_t r, int64_t c) { return bf16_value(x[c * C + r]); }, C, R, col_codes, col_sf);
}

// MX quantization of any element format (E4M3 and E5M2: 1 byte per code, E2M1:
// packed): row-wise codes [R, C (/2)] + E8M0 [R, C/32]; column-wise copy the
// transpose re-blocked along R.  fmt = E4M3 is orc_mxfp8 ([NeMo] MXFP8); E5M2
// is the gradient variant ([FP8]: E5M2 for backward gradients); E2M1 is MXFP4
// ([NVFP4] technical deep dive: the 32-value blocks NVFP4 narrows to 16).
void orc_mx(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* row_codes, uint8_t* row_sf,
            uint8_t* col_codes, uint8_t* col_sf) {
  if (row_codes)
    mx_copy([&](int64_t r, int64_t c) { return bf16_value(x[r * C + c]); }, R, C, fmt, row_codes, row_sf);
  if (col_codes)
    mx_copy([&](int64_t r, int64_t c) { return bf16_value(x[c * C + r]); }, C, R, fmt, col_codes, col_sf);
}
int orc_mx_exponent_fmt(float a, int fmt) { return mx_exponent_fmt(a, fmt); }

// ---------------------------------------------------------------- NVFP4
// Quantizes one copy whose values are already materialised as floats v
// [rows, cols] (RHT applied when requested).  Two-level scaling ([NVFP4]):
//   A      = max |v| over the copy
//   s_enc  = 2688 / A   (2688 = 448 * 6: the largest block scale times the
//                        largest E2M1 value), 1 when A is 0 or not finite
//   ts_dec = A / 2688   (the stored FP32 tensor scale), 1 likewise
//   per block: d = (blockmax / 6) * s_enc, S = E4M3 RNE-sat encode of d;
//   if S decodes to 0 all codes of the block are +0, else
//   y = v * (s_enc / dec(S)) and the code is E2M1 (RNE-sat, or stochastic).
// Both quotients (s_enc and s_enc / dec(S)) are clamped to the largest finite
// float when they overflow, which only a tiny A (below about 4e-33) can cause.
// Reading: the constant 2688, the operation order and ts_dec = A / 2688 are
// choices; the pages give only "E4M3 per 16 values plus an FP32 per-tensor
// scale".  tile2d selects one scale per 16x16 tile (weights, [TE] "2D block
// scaling of weights"): the tile scale is written for each of its 16 rows.
// Packing: byte j of a row holds code 2j in its low nibble and 2j+1 high.
static void nvfp4_copy(const std::vector<float>& v, int64_t rows, int64_t cols, bool tile2d, bool sr,
                       uint64_t seed, uint64_t ctr_off, uint32_t copy_id, uint8_t* codes, uint8_t* sf,
                       float* ts_out, float* amax_out) {
  float A = 0.f;
  {
    int t = num_threads();
    std::vector<float> part(t, 0.f);
    int64_t chunk = (rows + t - 1) / t;
    parallel_for(t, [&](int64_t lo, int64_t hi) {
      for (int64_t i = lo; i < hi; ++i) {
        int64_t a = i * chunk, b = std::min<int64_t>(rows, a + chunk);
        float m = 0.f;
        if (a < b) m = absmax(v.data() + a * cols, (b - a) * cols, 1);
        part[i] = m;
      }
    }, rows * cols < (1 << 16) ? t + 1 : 1);
    for (float p : part) A = std::max(A, p);
  }
  bool ok = A > 0.f && std::isfinite(A);
  float s_enc = ok ? finite_scale(2688.0f / A) : 1.0f;
  float ts_dec = ok ? A / 2688.0f : 1.0f;
  int64_t nb = cols / 16;
  auto block_scale = [&](float bmax) {
    float d = (bmax / 6.0f) * s_enc;
    return encode(E4M3, d);
  };
  // For 2D tiles: the per-tile amax first (rows grouped by 16).
  std::vector<uint8_t> tile_sf;
  if (tile2d) {
    int64_t tr = rows / 16;
    tile_sf.assign(tr * nb, 0);
    parallel_for(tr, [&](int64_t lo, int64_t hi) {
      for (int64_t i = lo; i < hi; ++i)
        for (int64_t b = 0; b < nb; ++b) {
          float m = 0.f;
          for (int rr = 0; rr < 16; ++rr)
            m = std::max(m, absmax(v.data() + (i * 16 + rr) * cols + b * 16, 16, 1));
          tile_sf[i * nb + b] = block_scale(m);
        }
    });
  }
  parallel_for(rows, [&](int64_t lo, int64_t hi) {
    for (int64_t r = lo; r < hi; ++r)
      for (int64_t b = 0; b < nb; ++b) {
        const float* blk = v.data() + r * cols + b * 16;
        uint8_t S = tile2d ? tile_sf[(r / 16) * nb + b] : block_scale(absmax(blk, 16, 1));
        sf[r * nb + b] = S;
        float Sd = (float)decode(E4M3, S);
        uint8_t q[16];
        if (Sd == 0.f) {
          for (int i = 0; i < 16; ++i) q[i] = 0;
        } else {
          float f = finite_scale(s_enc / Sd);
          for (int i = 0; i < 16; ++i) {
            float y = blk[i] * f;
            if (sr) {
              uint64_t j = ctr_off + (uint64_t)(r * cols + b * 16 + i);
              q[i] = sr_encode_e2m1(y, sr_word(seed, j, copy_id));
            } else {
              q[i] = encode(E2M1, y);
            }
          }
        }
        for (int i = 0; i < 8; ++i) codes[r * (cols / 2) + b * 8 + i] = (uint8_t)(q[2 * i] | (q[2 * i + 1] << 4));
      }
  });
  if (ts_out) *ts_out = ts_dec;
  if (amax_out) *amax_out = A;
}

// NVFP4 quantize of x [R, C] bf16.  flags: 1 row-wise copy, 2 column-wise
// copy, 4 random Hadamard transform on the column-wise copy, 8 stochastic
// rounding (both copies), 16 2D 16x16 tiles (weights: no RHT, no SR; the
// column-wise copy is the exact transpose of the row-wise one and shares the
// tensor's single amax).  Row copy: codes [R, C/2], E4M3 scales [R, C/16];
// column copy: codes [C, R/2], scales [C, R/16].  Each copy has its own amax
// and tensor scale (the RHT copy's amax is that of the transformed values).
void orc_nvfp4(const uint16_t* x, int64_t R, int64_t C, unsigned flags, uint64_t seed,
               uint64_t ctr_off, uint32_t rht_seed, uint8_t* row_codes, uint8_t* row_sf,
               float* row_ts, float* row_amax, uint8_t* col_codes, uint8_t* col_sf, float* col_ts,
               float* col_amax) {
  bool tile2d = flags & 16, sr = flags & 8, rht = flags & 4;
  if (tile2d) {
    std::vector<float> v(R * C);
    for (int64_t i = 0; i < R * C; ++i) v[i] = bf16_value(x[i]);
    std::vector<uint8_t> rc(R * C / 2), rs(R * C / 16);
    float ts, am;
    nvfp4_copy(v, R, C, true, false, 0, 0, 0, rc.data(), rs.data(), &ts, &am);
    if (flags & 1) {
      std::memcpy(row_codes, rc.data(), rc.size());
      std::memcpy(row_sf, rs.data(), rs.size());
      if (row_ts) *row_ts = ts;
      if (row_amax) *row_amax = am;
    }
    if (flags & 2) {
      // exact transpose of codes (nibble by nibble) and of the tile scales
      for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c) {
          uint8_t q = (rc[r * (C / 2) + c / 2] >> ((c & 1) * 4)) & 0xF;
          uint8_t& dst = col_codes[c * (R / 2) + r / 2];
          if ((r & 1) == 0) dst = q; else dst = (uint8_t)(dst | (q << 4));
        }
      for (int64_t c = 0; c < C; ++c)
        for (int64_t rb = 0; rb < R / 16; ++rb) col_sf[c * (R / 16) + rb] = rs[(rb * 16) * (C / 16) + c / 16];
      if (col_ts) *col_ts = ts;
      if (col_amax) *col_amax = am;
    }
    return;
  }
  if (flags & 1) {
    std::vector<float> v(R * C);
    for (int64_t i = 0; i < R * C; ++i) v[i] = bf16_value(x[i]);
    nvfp4_copy(v, R, C, false, sr, seed, ctr_off, 0, row_codes, row_sf, row_ts, row_amax);
  }
  if (flags & 2) {
    std::vector<float> v(C * R);
    uint32_t signs = rht_sign_mask(rht_seed);
    parallel_for(C, [&](int64_t lo, int64_t hi) {
      float in[16], out[16];
      for (int64_t c = lo; c < hi; ++c)
        for (int64_t r0 = 0; r0 < R; r0 += 16) {
          for (int i = 0; i < 16; ++i) in[i] = bf16_value(x[(r0 + i) * C + c]);
          if (rht) rht16(in, signs, out); else std::memcpy(out, in, sizeof(in));
          for (int i = 0; i < 16; ++i) v[c * R + r0 + i] = out[i];
        }
    });
    nvfp4_copy(v, C, R, false, sr, seed, ctr_off, 1, col_codes, col_sf, col_ts, col_amax);
  }
}

// ---------------------------------------------------------------- sub-channel FP8
// Generic block FP8 ([NeMo] sub-channel scaling, e.g. 1x128 activation and
// 128x128 weight blocks): per block, scale = 448 / blockmax (fp32; 1 when the
// max is 0 or not finite), codes = E4M3 RNE-sat of x * scale, and the stored
// FP32 factor is scale_inv = 1 / scale.  block_rows = 1 (activations) or 128
// (weights).  Row copy: codes [R, C], scale_inv [R / block_rows, C / 128].
// Column copy: for 1x128 the transpose re-blocked 1x128 along R (codes [C, R],
// scale_inv [C, R / 128]); for 128x128 the transpose of the codes and of the
// block factors ([C / 128, R / 128]).
static void fp8_block_copy(const std::function<float(int64_t, int64_t)>& v, int64_t rows, int64_t cols,
                           int block_rows, uint8_t* codes, float* sinv) {
  int64_t nb = cols / 128, nrb = (rows + block_rows - 1) / block_rows;
  parallel_for(nrb, [&](int64_t lo, int64_t hi) {
    for (int64_t rb = lo; rb < hi; ++rb) {
      int64_t r0 = rb * block_rows, r1 = std::min<int64_t>(rows, r0 + block_rows);
      for (int64_t b = 0; b < nb; ++b) {
        float m = 0.f;
        for (int64_t r = r0; r < r1; ++r)
          for (int i = 0; i < 128; ++i) m = std::max(m, std::fabs(v(r, b * 128 + i)));
        float scale = (m > 0.f && std::isfinite(m)) ? finite_scale(448.0f / m) : 1.0f;
        for (int64_t r = r0; r < r1; ++r)
          for (int i = 0; i < 128; ++i) codes[r * cols + b * 128 + i] = encode(E4M3, v(r, b * 128 + i) * scale);
        sinv[rb * nb + b] = 1.0f / scale;
      }
    }
  });
}

void orc_fp8_block(const uint16_t* x, int64_t R, int64_t C, int block_rows, uint8_t* row_codes,
                   float* row_sinv, uint8_t* col_codes, float* col_sinv) {
  auto xv = [&](int64_t r, int64_t c) { return bf16_value(x[r * C + c]); };
  if (block_rows == 1) {
    if (row_codes) fp8_block_copy(xv, R, C, 1, row_codes, row_sinv);
    if (col_codes)
      fp8_block_copy([&](int64_t r, int64_t c) { return bf16_value(x[c * C + r]); }, C, R, 1, col_codes, col_sinv);
    return;
  }
  std::vector<uint8_t> rc(R * C);
  std::vector<float> rs(((R + 127) / 128) * (C / 128));
  fp8_block_copy(xv, R, C, 128, rc.data(), rs.data());
  if (row_codes) {
    std::memcpy(row_codes, rc.data(), rc.size());
    std::memcpy(row_sinv, rs.data(), rs.size() * sizeof(float));
  }
  if (col_codes) {
    for (int64_t r = 0; r < R; ++r)
      for (int64_t c = 0; c < C; ++c) col_codes[c * R + r] = rc[r * C + c];
    int64_t nrb = (R + 127) / 128, ncb = C / 128;
    for (int64_t cb = 0; cb < ncb; ++cb)
      for (int64_t rb = 0; rb < nrb; ++rb) col_sinv[cb * nrb + rb] = rs[rb * ncb + cb];
  }
}

// ---------------------------------------------------------------- GEMM
// Operand description for the FP64 GEMM.  kind: 0 bf16 (codes = bf16 bits),
// 1 per-tensor FP8 E4M3, 2 per-tensor FP8 E5M2 (value = code * ts),
// 3 MXFP8 (E4M3 code * 2^(sf - 127), sf [rows, K/32]),
// 4 NVFP4 (E2M1 nibble * E4M3 sf [rows, K/16] * ts),
// 5 block FP8 E4M3 (code * sinv[row / block_rows, k / 128]),
// 6 MXFP8 with E5M2 codes (code * 2^(sf - 127), sf [rows, K/32]),
// 7 MXFP4 (E2M1 nibble * 2^(sf - 127), sf [rows, K/32]).
struct OrcOperand {
  int32_t kind;
  int32_t block_rows;
  const void* codes;
  const void* sf;
  double ts;
};

static inline double deq(const OrcOperand& o, int64_t K, int64_t r, int64_t k) {
  switch (o.kind) {
    case 0: return (double)bf16_value(((const uint16_t*)o.codes)[r * K + k]);
    case 1: return decode(E4M3, ((const uint8_t*)o.codes)[r * K + k]) * o.ts;
    case 2: return decode(E5M2, ((const uint8_t*)o.codes)[r * K + k]) * o.ts;
    case 3: {
      uint8_t s = ((const uint8_t*)o.sf)[r * (K / 32) + k / 32];
      return decode(E4M3, ((const uint8_t*)o.codes)[r * K + k]) * std::ldexp(1.0, (int)s - 127);
    }
    case 4: {
      uint8_t b = ((const uint8_t*)o.codes)[r * (K / 2) + k / 2];
      uint8_t q = (k & 1) ? (b >> 4) : (b & 0xF);
      uint8_t s = ((const uint8_t*)o.sf)[r * (K / 16) + k / 16];
      return decode(E2M1, q) * decode(E4M3, s) * o.ts;
    }
    case 5: {
      float s = ((const float*)o.sf)[(r / o.block_rows) * (K / 128) + k / 128];
      return decode(E4M3, ((const uint8_t*)o.codes)[r * K + k]) * (double)s;
    }
    case 6: {
      uint8_t s = ((const uint8_t*)o.sf)[r * (K / 32) + k / 32];
      return decode(E5M2, ((const uint8_t*)o.codes)[r * K + k]) * std::ldexp(1.0, (int)s - 127);
    }
    case 7: {
      uint8_t b = ((const uint8_t*)o.codes)[r * (K / 2) + k / 2];
      uint8_t q = (k & 1) ? (b >> 4) : (b & 0xF);
      uint8_t s = ((const uint8_t*)o.sf)[r * (K / 32) + k / 32];
      return decode(E2M1, q) * std::ldexp(1.0, (int)s - 127);
    }
  }
  return std::nan("");
}

// C[m, n] = sum_k deq(a)[m, k] * deq(b)[n, k] in FP64 for each requested
// (m, n) pair, with bound[i] = sum_k |deq(a)[m, k] * deq(b)[n, k]| (the
// tolerance scale of the accuracy gate).  pairs = NULL means every (m, n) in
// row-major order.  Both operands are contiguous along K ("TN"), which is how
// Fprop, Dgrad and Wgrad are all posed ([TE] autocast vs pre-quantize: the
// three GEMMs of each linear are benchmarked separately).
void orc_gemm(const OrcOperand* a, const OrcOperand* b, int64_t M, int64_t N, int64_t K,
              const int64_t* pairs, int64_t npairs, double* c, double* bound) {
  int64_t n_out = pairs ? npairs : M * N;
  parallel_for(n_out, [&](int64_t lo, int64_t hi) {
    for (int64_t i = lo; i < hi; ++i) {
      int64_t m = pairs ? pairs[2 * i] : i / N;
      int64_t n = pairs ? pairs[2 * i + 1] : i % N;
      double s = 0.0, bs = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = deq(*a, K, m, k) * deq(*b, K, n, k);
        s += p;
        bs += std::fabs(p);
      }
      c[i] = s;
      if (bound) bound[i] = bs;
    }
  });
}

// Dequantizes rows [r0, r1) of an operand into FP64 (for numpy checks).
void orc_dequant(const OrcOperand* o, int64_t K, int64_t r0, int64_t r1, double* out) {
  for (int64_t r = r0; r < r1; ++r)
    for (int64_t k = 0; k < K; ++k) out[(r - r0) * K + k] = deq(*o, K, r, k);
}

// ---------------------------------------------------------------- shapes
// The 12 GEMMs of one transformer layer ([TE] "model configuration and
// training input" and "autocast vs pre-quantize"): M = micro_batch * seq
// tokens; QKV (K = hidden, N = 3 * hidden; the QKV Dgrad swaps K = 4096 and
// N = 12288), attention output (hidden x hidden, the smallest weight), MLP up
// (hidden -> intermediate) and MLP down (intermediate -> hidden), each as
// Fprop (M, K, N), Dgrad (M, N, K) and Wgrad (N, M, K).  Output rows of
// (m, k, n) triples, 12 of them, linear-major then Fprop/Dgrad/Wgrad.
void orc_layer_shapes(int64_t hidden, int64_t intermediate, int64_t micro_batch, int64_t seq,
                      int64_t* mkn /* [12][3] */) {
  int64_t M = micro_batch * seq;
  int64_t lin[4][2] = {{hidden, 3 * hidden}, {hidden, hidden}, {hidden, intermediate}, {intermediate, hidden}};
  for (int l = 0; l < 4; ++l) {
    int64_t K = lin[l][0], N = lin[l][1];
    int64_t t[3][3] = {{M, K, N}, {M, N, K}, {N, M, K}};
    for (int g = 0; g < 3; ++g)
      for (int j = 0; j < 3; ++j) mkn[(l * 3 + g) * 3 + j] = t[g][j];
  }
}

}  // extern "C"
