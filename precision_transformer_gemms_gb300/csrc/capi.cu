// C ABI of liblpq: argument validation, status codes and the host-only
// helpers (copy sizes, the 12 GEMM shapes of a layer).  No entry point
// allocates device memory or falls back to another format ("How to optimize
// Transformer-based models for low-precision training", interpreting
// real-model results: a silent fallback to FP8/BF16 is what to avoid).
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <map>
#include <set>
#include <utility>

#include "lpq_internal.h"

namespace lpq {

namespace {
thread_local char g_last_error[512] = "";

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_fp8_pertensor(int32_t f) { return f == LPQ_FP8_E4M3 || f == LPQ_FP8_E5M2; }
bool is_nvfp4(int32_t f) { return f == LPQ_NVFP4 || f == LPQ_NVFP4_2D; }
bool is_block(int32_t f) { return f == LPQ_FP8_BLOCK_1x128 || f == LPQ_FP8_BLOCK_128x128; }
bool is_mx8(int32_t f) { return f == LPQ_MXFP8 || f == LPQ_MXFP8_E5M2; }
// Formats with u8 block scales in the tensor-core scale layout.
bool is_u8_scaled(int32_t f) { return is_mx8(f) || f == LPQ_MXFP4 || is_nvfp4(f); }
bool valid_fmt(int32_t f) { return f >= LPQ_BF16 && f <= LPQ_MXFP4; }

// Column-block length of a format's row-wise scales (0 = none).
int64_t row_block(int32_t f) {
  switch (f) {
    case LPQ_MXFP8: case LPQ_MXFP8_E5M2: case LPQ_MXFP4: return 32;
    case LPQ_NVFP4: case LPQ_NVFP4_2D: return 16;
    case LPQ_FP8_BLOCK_1x128: case LPQ_FP8_BLOCK_128x128: return 128;
  }
  return 0;
}

// Rows of the input that a column-wise copy needs as a multiple.
int64_t col_rows_multiple(int32_t f) {
  switch (f) {
    case LPQ_MXFP8: case LPQ_MXFP8_E5M2: case LPQ_MXFP4: return 32;
    case LPQ_FP8_BLOCK_1x128: case LPQ_FP8_BLOCK_128x128: return 128;
  }
  return 16;
}

lpq_status check_arch() {
  static int ok = -1;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  static int checked_dev = -1;
  if (ok < 0 || checked_dev != dev) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    ok = (major == 10 && minor == 3) ? 1 : 0;
    checked_dev = dev;
    if (!ok)
      return set_error(LPQ_ERR_ARCH, "device %d is sm_%d%d; liblpq is built for sm_103a only", dev, major, minor);
  }
  return ok ? LPQ_OK : set_error(LPQ_ERR_ARCH, "device is not sm_103");
}

lpq_status check_view(const lpq_qview* v, const char* name, int32_t fmt, int64_t rows, int64_t cols, int colwise,
                      bool need_ts, bool need_amax) {
  if (v->fmt != fmt) return set_error(LPQ_ERR_INVALID_ARG, "%s.fmt is %d, expected %d", name, v->fmt, fmt);
  if (v->rows != rows || v->cols != cols)
    return set_error(LPQ_ERR_SHAPE, "%s is %lld x %lld, expected %lld x %lld", name, (long long)v->rows,
                     (long long)v->cols, (long long)rows, (long long)cols);
  if (v->colwise != colwise) return set_error(LPQ_ERR_INVALID_ARG, "%s.colwise must be %d", name, colwise);
  if (v->sf_layout != LPQ_SF_PLAIN && v->sf_layout != LPQ_SF_GEMM)
    return set_error(LPQ_ERR_INVALID_ARG, "%s.sf_layout %d", name, v->sf_layout);
  if (rows * cols > 0 && !v->codes) return set_error(LPQ_ERR_INVALID_ARG, "%s.codes is NULL", name);
  if (!aligned16(v->codes)) return set_error(LPQ_ERR_ALIGN, "%s.codes not 16-byte aligned", name);
  if (row_block(fmt) && rows * cols > 0 && !v->scales) return set_error(LPQ_ERR_INVALID_ARG, "%s.scales is NULL", name);
  if (row_block(fmt) && v->sf_layout == LPQ_SF_GEMM && !aligned16(v->scales))
    return set_error(LPQ_ERR_ALIGN, "%s.scales not 16-byte aligned", name);
  if (is_block(fmt) && (reinterpret_cast<uintptr_t>(v->scales) & 3u))
    return set_error(LPQ_ERR_ALIGN, "%s.scales not 4-byte aligned", name);
  if (need_ts && !v->tensor_scale) return set_error(LPQ_ERR_INVALID_ARG, "%s.tensor_scale is NULL", name);
  if (need_amax && !v->amax) return set_error(LPQ_ERR_INVALID_ARG, "%s.amax is NULL", name);
  return LPQ_OK;
}
}  // namespace

lpq_status set_error(lpq_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

lpq_status cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return LPQ_OK;
  return set_error(LPQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {
std::mutex g_dev_mu;
std::set<int>* g_sms_known = nullptr;  // devices whose SM count is cached
int g_sms_of[256];
std::set<std::pair<int, const void*>>* g_smem_set = nullptr;  // (device, kernel) pairs already raised
std::map<std::pair<int, const void*>, int>* g_resident = nullptr;  // (device, kernel) -> CTAs per SM
}  // namespace

int device_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_sms_known) g_sms_known = new std::set<int>();
  if (dev >= 0 && dev < 256 && g_sms_known->count(dev)) return g_sms_of[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 148;
  if (dev >= 0 && dev < 256) {
    g_sms_of[dev] = n;
    g_sms_known->insert(dev);
  }
  return n;
}

int resident_ctas(const void* kernel, int threads) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_resident) g_resident = new std::map<std::pair<int, const void*>, int>();
  auto it = g_resident->find({dev, kernel});
  if (it != g_resident->end()) return it->second;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) n = 1;
  (*g_resident)[{dev, kernel}] = n;
  return n;
}

lpq_status set_smem_attr(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_check(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!g_smem_set) g_smem_set = new std::set<std::pair<int, const void*>>();
  if (g_smem_set->count({dev, kernel})) return LPQ_OK;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return cuda_check(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  g_smem_set->insert({dev, kernel});
  return LPQ_OK;
}

}  // namespace lpq

using namespace lpq;

extern "C" {

int32_t lpq_version(void) { return 100; }

const char* lpq_last_error(void) { return g_last_error; }

lpq_status lpq_copy_bytes(int32_t fmt, int64_t rows, int64_t cols, int32_t sf_layout, size_t* codes_bytes,
                          size_t* scale_bytes) {
  if (!codes_bytes || !scale_bytes) return set_error(LPQ_ERR_INVALID_ARG, "NULL output pointer");
  if (!valid_fmt(fmt)) return set_error(LPQ_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (rows < 0 || cols < 0) return set_error(LPQ_ERR_SHAPE, "negative dimension");
  if (sf_layout != LPQ_SF_PLAIN && sf_layout != LPQ_SF_GEMM) return set_error(LPQ_ERR_INVALID_ARG, "sf_layout");
  const int64_t blk = row_block(fmt);
  if (blk && cols % blk) return set_error(LPQ_ERR_SHAPE, "cols %lld not a multiple of %lld", (long long)cols, (long long)blk);
  const size_t n = (size_t)rows * (size_t)cols;
  size_t cb = 0, sb = 0;
  switch (fmt) {
    case LPQ_BF16: cb = 2 * n; break;
    case LPQ_FP8_E4M3: case LPQ_FP8_E5M2: cb = n; break;
    case LPQ_MXFP8: case LPQ_MXFP8_E5M2: case LPQ_MXFP4: case LPQ_NVFP4: case LPQ_NVFP4_2D:
      cb = is_mx8(fmt) ? n : n / 2;
      sb = sf_layout == LPQ_SF_GEMM ? (size_t)sf_row_groups(rows) * (size_t)sf_kt_atoms(fmt, cols) * 512
                                    : (size_t)rows * (size_t)(cols / blk);
      break;
    case LPQ_FP8_BLOCK_1x128: cb = n; sb = 4 * (size_t)rows * (size_t)(cols / 128); break;
    case LPQ_FP8_BLOCK_128x128: cb = n; sb = 4 * (size_t)((rows + 127) / 128) * (size_t)(cols / 128); break;
  }
  *codes_bytes = cb;
  *scale_bytes = sb;
  return LPQ_OK;
}

lpq_status lpq_quantize(const void* x, int64_t rows, int64_t cols, int32_t fmt, int32_t scaling, uint32_t flags,
                        uint64_t seed, uint64_t counter_offset, uint32_t rht_seed, const lpq_delayed_state* state,
                        lpq_qtensor* out, lpq_stream_t stream) {
  if (!valid_fmt(fmt)) return set_error(LPQ_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (!out) return set_error(LPQ_ERR_INVALID_ARG, "out is NULL");
  if (rows < 0 || cols < 0) return set_error(LPQ_ERR_SHAPE, "negative dimension");
  if (flags & ~uint32_t(LPQ_ROWWISE | LPQ_COLWISE | LPQ_RHT_COLWISE | LPQ_STOCHASTIC | LPQ_GIVEN_AMAX))
    return set_error(LPQ_ERR_INVALID_ARG, "unknown flag bits 0x%x", flags);
  const bool do_row = flags & LPQ_ROWWISE, do_col = flags & LPQ_COLWISE;
  if (!do_row && !do_col) return set_error(LPQ_ERR_INVALID_ARG, "neither LPQ_ROWWISE nor LPQ_COLWISE requested");
  if ((flags & (LPQ_RHT_COLWISE | LPQ_STOCHASTIC)) && fmt != LPQ_NVFP4)
    return set_error(LPQ_ERR_UNSUPPORTED, "Hadamard transform and stochastic rounding apply to 1D NVFP4 only");
  if ((flags & LPQ_RHT_COLWISE) && !do_col)
    return set_error(LPQ_ERR_INVALID_ARG, "LPQ_RHT_COLWISE needs LPQ_COLWISE");
  if (counter_offset % 4) return set_error(LPQ_ERR_INVALID_ARG, "counter_offset must be a multiple of 4");
  const bool pt = is_fp8_pertensor(fmt);
  if (pt && scaling != LPQ_SCALING_CURRENT && scaling != LPQ_SCALING_DELAYED)
    return set_error(LPQ_ERR_INVALID_ARG, "scaling %d", scaling);
  if (!pt && scaling != LPQ_SCALING_CURRENT)
    return set_error(LPQ_ERR_UNSUPPORTED, "delayed scaling applies to per-tensor FP8 only");
  if ((flags & LPQ_GIVEN_AMAX) && !((pt && scaling == LPQ_SCALING_CURRENT) || is_nvfp4(fmt)))
    return set_error(LPQ_ERR_UNSUPPORTED, "LPQ_GIVEN_AMAX applies to current-scaled FP8 and NVFP4 only");
  if (pt && scaling == LPQ_SCALING_DELAYED) {
    if (!state || !state->scale || !state->scale_inv || !state->amax_history || !state->pos || state->len < 1 ||
        state->len > 1024)
      return set_error(LPQ_ERR_INVALID_ARG, "delayed scaling needs a complete state");
  }
  if (rows * cols > 0 && !x) return set_error(LPQ_ERR_INVALID_ARG, "x is NULL");
  if (!aligned16(x)) return set_error(LPQ_ERR_ALIGN, "x not 16-byte aligned");
  // shape rules
  if (cols % 16) return set_error(LPQ_ERR_SHAPE, "cols %lld not a multiple of 16", (long long)cols);
  const int64_t blk = row_block(fmt);
  if (blk && cols % blk) return set_error(LPQ_ERR_SHAPE, "cols %lld not a multiple of %lld", (long long)cols, (long long)blk);
  if (fmt == LPQ_NVFP4_2D && rows % 16) return set_error(LPQ_ERR_SHAPE, "NVFP4_2D needs rows % 16 == 0");
  if (do_col && rows % col_rows_multiple(fmt))
    return set_error(LPQ_ERR_SHAPE, "column-wise copy needs rows %% %lld == 0 (rows = %lld)",
                     (long long)col_rows_multiple(fmt), (long long)rows);
  const bool need_ts = pt || is_nvfp4(fmt);
  const bool need_amax = pt || is_nvfp4(fmt);
  lpq_status st;
  if (do_row && (st = check_view(&out->row, "out.row", fmt, rows, cols, 0, need_ts, need_amax)) != LPQ_OK) return st;
  if (do_col && (st = check_view(&out->col, "out.col", fmt, cols, rows, 1, need_ts, need_amax)) != LPQ_OK) return st;
  if ((st = check_arch()) != LPQ_OK) return st;
  return launch_quantize(x, rows, cols, fmt, scaling, flags, seed, counter_offset, rht_seed, state, out,
                         reinterpret_cast<cudaStream_t>(stream));
}

lpq_status lpq_amax(const void* x, int64_t rows, int64_t cols, uint32_t flags, uint32_t rht_seed, float* amax,
                    float* rht_amax, lpq_stream_t stream) {
  if (flags & ~uint32_t(LPQ_RHT_COLWISE)) return set_error(LPQ_ERR_INVALID_ARG, "lpq_amax flags 0x%x", flags);
  const bool rht = flags & LPQ_RHT_COLWISE;
  if (!amax && !(rht && rht_amax)) return set_error(LPQ_ERR_INVALID_ARG, "no amax output");
  if (rht && !rht_amax) return set_error(LPQ_ERR_INVALID_ARG, "LPQ_RHT_COLWISE needs rht_amax");
  if (rows < 0 || cols < 0) return set_error(LPQ_ERR_SHAPE, "negative dimension");
  if (cols % 16) return set_error(LPQ_ERR_SHAPE, "cols %lld not a multiple of 16", (long long)cols);
  if (rht && rows % 16) return set_error(LPQ_ERR_SHAPE, "the RHT amax needs rows %% 16 == 0 (rows = %lld)", (long long)rows);
  if (rows * cols > 0 && !x) return set_error(LPQ_ERR_INVALID_ARG, "x is NULL");
  if (!aligned16(x)) return set_error(LPQ_ERR_ALIGN, "x not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(amax) & 3u) || (reinterpret_cast<uintptr_t>(rht_amax) & 3u))
    return set_error(LPQ_ERR_ALIGN, "amax outputs not 4-byte aligned");
  lpq_status st = check_arch();
  if (st != LPQ_OK) return st;
  return launch_amax(x, rows, cols, rht, rht_seed, amax, rht_amax, reinterpret_cast<cudaStream_t>(stream));
}

lpq_status lpq_scale_update(const lpq_delayed_state* state, const float* amax, float fmax, lpq_stream_t stream) {
  if (!state || !amax || !state->scale || !state->scale_inv || !state->amax_history || !state->pos)
    return set_error(LPQ_ERR_INVALID_ARG, "NULL state or amax");
  if (state->len < 1 || state->len > 1024) return set_error(LPQ_ERR_INVALID_ARG, "history length %d", state->len);
  if (!(fmax > 0.f)) return set_error(LPQ_ERR_INVALID_ARG, "fmax must be positive");
  lpq_status st = check_arch();
  if (st != LPQ_OK) return st;
  return launch_scale_update(state, amax, fmax, reinterpret_cast<cudaStream_t>(stream));
}

lpq_status lpq_gemm(int32_t layout, const lpq_qview* a, const lpq_qview* b, void* c, int32_t c_is_fp32, int64_t m,
                    int64_t n, int64_t k, lpq_stream_t stream) {
  return lpq_gemm_ex(layout, a, b, c, c_is_fp32, m, n, k, nullptr, stream);
}

lpq_status lpq_gemm_ex(int32_t layout, const lpq_qview* a, const lpq_qview* b, void* c, int32_t c_is_fp32, int64_t m,
                       int64_t n, int64_t k, const lpq_gemm_opts* opts, lpq_stream_t stream) {
  if (!a || !b) return set_error(LPQ_ERR_INVALID_ARG, "NULL operand");
  if (opts) {
    if (opts->single_cta < 0 || opts->single_cta > 1 || opts->scale_copies < 0 || opts->scale_copies > 1 ||
        opts->direct_store < 0 || opts->direct_store > 1 || opts->whole_tiles < 0 || opts->whole_tiles > 1 ||
        !(opts->tile_n == 0 || opts->tile_n == 128 || opts->tile_n == 256))
      return set_error(LPQ_ERR_INVALID_ARG,
                       "lpq_gemm_opts: single_cta, scale_copies, direct_store, whole_tiles 0/1; tile_n 0, 128 or 256");
    for (int i = 0; i < 3; ++i)
      if (opts->reserved[i]) return set_error(LPQ_ERR_INVALID_ARG, "lpq_gemm_opts.reserved must be 0");
  }
  if (layout < LPQ_FPROP || layout > LPQ_WGRAD) return set_error(LPQ_ERR_INVALID_ARG, "layout %d", layout);
  if (m < 0 || n < 0 || k < 0) return set_error(LPQ_ERR_SHAPE, "negative dimension");
  if (a->rows != m || a->cols != k) return set_error(LPQ_ERR_SHAPE, "a is %lld x %lld, expected m x k = %lld x %lld",
                                                     (long long)a->rows, (long long)a->cols, (long long)m, (long long)k);
  if (b->rows != n || b->cols != k) return set_error(LPQ_ERR_SHAPE, "b is %lld x %lld, expected n x k = %lld x %lld",
                                                     (long long)b->rows, (long long)b->cols, (long long)n, (long long)k);
  const int want_a = layout == LPQ_WGRAD ? 1 : 0, want_b = layout == LPQ_FPROP ? 0 : 1;
  if (a->colwise != want_a || b->colwise != want_b)
    return set_error(LPQ_ERR_INVALID_ARG, "layout %d reads a %s a and a %s b", layout, want_a ? "column-wise" : "row-wise",
                     want_b ? "column-wise" : "row-wise");
  const int32_t fa = a->fmt, fb = b->fmt;
  const bool pair_ok = (fa == LPQ_BF16 && fb == LPQ_BF16) || (is_fp8_pertensor(fa) && is_fp8_pertensor(fb)) ||
                       (is_mx8(fa) && is_mx8(fb)) || (fa == LPQ_MXFP4 && fb == LPQ_MXFP4) ||
                       (is_nvfp4(fa) && is_nvfp4(fb)) ||
                       (is_block(fa) && is_block(fb));
  if (!pair_ok) return set_error(LPQ_ERR_UNSUPPORTED, "no GEMM for the pairing %d x %d (no fallback)", fa, fb);
  const int64_t kmul = is_block(fa) ? 128 : 32;
  if (k % kmul) return set_error(LPQ_ERR_SHAPE, "k %lld not a multiple of %lld", (long long)k, (long long)kmul);
  if (m > 0 && n > 0) {
    if (!c) return set_error(LPQ_ERR_INVALID_ARG, "c is NULL");
    if (!aligned16(c)) return set_error(LPQ_ERR_ALIGN, "c not 16-byte aligned");
    if (k > 0) {
      for (const lpq_qview* v : {a, b}) {
        if (!v->codes) return set_error(LPQ_ERR_INVALID_ARG, "operand codes NULL");
        if (!aligned16(v->codes)) return set_error(LPQ_ERR_ALIGN, "operand codes not 16-byte aligned");
        if (is_u8_scaled(v->fmt)) {
          if (v->sf_layout != LPQ_SF_GEMM)
            return set_error(LPQ_ERR_INVALID_ARG, "block-scaled operands need LPQ_SF_GEMM scales");
          if (!v->scales || !aligned16(v->scales)) return set_error(LPQ_ERR_ALIGN, "operand scales NULL/unaligned");
        }
        if (is_block(v->fmt)) {
          if (v->sf_layout != LPQ_SF_GEMM)
            return set_error(LPQ_ERR_INVALID_ARG, "sub-channel operands need LPQ_SF_GEMM factors");
          if (!v->scales || (reinterpret_cast<uintptr_t>(v->scales) & 3u))
            return set_error(LPQ_ERR_ALIGN, "operand factors NULL/unaligned");
        }
        if ((is_fp8_pertensor(v->fmt) || is_nvfp4(v->fmt)) && !v->tensor_scale)
          return set_error(LPQ_ERR_INVALID_ARG, "operand tensor_scale NULL");
      }
    }
  }
  lpq_status st = check_arch();
  if (st != LPQ_OK) return st;
  return launch_gemm(a, b, c, c_is_fp32, m, n, k, opts, reinterpret_cast<cudaStream_t>(stream));
}

lpq_status lpq_layer_shapes(const lpq_transformer_cfg* cfg, lpq_gemm_shape out[12], int32_t* count) {
  if (!cfg || !out || !count) return set_error(LPQ_ERR_INVALID_ARG, "NULL argument");
  if (cfg->hidden <= 0 || cfg->intermediate <= 0 || cfg->micro_batch <= 0 || cfg->seq <= 0)
    return set_error(LPQ_ERR_SHAPE, "config dimensions must be positive");
  const int64_t M = cfg->micro_batch * cfg->seq;
  const int64_t h = cfg->hidden, f = cfg->intermediate;
  const struct {
    const char* name;
    int64_t k, n;
  } lin[4] = {{"qkv", h, 3 * h}, {"attn_out", h, h}, {"mlp_up", h, f}, {"mlp_down", f, h}};
  const char* pass[3] = {"fprop", "dgrad", "wgrad"};
  int i = 0;
  for (const auto& l : lin)
    for (int p = 0; p < 3; ++p, ++i) {
      lpq_gemm_shape& s = out[i];
      memset(&s, 0, sizeof(s));
      snprintf(s.name, sizeof(s.name), "%s_%s", l.name, pass[p]);
      s.layout = p;
      if (p == 0) { s.m = M; s.k = l.k; s.n = l.n; }
      else if (p == 1) { s.m = M; s.k = l.n; s.n = l.k; }
      else { s.m = l.n; s.k = M; s.n = l.k; }
    }
  *count = 12;
  return LPQ_OK;
}

lpq_status lpq_device_status(lpq_stream_t stream, int32_t* code) {
  if (!code) return set_error(LPQ_ERR_INVALID_ARG, "code is NULL");
  return read_and_clear_device_error(reinterpret_cast<cudaStream_t>(stream), code);
}

lpq_status lpq_selftest_wait(uint64_t limit_ns, lpq_stream_t stream) {
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return set_error(LPQ_ERR_INVALID_ARG, "limit_ns must be in (0, 1 s]");
  lpq_status st = check_arch();
  if (st != LPQ_OK) return st;
  return launch_selftest_wait(limit_ns, reinterpret_cast<cudaStream_t>(stream));
}

lpq_status lpq_selftest_arith(int32_t which, uint64_t begin, uint64_t count, uint32_t param, int64_t* result,
                              lpq_stream_t stream) {
  if (which < 0 || which > 2) return set_error(LPQ_ERR_INVALID_ARG, "which %d", which);
  if (!result || (reinterpret_cast<uintptr_t>(result) & 7u)) return set_error(LPQ_ERR_INVALID_ARG, "result");
  const uint64_t limit = which == 0 ? 0x7F800001ull : which == 1 ? 8ull * 0x100000000ull : 1ull << 24;
  if (begin > limit || count > limit - begin) return set_error(LPQ_ERR_INVALID_ARG, "index range beyond %llu",
                                                               (unsigned long long)limit);
  lpq_status st = check_arch();
  if (st != LPQ_OK) return st;
  return launch_selftest_arith(which, begin, count, param, result, reinterpret_cast<cudaStream_t>(stream));
}

lpq_status lpq_mma_peak(int32_t kind, int32_t iters, int32_t with_scale_copies, lpq_stream_t stream) {
  if (kind < 0 || kind > 3) return set_error(LPQ_ERR_INVALID_ARG, "kind %d", kind);
  if (iters < 1 || iters > (1 << 24)) return set_error(LPQ_ERR_INVALID_ARG, "iters %d", iters);
  const bool ok_mode = (with_scale_copies >= 0 && with_scale_copies <= 1) ||
                       (with_scale_copies >= 2 && with_scale_copies <= 5 && kind == 3) || with_scale_copies == 6 ||
                       with_scale_copies == 8 ||
                       (with_scale_copies == 7 && (kind == 2 || kind == 3));
  if (!ok_mode) return set_error(LPQ_ERR_INVALID_ARG, "with_scale_copies %d for kind %d", with_scale_copies, kind);
  lpq_status st = check_arch();
  if (st != LPQ_OK) return st;
  return launch_mma_peak(kind, iters, with_scale_copies, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
