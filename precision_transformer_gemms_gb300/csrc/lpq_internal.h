// Internal declarations shared by the translation units of liblpq.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "lpq.h"

namespace lpq {

// Device-side bounded waits give up after this long (a healthy wait in these
// kernels lasts microseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Tensor-core instruction kinds used by the GEMM kernels.
enum { kKindF16 = 0, kKindF8F6F4 = 1, kKindMXF8 = 2, kKindNVF4 = 3, kKindMXF4 = 4 };

// Thread-local error text (capi.cu).
lpq_status set_error(lpq_status st, const char* fmt, ...);
lpq_status cuda_check(cudaError_t e, const char* what);

// Per-device launch settings (capi.cu), safe to call from several threads:
// the current device's SM count, and raising a kernel's dynamic shared-memory
// limit once per (device, kernel) -- cudaFuncSetAttribute acts on the current
// device only, so a second GPU in the same process needs its own call.
int device_sms();
lpq_status set_smem_attr(const void* kernel, int bytes);
// CTAs of `kernel` (with `threads` threads, no dynamic shared memory) that fit
// on one SM of the current device at once (at least 1); cached per device.
int resident_ctas(const void* kernel, int threads);

// Scale-factor geometry of the tensor-core layout.
// Atoms (4 scales of 128 rows) per 128-row group: one per 128 columns for
// MXFP8, two per 256 columns for MXFP4 (a 256-value k-step of packed E2M1
// holds 8 blocks of 32), four per 256 columns for NVFP4 (16 blocks of 16).
inline int64_t sf_kt_atoms(int32_t fmt, int64_t cols) {
  if (fmt == LPQ_MXFP8 || fmt == LPQ_MXFP8_E5M2) return (cols + 127) / 128;
  if (fmt == LPQ_MXFP4) return ((cols + 255) / 256) * 2;
  return ((cols + 255) / 256) * 4;  // NVFP4 / NVFP4_2D
}
inline int64_t sf_row_groups(int64_t rows) { return (rows + 127) / 128; }

// Quantizer launchers (quantize.cu).  `x` bf16 [rows, cols]; views validated.
lpq_status launch_quantize(const void* x, int64_t rows, int64_t cols, int32_t fmt, int32_t scaling,
                           uint32_t flags, uint64_t seed, uint64_t counter_offset, uint32_t rht_seed,
                           const lpq_delayed_state* state, lpq_qtensor* out, cudaStream_t stream);
lpq_status launch_amax(const void* x, int64_t rows, int64_t cols, bool rht, uint32_t rht_seed, float* amax,
                       float* rht_amax, cudaStream_t stream);
lpq_status launch_selftest_arith(int32_t which, uint64_t begin, uint64_t count, uint32_t param, int64_t* out,
                                 cudaStream_t stream);
lpq_status launch_scale_update(const lpq_delayed_state* state, const float* amax, float fmax,
                               cudaStream_t stream);

// GEMM launcher (gemm.cu).  Operands validated.
lpq_status launch_gemm(const lpq_qview* a, const lpq_qview* b, void* c, int32_t c_is_fp32, int64_t m,
                       int64_t n, int64_t k, const lpq_gemm_opts* opts, cudaStream_t stream);

// Device error word (gemm.cu owns it).
lpq_status read_and_clear_device_error(cudaStream_t stream, int32_t* code);
lpq_status launch_selftest_wait(uint64_t limit_ns, cudaStream_t stream);
lpq_status launch_mma_peak(int32_t kind, int32_t iters, int32_t with_sf, cudaStream_t stream);

}  // namespace lpq
