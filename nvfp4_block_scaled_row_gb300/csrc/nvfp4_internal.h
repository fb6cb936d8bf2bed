// nvfp4_internal.h -- host-side interface between the C ABI (nvfp4_capi.cu) and the kernel
// translation units.  Not installed; the public interface is include/nvfp4.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4_device.cuh"

namespace nvfp4 {

// Launches `kern` as a programmatic dependent of the previous kernel on `stream`: its blocks may
// start while that kernel finishes, and wait for it (pdl_wait) before touching global memory.
template <typename... Params, typename... Args>
cudaError_t launch_programmatic(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Bound on every device-side barrier wait of the library: 4 s.
constexpr uint64_t kWaitTimeoutNs = 4000000000ull;

// Quantize parameters with the library's wait bounds (and the withheld-row self-test setting of
// nvfp4_selftest_withhold_row); the caller fills the mode-specific fields.
QuantParams make_quant_params(const void* x, int64_t rows, int64_t cols, uint8_t* codes,
                              uint8_t* block_scales, float* scale, void* y, int* status);

// Launch-shape overrides (0 = automatic), set through nvfp4_set_launch_config.
struct LaunchOverride {
  int warps_per_cta;
  int stages;
  int max_ctas;
};
LaunchOverride launch_override();

// Multiprocessor count of the current device (cached per device).
int sm_count(int device);

// Quantize: row scale (kTensor = false) or tensor scale, plain or fused round trip.
// Chooses the ring shape from cols; returns cudaErrorInvalidValue when cols cannot be staged.
// after_amax_kernel: a tensor-scale launch that directly follows launch_amax_partials* on the
// same stream (p.amax_src = its partials) starts as that kernel's programmatic dependent.
cudaError_t launch_quantize(int mode, bool tensor_scale, bool fused, QuantParams p,
                            cudaStream_t stream, bool after_amax_kernel = false);

// Row-scale quantization of x and of its BF16 residual x - DQ(Q(x)) in one pass over x
// (p.res_codes, p.res_scales, p.res_scale_out receive the residual's outputs).
cudaError_t launch_quantize_residual(int mode, QuantParams p, cudaStream_t stream);

// TRACE-guided codes (see GuidedParams).
cudaError_t launch_quantize_guided(int mode, const GuidedParams& p, cudaStream_t stream);

// amax[r] = max |x[r][k]| over each row.
cudaError_t launch_row_amax(const uint16_t* x, int64_t rows, int cols, float* amax,
                            cudaStream_t stream);

// Whether the quantize kernels can stage a row of `cols` BF16 values.
bool quantize_cols_supported(int64_t cols);

cudaError_t launch_dequantize(bool tensor_scale, const DequantParams& p, cudaStream_t stream);

// Partial maxima of |x| over n BF16 values into `partials`; returns how many were written.
cudaError_t launch_amax_partials(const uint16_t* x, int64_t n, float* partials, int* n_partials,
                                 cudaStream_t stream);

// Reduces n partial maxima into *out.
cudaError_t launch_amax_finalize(const float* partials, int n, float* out, cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(int* status, uint64_t timeout_ns, cudaStream_t stream);

// As launch_amax_partials, but into a fixed-capacity buffer: sets *too_small and launches
// nothing when the partial maxima would not fit in `capacity` floats.
cudaError_t launch_amax_partials_into(const uint16_t* x, int64_t n, float* partials, int capacity,
                                      int* n_partials, bool* too_small, cudaStream_t stream);

// Host-side argument checks of the per-tensor quantize calls (the rules nvfp4_quantize_tensor
// applies, without the workspace); *noop is set for rows == 0.
int check_tensor_quantize_args(const void* x, int64_t rows, int64_t cols, int mode,
                               const uint8_t* codes, const uint8_t* block_scales,
                               const float* tensor_scale, bool* noop);

// Device address of the status word on the current device.
cudaError_t device_status_word(int** out);

}  // namespace nvfp4
