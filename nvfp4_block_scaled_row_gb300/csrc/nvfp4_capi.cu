// nvfp4_capi.cu -- the extern "C" entry points declared in include/nvfp4.h.
//
// Each entry point validates its arguments on the host (before any CUDA call, so a rejected
// call touches neither the device nor memory), then enqueues its kernels on the caller's stream
// and returns without synchronizing.  Device-side errors land in a per-device status word that
// nvfp4_get_device_status() reads.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4.h"
#include "nvfp4_internal.h"

// Device status word: NVFP4_OK, or the first device-side error recorded since the last clear.
__device__ int g_nvfp4_status = 0;

namespace nvfp4 {
namespace {

constexpr int kMaxDevices = 64;

std::atomic<int> g_override_warps{0};
std::atomic<int> g_override_stages{0};
std::atomic<int> g_override_max_ctas{0};
std::atomic<long long> g_withhold_row{-1};        // nvfp4_selftest_withhold_row
std::atomic<unsigned long long> g_withhold_timeout_ns{0};
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int*> g_status_ptr[kMaxDevices];

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  if (a == nullptr || b == nullptr || an == 0 || bn == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

bool valid_mode(int mode) {
  return mode == NVFP4_MODE_SIX || mode == NVFP4_MODE_FOUR_OVER_SIX ||
         mode == NVFP4_MODE_FOUR_OVER_SIX_FP16;
}
bool valid_kind(int kind) { return kind == NVFP4_SCALE_ROW || kind == NVFP4_SCALE_TENSOR; }

// The status word's device address for the current device (looked up once per device).
cudaError_t status_ptr(int** out) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  if (device >= 0 && device < kMaxDevices) {
    int* cached = g_status_ptr[device].load();
    if (cached != nullptr) {
      *out = cached;
      return cudaSuccess;
    }
  }
  void* p = nullptr;
  err = cudaGetSymbolAddress(&p, g_nvfp4_status);
  if (err != cudaSuccess) return err;
  if (device >= 0 && device < kMaxDevices) g_status_ptr[device].store(static_cast<int*>(p));
  *out = static_cast<int*>(p);
  return cudaSuccess;
}

nvfp4_status from_cuda(cudaError_t err) { return err == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

// Shared checks of the quantize calls.  Returns NVFP4_OK and sets *noop for rows == 0.
nvfp4_status check_quantize(const void* x, int64_t rows, int64_t cols, int mode,
                            const uint8_t* codes, const uint8_t* block_scales, const float* scale,
                            bool tensor_scale, const void* y, bool fused, bool* noop) {
  *noop = false;
  if (!valid_mode(mode) || rows < 0) return NVFP4_ERR_INVALID_ARG;
  if (cols <= 0 || cols % kBlockElems != 0 || !quantize_cols_supported(cols))
    return NVFP4_ERR_SHAPE;
  if (rows == 0) {
    *noop = true;
    return NVFP4_OK;
  }
  if (x == nullptr || codes == nullptr || block_scales == nullptr || scale == nullptr ||
      (fused && y == nullptr))
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scale, 4) || (fused && !aligned(y, 16)))
    return NVFP4_ERR_ALIGNMENT;
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols);
  const size_t nscale = tensor_scale ? 1 : static_cast<size_t>(rows);
  if (overlap(x, 2 * n, codes, n / 2) || overlap(x, 2 * n, block_scales, n / 16) ||
      overlap(x, 2 * n, scale, 4 * nscale) || (fused && overlap(x, 2 * n, y, 2 * n)) ||
      overlap(codes, n / 2, block_scales, n / 16) || overlap(codes, n / 2, scale, 4 * nscale) ||
      overlap(block_scales, n / 16, scale, 4 * nscale) ||
      (fused && (overlap(y, 2 * n, codes, n / 2) || overlap(y, 2 * n, block_scales, n / 16) ||
                 overlap(y, 2 * n, scale, 4 * nscale))))
    return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

nvfp4_status check_workspace(const void* workspace, size_t bytes) {
  if (workspace == nullptr || bytes < static_cast<size_t>(kAmaxMaxPartials) * sizeof(float) ||
      !aligned(workspace, 16))
    return NVFP4_ERR_WORKSPACE;
  return NVFP4_OK;
}

// Tensor-scale quantize (optionally fused): amax partials into the workspace, then the encoder.
nvfp4_status run_tensor(const void* x, int64_t rows, int64_t cols, int mode, uint8_t* codes,
                        uint8_t* block_scales, float* scale, void* y, bool fused, void* workspace,
                        cudaStream_t stream) {
  int* status = nullptr;
  cudaError_t err = status_ptr(&status);
  if (err != cudaSuccess) return NVFP4_ERR_CUDA;
  float* partials = static_cast<float*>(workspace);
  int n_partials = 0;
  err = launch_amax_partials(static_cast<const uint16_t*>(x), rows * cols, partials, &n_partials,
                             stream);
  if (err != cudaSuccess) return NVFP4_ERR_CUDA;
  QuantParams p = make_quant_params(x, rows, cols, codes, block_scales, scale, y, status);
  p.amax_src = partials;
  p.n_amax = n_partials;
  return from_cuda(launch_quantize(mode, true, fused, p, stream, true));
}

}  // namespace

int check_tensor_quantize_args(const void* x, int64_t rows, int64_t cols, int mode,
                               const uint8_t* codes, const uint8_t* block_scales,
                               const float* tensor_scale, bool* noop) {
  return check_quantize(x, rows, cols, mode, codes, block_scales, tensor_scale, true, nullptr,
                        false, noop);
}

cudaError_t device_status_word(int** out) { return status_ptr(out); }

QuantParams make_quant_params(const void* x, int64_t rows, int64_t cols, uint8_t* codes,
                              uint8_t* block_scales, float* scale, void* y, int* status) {
  QuantParams p{};
  p.x = static_cast<const uint16_t*>(x);
  p.rows = rows;
  p.cols = static_cast<int32_t>(cols);
  p.codes = codes;
  p.scales = block_scales;
  p.scale_out = scale;
  p.y = static_cast<uint16_t*>(y);
  p.status = status;
  p.timeout_ns = kWaitTimeoutNs;
  p.drain_timeout_ns = kWaitTimeoutNs;
  p.withhold_row = g_withhold_row.load();
  if (p.withhold_row >= 0) p.timeout_ns = g_withhold_timeout_ns.load();
  return p;
}

LaunchOverride launch_override() {
  return {g_override_warps.load(), g_override_stages.load(), g_override_max_ctas.load()};
}

int sm_count(int device) {
  int v = 0;
  if (device >= 0 && device < kMaxDevices) v = g_sm_count[device].load();
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v < 1)
    v = 1;
  if (device >= 0 && device < kMaxDevices) g_sm_count[device].store(v);
  return v;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

nvfp4_status nvfp4_quantize_rowwise(const void* x, int64_t rows, int64_t cols,
                                    const int32_t* group_offsets, int32_t num_groups,
                                    nvfp4_mode mode, uint8_t* codes, uint8_t* block_scales,
                                    float* row_scale, nvfp4_stream_t stream) {
  if (group_offsets == nullptr ? num_groups != 0 : (num_groups < 0 || !aligned(group_offsets, 4)))
    return NVFP4_ERR_INVALID_ARG;
  bool noop = false;
  nvfp4_status st = check_quantize(x, rows, cols, mode, codes, block_scales, row_scale, false,
                                   nullptr, false, &noop);
  if (st != NVFP4_OK || noop) return st;
  int* status = nullptr;
  if (status_ptr(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  QuantParams p = make_quant_params(x, rows, cols, codes, block_scales, row_scale, nullptr, status);
  p.offsets = group_offsets;
  p.num_groups = num_groups;
  return from_cuda(launch_quantize(mode, false, false, p, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize_residual(const void* x, int64_t rows, int64_t cols, nvfp4_mode mode,
                                     uint8_t* codes, uint8_t* block_scales, float* row_scale,
                                     uint8_t* res_codes, uint8_t* res_block_scales,
                                     float* res_row_scale, nvfp4_stream_t stream) {
  bool noop = false;
  nvfp4_status st = check_quantize(x, rows, cols, mode, codes, block_scales, row_scale, false,
                                   nullptr, false, &noop);
  if (st != NVFP4_OK || noop) return st;
  st = check_quantize(x, rows, cols, mode, res_codes, res_block_scales, res_row_scale, false,
                      nullptr, false, &noop);
  if (st != NVFP4_OK) return st;
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols);
  const void* a[3] = {codes, block_scales, row_scale};
  const size_t an[3] = {n / 2, n / 16, 4 * static_cast<size_t>(rows)};
  const void* b[3] = {res_codes, res_block_scales, res_row_scale};
  for (int i = 0; i < 3; ++i)
    for (int j = 0; j < 3; ++j)
      if (overlap(a[i], an[i], b[j], an[j])) return NVFP4_ERR_INVALID_ARG;
  int* status = nullptr;
  if (status_ptr(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  QuantParams p = make_quant_params(x, rows, cols, codes, block_scales, row_scale, nullptr, status);
  p.res_codes = res_codes;
  p.res_scales = res_block_scales;
  p.res_scale_out = res_row_scale;
  return from_cuda(launch_quantize_residual(mode, p, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_row_amax(const void* x, int64_t rows, int64_t cols, float* row_amax,
                            nvfp4_stream_t stream) {
  if (rows < 0) return NVFP4_ERR_INVALID_ARG;
  if (cols <= 0 || cols % kBlockElems != 0 || cols > (int64_t{1} << 30)) return NVFP4_ERR_SHAPE;
  if (rows == 0) return NVFP4_OK;
  if (x == nullptr || row_amax == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(row_amax, 4)) return NVFP4_ERR_ALIGNMENT;
  if (overlap(x, 2 * static_cast<size_t>(rows * cols), row_amax, 4 * static_cast<size_t>(rows)))
    return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_row_amax(static_cast<const uint16_t*>(x), rows, static_cast<int>(cols),
                                   row_amax, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_quantize_guided(const void* x, int64_t rows, int64_t cols, nvfp4_mode mode,
                                   const float* row_amax, const uint8_t* ref_codes,
                                   const uint8_t* ref_block_scales, uint8_t* codes,
                                   nvfp4_stream_t stream) {
  if (!valid_mode(mode) || rows < 0) return NVFP4_ERR_INVALID_ARG;
  if (cols <= 0 || cols % kBlockElems != 0 || cols > (int64_t{1} << 30)) return NVFP4_ERR_SHAPE;
  if (rows == 0) return NVFP4_OK;
  if (x == nullptr || row_amax == nullptr || ref_codes == nullptr || ref_block_scales == nullptr ||
      codes == nullptr)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(row_amax, 4) || !aligned(ref_codes, 4) || !aligned(codes, 4))
    return NVFP4_ERR_ALIGNMENT;
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols);
  if (overlap(codes, n / 2, x, 2 * n) || overlap(codes, n / 2, row_amax, 4 * static_cast<size_t>(rows)) ||
      overlap(codes, n / 2, ref_codes, n / 2) || overlap(codes, n / 2, ref_block_scales, n / 16))
    return NVFP4_ERR_INVALID_ARG;
  int* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  GuidedParams p{static_cast<const uint16_t*>(x), rows, static_cast<int32_t>(cols), row_amax,
                 ref_codes, ref_block_scales, codes, status, kWaitTimeoutNs, kWaitTimeoutNs,
                 static_cast<int64_t>(g_withhold_row.load())};
  if (p.withhold_row >= 0) p.timeout_ns = g_withhold_timeout_ns.load();
  return from_cuda(launch_quantize_guided(mode, p, reinterpret_cast<cudaStream_t>(stream)));
}

size_t nvfp4_tensor_workspace_bytes(void) {
  return static_cast<size_t>(kAmaxMaxPartials) * sizeof(float);
}

nvfp4_status nvfp4_quantize_tensor(const void* x, int64_t rows, int64_t cols, nvfp4_mode mode,
                                   uint8_t* codes, uint8_t* block_scales, float* tensor_scale,
                                   void* workspace, size_t workspace_bytes, nvfp4_stream_t stream) {
  bool noop = false;
  nvfp4_status st = check_quantize(x, rows, cols, mode, codes, block_scales, tensor_scale, true,
                                   nullptr, false, &noop);
  if (st != NVFP4_OK || noop) return st;
  if ((st = check_workspace(workspace, workspace_bytes)) != NVFP4_OK) return st;
  return run_tensor(x, rows, cols, mode, codes, block_scales, tensor_scale, nullptr, false,
                    workspace, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_tensor_amax(const void* x, int64_t n, float* amax, void* workspace,
                               size_t workspace_bytes, nvfp4_stream_t stream) {
  if (n < 0 || amax == nullptr || (n > 0 && x == nullptr)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(amax, 4) || (n > 0 && !aligned(x, 16))) return NVFP4_ERR_ALIGNMENT;
  nvfp4_status st = check_workspace(workspace, workspace_bytes);
  if (st != NVFP4_OK) return st;
  if (overlap(x, 2 * static_cast<size_t>(n), amax, 4)) return NVFP4_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* partials = static_cast<float*>(workspace);
  int n_partials = 0;
  if (launch_amax_partials(static_cast<const uint16_t*>(x), n, partials, &n_partials, s) !=
      cudaSuccess)
    return NVFP4_ERR_CUDA;
  return from_cuda(launch_amax_finalize(partials, n_partials, amax, s));
}

nvfp4_status nvfp4_quantize_tensor_with_amax(const void* x, int64_t rows, int64_t cols,
                                             nvfp4_mode mode, const float* amax, uint8_t* codes,
                                             uint8_t* block_scales, float* tensor_scale,
                                             nvfp4_stream_t stream) {
  bool noop = false;
  nvfp4_status st = check_quantize(x, rows, cols, mode, codes, block_scales, tensor_scale, true,
                                   nullptr, false, &noop);
  if (st != NVFP4_OK || noop) return st;
  if (amax == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(amax, 4)) return NVFP4_ERR_ALIGNMENT;
  int* status = nullptr;
  if (status_ptr(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  QuantParams p = make_quant_params(x, rows, cols, codes, block_scales, tensor_scale, nullptr, status);
  p.amax_src = amax;
  p.n_amax = 1;
  return from_cuda(launch_quantize(mode, true, false, p, reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* block_scales,
                              const float* scale, nvfp4_scale_kind kind, int64_t rows,
                              int64_t cols, void* y, nvfp4_stream_t stream) {
  if (!valid_kind(kind) || rows < 0) return NVFP4_ERR_INVALID_ARG;
  if (cols <= 0 || cols % kBlockElems != 0 || cols > (int64_t{1} << 30)) return NVFP4_ERR_SHAPE;
  if (rows == 0) return NVFP4_OK;
  if (codes == nullptr || block_scales == nullptr || scale == nullptr || y == nullptr)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(codes, 4) || !aligned(scale, 4) || !aligned(y, 16)) return NVFP4_ERR_ALIGNMENT;
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols);
  const size_t nscale = kind == NVFP4_SCALE_TENSOR ? 1 : static_cast<size_t>(rows);
  if (overlap(y, 2 * n, codes, n / 2) || overlap(y, 2 * n, block_scales, n / 16) ||
      overlap(y, 2 * n, scale, 4 * nscale))
    return NVFP4_ERR_INVALID_ARG;
  DequantParams p{codes, block_scales, scale, rows, static_cast<int32_t>(cols),
                  static_cast<uint16_t*>(y)};
  return from_cuda(launch_dequantize(kind == NVFP4_SCALE_TENSOR, p,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_fused_roundtrip(const void* x, int64_t rows, int64_t cols,
                                   nvfp4_scale_kind kind, nvfp4_mode mode, uint8_t* codes,
                                   uint8_t* block_scales, float* scale, void* y, void* workspace,
                                   size_t workspace_bytes, nvfp4_stream_t stream) {
  if (!valid_kind(kind)) return NVFP4_ERR_INVALID_ARG;
  const bool tensor = kind == NVFP4_SCALE_TENSOR;
  bool noop = false;
  nvfp4_status st =
      check_quantize(x, rows, cols, mode, codes, block_scales, scale, tensor, y, true, &noop);
  if (st != NVFP4_OK || noop) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (tensor) {
    if ((st = check_workspace(workspace, workspace_bytes)) != NVFP4_OK) return st;
    return run_tensor(x, rows, cols, mode, codes, block_scales, scale, y, true, workspace, s);
  }
  int* status = nullptr;
  if (status_ptr(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  QuantParams p = make_quant_params(x, rows, cols, codes, block_scales, scale, y, status);
  return from_cuda(launch_quantize(mode, false, true, p, s));
}

nvfp4_status nvfp4_get_device_status(int clear, nvfp4_status* status_out) {
  if (status_out == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_nvfp4_status, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (clear) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_nvfp4_status, &zero, sizeof(int)) != cudaSuccess)
      return NVFP4_ERR_CUDA;
  }
  *status_out = static_cast<nvfp4_status>(v);
  return NVFP4_OK;
}

const char* nvfp4_status_string(nvfp4_status status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_SHAPE: return "unsupported shape (cols must be a positive multiple of 16)";
    case NVFP4_ERR_ALIGNMENT: return "misaligned pointer";
    case NVFP4_ERR_CUDA: return "CUDA runtime error";
    case NVFP4_ERR_TIMEOUT: return "device-side bounded wait ran out";
    case NVFP4_ERR_OFFSETS: return "group offsets are not monotone from 0 to rows";
    case NVFP4_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
  }
  return "unknown status";
}

nvfp4_status nvfp4_set_launch_config(int warps_per_cta, int stages, int max_ctas) {
  if (warps_per_cta < 0 || warps_per_cta > kMaxWarpsPerCta || stages < 0 || stages > kMaxStages ||
      max_ctas < 0)
    return NVFP4_ERR_INVALID_ARG;
  g_override_warps.store(warps_per_cta);
  g_override_stages.store(stages);
  g_override_max_ctas.store(max_ctas);
  return NVFP4_OK;
}

nvfp4_status nvfp4_selftest_wait_timeout(uint64_t timeout_ns, nvfp4_stream_t stream) {
  int* status = nullptr;
  if (status_ptr(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  return from_cuda(launch_wait_timeout_selftest(status, timeout_ns ? timeout_ns : 1000000ull,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_selftest_withhold_row(int64_t row, uint64_t timeout_ns) {
  if (row < -1 || (row >= 0 && (timeout_ns == 0 || timeout_ns > kWaitTimeoutNs)))
    return NVFP4_ERR_INVALID_ARG;
  g_withhold_timeout_ns.store(timeout_ns);
  g_withhold_row.store(row);
  return NVFP4_OK;
}

int nvfp4_abi_version(void) { return 1; }

}  // extern "C"
