// nvfp4_noalloc.cu -- per-tensor quantization for callers that cannot allocate device memory.
//
// nvfp4_quantize_tensor needs a small device workspace from its caller: the tensor amax is
// reduced in two steps, and the per-CTA partial maxima of the first step have to live somewhere
// in global memory until the encoder reads them.  Some callers have no way to provide that
// buffer: code running where cudaMalloc is off limits (inside an allocator or memory-pool
// callback, in a host framework's plugin that receives only its input and output tensors and owns
// no allocator, or on a path where an allocation's implicit synchronization or fragmentation is
// unacceptable).  For them, nvfp4_quantize_tensor_noalloc keeps that scratch in a fixed array
// of device memory that belongs to the library itself.
//
// The array is a file-scope `static __device__` variable: every GPU that loads the library holds
// its kNoAllocPartials floats (2 KB) until the process exits.  Host code cannot use the array's
// name as a device address, so on the first call on each device this file asks the runtime for
// that device's address of the array (cudaGetSymbolAddress, with the device current), checks the
// result, and caches it; later calls on that device reuse the cached address.
//
// Every call shares the one array and it keeps whatever the last call left there.  Nothing in it
// has to start at zero: the amax pass writes every partial maximum the encoder then reads.  Two
// calls whose kernels overlap on the GPU (different streams without ordering between them) race
// on the array and can produce a wrong tensor amax; order such calls on one stream.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "nvfp4.h"
#include "nvfp4_internal.h"

namespace {

constexpr int kNoAllocPartials = 512;  // floats: room for the amax pass of a 256-SM GPU
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

std::atomic<float*> g_noalloc_ptr[kNoAllocMaxDevices];

// Device address of g_noalloc_partials on the current device (looked up on first use).
cudaError_t noalloc_scratch(float** out) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  if (device < 0 || device >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  float* cached = g_noalloc_ptr[device].load();
  if (cached == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_noalloc_partials);
    if (err != cudaSuccess) return err;
    cached = static_cast<float*>(p);
    g_noalloc_ptr[device].store(cached);
  }
  *out = cached;
  return cudaSuccess;
}

}  // namespace

extern "C" nvfp4_status nvfp4_quantize_tensor_noalloc(const void* x, int64_t rows, int64_t cols,
                                                      nvfp4_mode mode, uint8_t* codes,
                                                      uint8_t* block_scales, float* tensor_scale,
                                                      nvfp4_stream_t stream) {
  bool noop = false;
  const int st = nvfp4::check_tensor_quantize_args(x, rows, cols, mode, codes, block_scales,
                                                   tensor_scale, &noop);
  if (st != NVFP4_OK || noop) return static_cast<nvfp4_status>(st);
  float* scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return NVFP4_ERR_CUDA;
  int* status = nullptr;
  if (nvfp4::device_status_word(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int n_partials = 0;
  bool too_small = false;
  const cudaError_t err =
      nvfp4::launch_amax_partials_into(static_cast<const uint16_t*>(x), rows * cols, scratch,
                                       kNoAllocPartials, &n_partials, &too_small, s);
  if (err != cudaSuccess) return NVFP4_ERR_CUDA;
  if (too_small) return NVFP4_ERR_WORKSPACE;  // more partial maxima than the array holds
  nvfp4::QuantParams p = nvfp4::make_quant_params(x, rows, cols, codes, block_scales,
                                                  tensor_scale, nullptr, status);
  p.amax_src = scratch;
  p.n_amax = n_partials;
  return nvfp4::launch_quantize(mode, true, false, p, s, true) == cudaSuccess ? NVFP4_OK
                                                                              : NVFP4_ERR_CUDA;
}
