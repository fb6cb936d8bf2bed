// nvfp4_host.cu -- quantize-and-dequantize of a matrix that lives in host memory, streamed through
// the GPU in row chunks ("NVFP4 RL" blog, Sec. 6: the same pipeline serves online post-training
// quantization of checkpoints, which starts and ends in host memory).
//
// Chunks rotate over three internal streams, each with its own third of the caller's device
// staging workspace.  On each stream a chunk is copied in, quantized and dequantized by the fused
// kernel, and its outputs are copied out; the other streams' chunks meanwhile use the other copy
// direction and the SMs, so host->device copies, kernels and device->host copies overlap.  Events
// order the internal streams after everything already queued on the caller's stream, and the
// caller's stream after all of them, so the call behaves like any other asynchronous call on
// `stream`.  The internal streams and events are created once per device and kept; one host
// thread at a time queues work on them (a per-device mutex), so concurrent callers stay ordered
// after their own streams.
// Per-token results do not depend on chunking, so the outputs equal nvfp4_fused_roundtrip's.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "nvfp4.h"
#include "nvfp4_internal.h"

namespace {

constexpr int64_t kChunkBytesTarget = 32ll << 20;  // ~32 MB of input per chunk
constexpr int kStages = 3;                          // chunk buffers / internal streams

struct ChunkLayout {
  int64_t rows;   // rows per chunk
  size_t x, codes, scales, sdec, y, total;  // byte offsets within one chunk buffer
};

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// The per-device internal streams and events (created on first use, kept for the process).
struct Pipe {
  bool ready = false;
  cudaStream_t s[kStages] = {};
  cudaEvent_t start = nullptr;
  cudaEvent_t done[kStages] = {};
};
constexpr int kMaxDevices = 64;
std::mutex g_pipe_mutex[kMaxDevices];
Pipe g_pipe[kMaxDevices];

// Creates the device's pipe if needed; the caller holds g_pipe_mutex[device].
cudaError_t ensure_pipe(Pipe& p) {
  if (p.ready) return cudaSuccess;
  cudaError_t e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
  for (int i = 0; i < kStages && e == cudaSuccess; ++i) {
    e = cudaStreamCreateWithFlags(&p.s[i], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.done[i], cudaEventDisableTiming);
  }
  if (e != cudaSuccess) {  // leave nothing half made
    for (int i = 0; i < kStages; ++i) {
      if (p.s[i] != nullptr) cudaStreamDestroy(p.s[i]);
      if (p.done[i] != nullptr) cudaEventDestroy(p.done[i]);
      p.s[i] = nullptr;
      p.done[i] = nullptr;
    }
    if (p.start != nullptr) cudaEventDestroy(p.start);
    p.start = nullptr;
    return e;
  }
  p.ready = true;
  return cudaSuccess;
}

ChunkLayout layout_for(int64_t cols) {
  ChunkLayout L;
  L.rows = kChunkBytesTarget / (cols * 2);
  if (L.rows < 1) L.rows = 1;
  L.x = 0;
  L.codes = align256(L.x + static_cast<size_t>(L.rows * cols * 2));
  L.scales = align256(L.codes + static_cast<size_t>(L.rows * cols / 2));
  L.sdec = align256(L.scales + static_cast<size_t>(L.rows * cols / 16));
  L.y = align256(L.sdec + static_cast<size_t>(L.rows) * 4);
  L.total = align256(L.y + static_cast<size_t>(L.rows * cols * 2));
  return L;
}

}  // namespace

extern "C" size_t nvfp4_roundtrip_host_workspace_bytes(int64_t cols) {
  if (cols <= 0 || cols % nvfp4::kBlockElems != 0) return 0;
  return kStages * layout_for(cols).total;
}

extern "C" nvfp4_status nvfp4_fused_roundtrip_host(const void* x, int64_t rows, int64_t cols,
                                                   nvfp4_mode mode, uint8_t* codes,
                                                   uint8_t* block_scales, float* row_scale,
                                                   void* y, void* workspace,
                                                   size_t workspace_bytes,
                                                   nvfp4_stream_t stream) {
  if ((mode != NVFP4_MODE_SIX && mode != NVFP4_MODE_FOUR_OVER_SIX &&
       mode != NVFP4_MODE_FOUR_OVER_SIX_FP16) ||
      rows < 0)
    return NVFP4_ERR_INVALID_ARG;
  if (cols <= 0 || cols % nvfp4::kBlockElems != 0 || !nvfp4::quantize_cols_supported(cols))
    return NVFP4_ERR_SHAPE;
  if (rows == 0) return NVFP4_OK;
  if (x == nullptr || codes == nullptr || block_scales == nullptr || row_scale == nullptr ||
      y == nullptr)
    return NVFP4_ERR_INVALID_ARG;
  const ChunkLayout L = layout_for(cols);
  if (workspace == nullptr || workspace_bytes < kStages * L.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return NVFP4_ERR_WORKSPACE;

  int* status = nullptr;
  if (nvfp4::device_status_word(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices)
    return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_pipe_mutex[device]);
  Pipe& pipe = g_pipe[device];
  if (ensure_pipe(pipe) != cudaSuccess) return NVFP4_ERR_CUDA;
  cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
  nvfp4_status result = NVFP4_OK;
  auto check = [&](cudaError_t e) {
    if (e != cudaSuccess && result == NVFP4_OK) result = NVFP4_ERR_CUDA;
    return e == cudaSuccess;
  };
  if (!check(cudaEventRecord(pipe.start, caller))) return result;
  for (int i = 0; i < kStages; ++i)
    if (!check(cudaStreamWaitEvent(pipe.s[i], pipe.start, 0))) return result;

  for (int64_t r0 = 0, c = 0; r0 < rows; r0 += L.rows, ++c) {
    const int64_t n = (rows - r0 < L.rows) ? rows - r0 : L.rows;
    const int h = static_cast<int>(c % kStages);
    cudaStream_t st = pipe.s[h];
    unsigned char* base = static_cast<unsigned char*>(workspace) + h * L.total;
    const size_t xb = static_cast<size_t>(n * cols * 2);
    const size_t cb = static_cast<size_t>(n * cols / 2);
    const size_t sb = static_cast<size_t>(n * cols / 16);
    if (!check(cudaMemcpyAsync(base + L.x, static_cast<const unsigned char*>(x) + r0 * cols * 2, xb,
                               cudaMemcpyHostToDevice, st)))
      break;
    const nvfp4::QuantParams p = nvfp4::make_quant_params(
        base + L.x, n, cols, base + L.codes, base + L.scales,
        reinterpret_cast<float*>(base + L.sdec), base + L.y, status);
    if (!check(nvfp4::launch_quantize(mode, false, true, p, st))) break;
    if (!check(cudaMemcpyAsync(codes + r0 * cols / 2, base + L.codes, cb, cudaMemcpyDeviceToHost,
                               st)) ||
        !check(cudaMemcpyAsync(block_scales + r0 * cols / 16, base + L.scales, sb,
                               cudaMemcpyDeviceToHost, st)) ||
        !check(cudaMemcpyAsync(row_scale + r0, base + L.sdec, static_cast<size_t>(n) * 4,
                               cudaMemcpyDeviceToHost, st)) ||
        !check(cudaMemcpyAsync(static_cast<unsigned char*>(y) + r0 * cols * 2, base + L.y, xb,
                               cudaMemcpyDeviceToHost, st)))
      break;
  }
  // Whatever was queued, the caller's stream waits for all of it.
  for (int i = 0; i < kStages; ++i)
    if (check(cudaEventRecord(pipe.done[i], pipe.s[i])))
      check(cudaStreamWaitEvent(caller, pipe.done[i], 0));
  return result;
}
