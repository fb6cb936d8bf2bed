// nvfp4_aux.cu -- the streaming kernels around the quantizer:
//   * dequantize ("NVFP4 RL" blog, Sec. 3, dequantized backward): y = bf16(fp32(fp32(q*s) * S_dec));
//   * per-tensor amax for weights (Sec. 4 applies 4/6 to weights with one FP32 scale);
//   * the bounded-wait self-test that exercises the device-side failure path.
//
// Dequantize reads 0.5625 B and writes 2 B per element.  A persistent grid of warps walks the
// rows; lane l of a warp owns half-block l of each 256-element chunk, so the 4-byte code loads
// and the 16-byte BF16 stores of a warp are both contiguous.  Loads for several chunks are issued
// before any of them is consumed to keep enough bytes in flight.
#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

constexpr int kDequantWarps = 8;
constexpr int kDequantUnroll = 4;

template <bool kTensor>
__global__ void __launch_bounds__(kDequantWarps * 32) dequantize_kernel(const DequantParams p) {
  pdl_wait();  // global memory only after the previous kernel on the stream
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kDequantWarps + (threadIdx.x >> 5);
  const int64_t NW = static_cast<int64_t>(gridDim.x) * kDequantWarps;
  const int cols = p.cols;
  const int nhalf = cols / 8;  // 8-element half blocks per row
  const f32x2 nzero = pack2(-0.0f, -0.0f);
  const float tensor_sdec = kTensor ? p.scale[0] : 0.0f;

  for (int64_t row = gw; row < p.rows; row += NW) {
    const float sdec = kTensor ? tensor_sdec : p.scale[row];
    const f32x2 sdec2 = pack2(sdec, sdec);
    const uint32_t* codes_row = reinterpret_cast<const uint32_t*>(p.codes + row * (cols / 2));
    const uint8_t* scales_row = p.scales + row * (cols / kBlockElems);
    uint4* y_row = reinterpret_cast<uint4*>(p.y + row * cols);
    for (int base = 0; base < nhalf; base += 32 * kDequantUnroll) {
      uint32_t cw[kDequantUnroll];
      uint32_t sb[kDequantUnroll];
#pragma unroll
      for (int u = 0; u < kDequantUnroll; ++u) {
        const int h = base + u * 32 + lane;
        cw[u] = h < nhalf ? __ldcs(codes_row + h) : 0u;
        sb[u] = h < nhalf ? scales_row[h >> 1] : 0u;
      }
#pragma unroll
      for (int u = 0; u < kDequantUnroll; ++u) {
        const int h = base + u * 32 + lane;
        if (h < nhalf) {
          const uint32_t s_h2 = f16x2_from_e4m3x2(sb[u] | (sb[u] << 8));  // (s, s) in FP16
          uint32_t r[4];
          f16x2_from_e2m1x8(cw[u], r);
          uint32_t out[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const f32x2 qs = fma_f16x2_f32x2(r[j], s_h2, nzero);  // q*s, exact
            out[j] = bf16x2_from_f32x2(mul2(qs, sdec2));
          }
          __stcs(y_row + h, make_uint4(out[0], out[1], out[2], out[3]));
        }
      }
    }
  }
}

constexpr int kAmaxThreads = 256;
constexpr int kAmaxUnroll = 8;

// Partial max |x| per CTA over a grid-strided range of 16-byte vectors, plus the scalar tail.
__global__ void __launch_bounds__(kAmaxThreads) amax_partials_kernel(const uint16_t* x, int64_t n,
                                                                     float* partials) {
  // Global memory only after the previous kernel on the stream.  The encoder that consumes the
  // partials may start its own prologue (and its reads of x, which this kernel does not write)
  // right away; it waits for this grid before reading the partials.
  pdl_wait();
  pdl_trigger();
  const int64_t nvec = n / 8;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kAmaxThreads;
  uint32_t m2 = 0;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kAmaxThreads + threadIdx.x;
  for (; i + (kAmaxUnroll - 1) * stride < nvec; i += kAmaxUnroll * stride) {
    uint4 v[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) v[u] = __ldcg(xv + i + u * stride);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u)
      m2 = max_abs_bf16x2(m2, max_abs_bf16x2(max_abs_bf16x2(v[u].x, v[u].y),
                                             max_abs_bf16x2(v[u].z, v[u].w)));
  }
  for (; i < nvec; i += stride) {
    const uint4 v = __ldcg(xv + i);
    m2 = max_abs_bf16x2(m2, max_abs_bf16x2(max_abs_bf16x2(v.x, v.y), max_abs_bf16x2(v.z, v.w)));
  }
  float a = abs_max_of_pair(m2);
  if (blockIdx.x == 0)
    for (int64_t t = nvec * 8 + threadIdx.x; t < n; t += kAmaxThreads)
      a = fmaxf(a, __uint_as_float((static_cast<uint32_t>(x[t]) & 0x7FFFu) << 16));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  __shared__ float warp_max[kAmaxThreads / 32];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.0f;
    for (int w = 0; w < kAmaxThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
    partials[blockIdx.x] = m;
  }
}

__global__ void __launch_bounds__(256) amax_finalize_kernel(const float* partials, int n,
                                                            float* out) {
  float a = 0.0f;
  for (int i = threadIdx.x; i < n; i += 256) a = fmaxf(a, partials[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
  __shared__ float warp_max[8];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = 0.0f;
    for (int w = 0; w < 8; ++w) m = fmaxf(m, warp_max[w]);
    out[0] = m;
  }
}

// One warp waits on a barrier that expects one arrival nobody makes; the bounded wait gives up
// after timeout_ns and records the timeout.  Nothing else is pending, so the warp then returns.
__global__ void wait_timeout_selftest_kernel(int* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) mbar_init(&bar, 1);
  fence_barrier_init();
  __syncwarp();
  int ok = 1;
  if (threadIdx.x == 0) ok = mbar_wait_bounded(&bar, 0, timeout_ns) ? 1 : 0;
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  if (!ok && threadIdx.x == 0) record_status(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_dequantize(bool tensor_scale, const DequantParams& p, cudaStream_t stream) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  int64_t grid = (p.rows + kDequantWarps - 1) / kDequantWarps;
  const int64_t cap = static_cast<int64_t>(sm_count(device)) * 8;
  if (grid > cap) grid = cap;
  const LaunchOverride ov = launch_override();
  if (ov.max_ctas > 0 && grid > ov.max_ctas) grid = ov.max_ctas;
  if (grid < 1) grid = 1;
  if (tensor_scale)
    return launch_programmatic(dequantize_kernel<true>, dim3(static_cast<unsigned>(grid)),
                               dim3(kDequantWarps * 32), 0, stream, p);
  return launch_programmatic(dequantize_kernel<false>, dim3(static_cast<unsigned>(grid)),
                             dim3(kDequantWarps * 32), 0, stream, p);
}

cudaError_t launch_amax_partials(const uint16_t* x, int64_t n, float* partials, int* n_partials,
                                 cudaStream_t stream) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  const int64_t per_cta = static_cast<int64_t>(kAmaxThreads) * 8 * kAmaxUnroll;
  int64_t grid = (n + per_cta - 1) / per_cta;
  // Six CTAs per SM with eight 16-byte loads per thread in flight (measured best of 2-6 x 4-8).
  int64_t cap = static_cast<int64_t>(sm_count(device)) * 6;
  if (cap > kAmaxMaxPartials) cap = kAmaxMaxPartials;
  if (grid > cap) grid = cap;
  const LaunchOverride ov = launch_override();
  if (ov.max_ctas > 0 && grid > ov.max_ctas) grid = ov.max_ctas;
  if (grid < 1) grid = 1;
  *n_partials = static_cast<int>(grid);
  return launch_programmatic(amax_partials_kernel, dim3(static_cast<unsigned>(grid)),
                             dim3(kAmaxThreads), 0, stream, x, n, partials);
}

cudaError_t launch_amax_partials_into(const uint16_t* x, int64_t n, float* partials, int capacity,
                                      int* n_partials, bool* too_small, cudaStream_t stream) {
  *too_small = false;
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  const int64_t per_cta = static_cast<int64_t>(kAmaxThreads) * 8 * kAmaxUnroll;
  int64_t grid = (n + per_cta - 1) / per_cta;
  int64_t cap = static_cast<int64_t>(sm_count(device)) * 2;
  if (cap > kAmaxMaxPartials) cap = kAmaxMaxPartials;
  if (grid > cap) grid = cap;
  const LaunchOverride ov = launch_override();
  if (ov.max_ctas > 0 && grid > ov.max_ctas) grid = ov.max_ctas;
  if (grid < 1) grid = 1;
  if (grid > capacity) {
    *too_small = true;
    return cudaSuccess;
  }
  *n_partials = static_cast<int>(grid);
  return launch_programmatic(amax_partials_kernel, dim3(static_cast<unsigned>(grid)),
                             dim3(kAmaxThreads), 0, stream, x, n, partials);
}

cudaError_t launch_amax_finalize(const float* partials, int n, float* out, cudaStream_t stream) {
  amax_finalize_kernel<<<1, 256, 0, stream>>>(partials, n, out);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(int* status, uint64_t timeout_ns, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace nvfp4
