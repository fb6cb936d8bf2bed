// nvfp4_gemm.cu -- the consumer side of the quantizer: the MMA-ready block-scale layout and an
// NVFP4 x NVFP4 GEMM for the forward y = x . Q(w) ("NVFP4 RL" blog, Sec. 3: the forward executed
// is y = x . Q(w); Sec. 2: activations carry a per-token FP32 scale).
//
// Block-scaled tensor-core GEMMs read E4M3 block scales in tiles of 128 rows x 4 scale columns
// (512 bytes each, tiles row-major over [ceil(rows/128)][ceil(cols/64)]): inside a tile the scale
// of (row r, scale column c) sits at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4), so one
// 16-byte read gives a row quadruple's scales for four consecutive 16-element blocks.  The
// quantizer writes scales row-major; nvfp4_swizzle_block_scales re-lays them (zero padding).
//
// nvfp4_gemm_nt runs the block-scaled FP4 matrix product on the tensor cores through cuBLASLt
// (FP32 accumulation and output into the caller's workspace) and then applies both FP32 scales in
// one epilogue pass: y[m][n] = bf16(fp32(fp32(D[m][n] * S_x[m]) * S_w)).
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cublasLt.h>
#include <cuda_runtime.h>

#include "nvfp4.h"
#include "nvfp4_internal.h"

namespace {

constexpr size_t kLtWorkspace = 32ull << 20;  // cuBLASLt scratch inside the caller's workspace

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// One thread per 16-byte line of the swizzled layout: line r32 of tile (tr, tc) holds, for each
// row quadrant q, the four scales of row tr*128 + q*32 + r32 at scale columns tc*4 .. tc*4+3
// (padding 0).  Rows whose four scales are 4-byte aligned in the source are read as one word.
__global__ void swizzle_scales_kernel(const uint8_t* __restrict__ in, int64_t rows, int64_t scols,
                                      uint8_t* __restrict__ out, int64_t lines, int64_t tiles_c) {
  for (int64_t l = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; l < lines;
       l += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t tile = l >> 5;
    const int r32 = static_cast<int>(l & 31);
    const int64_t tr = tile / tiles_c, tc = tile - tr * tiles_c;
    const int64_t c0 = tc * 4;
    uint32_t word[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t r = tr * 128 + q * 32 + r32;
      uint32_t w = 0;
      if (r < rows) {
        const uint8_t* src = in + r * scols + c0;
        if (c0 + 4 <= scols && (reinterpret_cast<uintptr_t>(src) & 3) == 0) {
          w = *reinterpret_cast<const uint32_t*>(src);
        } else {
          for (int k = 0; k < 4; ++k)
            if (c0 + k < scols) w |= static_cast<uint32_t>(src[k]) << (8 * k);
        }
      }
      word[q] = w;
    }
    reinterpret_cast<uint4*>(out)[l] = make_uint4(word[0], word[1], word[2], word[3]);
  }
}

// y = bf16(fp32(fp32(D * S_x[row]) * S_w)), D row-major FP32 [m][n] (n a multiple of 16).
// A block per row at a time; each thread keeps kEpiUnroll independent 16-byte loads in flight.
constexpr int kEpiThreads = 128;
constexpr int kEpiUnroll = 4;

__device__ __forceinline__ uint2 scale_to_bf16x4(const float4 v, float s, float w) {
  const float a = __fmul_rn(__fmul_rn(v.x, s), w), b = __fmul_rn(__fmul_rn(v.y, s), w);
  const float c = __fmul_rn(__fmul_rn(v.z, s), w), e = __fmul_rn(__fmul_rn(v.w, s), w);
  uint32_t lo, hi;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(hi) : "f"(e), "f"(c));
  return make_uint2(lo, hi);
}

__global__ void __launch_bounds__(kEpiThreads) scale_epilogue_kernel(
    const float* __restrict__ d, const float* __restrict__ sx, const float* __restrict__ sw,
    int64_t m, int64_t n, uint16_t* __restrict__ y) {
  nvfp4::pdl_wait();  // D is the previous kernel's output
  const float w = sw[0];
  const int n4 = static_cast<int>(n / 4);
  for (int64_t row = blockIdx.x; row < m; row += gridDim.x) {
    const float s = sx[row];
    const float4* dr = reinterpret_cast<const float4*>(d + row * n);
    uint2* yr = reinterpret_cast<uint2*>(y + row * n);
    int c = threadIdx.x;
    for (; c + (kEpiUnroll - 1) * kEpiThreads < n4; c += kEpiUnroll * kEpiThreads) {
      float4 v[kEpiUnroll];
#pragma unroll
      for (int u = 0; u < kEpiUnroll; ++u) v[u] = __ldcs(dr + c + u * kEpiThreads);
#pragma unroll
      for (int u = 0; u < kEpiUnroll; ++u) yr[c + u * kEpiThreads] = scale_to_bf16x4(v[u], s, w);
    }
    for (; c < n4; c += kEpiThreads) yr[c] = scale_to_bf16x4(__ldcs(dr + c), s, w);
  }
}

std::atomic<cublasLtHandle_t> g_lt[64];

cublasLtHandle_t lt_handle(int device) {
  if (device < 0 || device >= 64) return nullptr;
  cublasLtHandle_t h = g_lt[device].load();
  if (h != nullptr) return h;
  cublasLtHandle_t created = nullptr;
  if (cublasLtCreate(&created) != CUBLAS_STATUS_SUCCESS) return nullptr;
  cublasLtHandle_t expected = nullptr;
  if (!g_lt[device].compare_exchange_strong(expected, created)) {
    cublasLtDestroy(created);
    return expected;
  }
  return created;
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

}  // namespace

extern "C" size_t nvfp4_swizzled_scales_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0) return 0;
  return static_cast<size_t>(round_up(rows, 128) * round_up(cols / 16, 4));
}

extern "C" nvfp4_status nvfp4_swizzle_block_scales(const uint8_t* block_scales, int64_t rows,
                                                   int64_t cols, uint8_t* swizzled,
                                                   nvfp4_stream_t stream) {
  if (rows < 0) return NVFP4_ERR_INVALID_ARG;
  if (cols <= 0 || cols % 16 != 0) return NVFP4_ERR_SHAPE;
  if (rows == 0) return NVFP4_OK;
  if (block_scales == nullptr || swizzled == nullptr) return NVFP4_ERR_INVALID_ARG;
  const int64_t scols = cols / 16;
  const int64_t total = round_up(rows, 128) * round_up(scols, 4);
  const uintptr_t a = reinterpret_cast<uintptr_t>(block_scales), b = reinterpret_cast<uintptr_t>(swizzled);
  if (a < b + total && b < a + static_cast<uintptr_t>(rows * scols)) return NVFP4_ERR_INVALID_ARG;
  if ((b & 15) != 0) return NVFP4_ERR_ALIGNMENT;  // written in 16-byte lines
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return NVFP4_ERR_CUDA;
  const int64_t lines = total / 16;
  int64_t grid = (lines + 255) / 256;
  const int64_t cap = static_cast<int64_t>(nvfp4::sm_count(device)) * 8;
  if (grid > cap) grid = cap;
  swizzle_scales_kernel<<<static_cast<unsigned>(grid), 256, 0,
                          reinterpret_cast<cudaStream_t>(stream)>>>(block_scales, rows, scols,
                                                                    swizzled, lines,
                                                                    round_up(scols, 4) / 4);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

extern "C" size_t nvfp4_gemm_workspace_bytes(int64_t m, int64_t n) {
  if (m < 0 || n < 0) return 0;
  return kLtWorkspace + static_cast<size_t>(round_up(m * n * 4, 256));
}

extern "C" nvfp4_status nvfp4_gemm_nt(const uint8_t* x_codes, const uint8_t* x_scales_swizzled,
                                      const float* x_row_scale, const uint8_t* w_codes,
                                      const uint8_t* w_scales_swizzled, const float* w_tensor_scale,
                                      int64_t m, int64_t n, int64_t k, void* y, void* workspace,
                                      size_t workspace_bytes, nvfp4_stream_t stream) {
  if (m < 0 || n < 0 || k < 0) return NVFP4_ERR_INVALID_ARG;
  if (k == 0 || k % 64 != 0 || n % 16 != 0) return NVFP4_ERR_SHAPE;
  if (m == 0 || n == 0) return NVFP4_OK;
  if (!x_codes || !x_scales_swizzled || !x_row_scale || !w_codes || !w_scales_swizzled ||
      !w_tensor_scale || !y)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(x_codes, 256) || !aligned(w_codes, 256) || !aligned(x_scales_swizzled, 256) ||
      !aligned(w_scales_swizzled, 256) || !aligned(y, 16))
    return NVFP4_ERR_ALIGNMENT;
  if (workspace == nullptr || workspace_bytes < nvfp4_gemm_workspace_bytes(m, n) ||
      !aligned(workspace, 256))
    return NVFP4_ERR_WORKSPACE;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return NVFP4_ERR_CUDA;
  cublasLtHandle_t lt = lt_handle(device);
  if (lt == nullptr) return NVFP4_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* d = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + kLtWorkspace);

  // Column-major view: D[n][m] (col-major, ld n) = W[n][k] . X[m][k]^T, i.e. row-major y[m][n].
  // A = W (stored k x n col-major, transposed), B = X (stored k x m col-major).
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  nvfp4_status result = NVFP4_ERR_CUDA;
  const cublasOperation_t ta = CUBLAS_OP_T, tb = CUBLAS_OP_N;
  const cublasLtMatmulMatrixScale_t vec16 = CUBLASLT_MATMUL_MATRIX_SCALE_VEC16_UE4M3;
  const void* a_scale = w_scales_swizzled;
  const void* b_scale = x_scales_swizzled;
  const float alpha = 1.0f, beta = 0.0f;
  const size_t lt_ws = kLtWorkspace;
  cublasLtMatmulHeuristicResult_t heur;
  int found = 0;
  if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS)
    goto done;
  if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof ta) ||
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof tb) ||
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_MODE, &vec16, sizeof vec16) ||
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_MODE, &vec16, sizeof vec16) ||
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_A_SCALE_POINTER, &a_scale,
                                     sizeof a_scale) ||
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_B_SCALE_POINTER, &b_scale,
                                     sizeof b_scale))
    goto done;
  if (cublasLtMatrixLayoutCreate(&la, CUDA_R_4F_E2M1, k, n, k) ||
      cublasLtMatrixLayoutCreate(&lb, CUDA_R_4F_E2M1, k, m, k) ||
      cublasLtMatrixLayoutCreate(&lc, CUDA_R_32F, n, m, n))
    goto done;
  if (cublasLtMatmulPreferenceCreate(&pref) ||
      cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &lt_ws,
                                           sizeof lt_ws))
    goto done;
  if (cublasLtMatmulAlgoGetHeuristic(lt, op, la, lb, lc, lc, pref, 1, &heur, &found) ||
      found == 0) {
    result = NVFP4_ERR_SHAPE;  // no tensor-core algorithm for this problem
    goto done;
  }
  if (cublasLtMatmul(lt, op, &alpha, w_codes, la, x_codes, lb, &beta, d, lc, d, lc, &heur.algo,
                     workspace, lt_ws, s) != CUBLAS_STATUS_SUCCESS)
    goto done;
  {
    int64_t grid = m;
    const int64_t cap = static_cast<int64_t>(nvfp4::sm_count(device)) * 16;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    if (nvfp4::launch_programmatic(scale_epilogue_kernel, dim3(static_cast<unsigned>(grid)),
                                   dim3(kEpiThreads), 0, s, static_cast<const float*>(d),
                                   x_row_scale, w_tensor_scale, m, n,
                                   static_cast<uint16_t*>(y)) == cudaSuccess)
      result = NVFP4_OK;
  }
done:
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (lc) cublasLtMatrixLayoutDestroy(lc);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  return result;
}
