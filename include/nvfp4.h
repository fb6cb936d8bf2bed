/*
 * nvfp4.h -- C ABI of the GB300 NVFP4 quantization library (libnvfp4_gb300.so).
 *
 * What it computes (web pages, cited by title and section):
 *   "NVFP4 RL" blog post (jianyuh.github.io/nvfp4/2026/07/11/NVFP4-RL):
 *     Sec. 2 "Baseline: Per-Token Scales & Targeted MoE Quantization" -- every token (row) gets its
 *       own FP32 scale from its amax over the hidden dimension; FP8 E4M3 block scales; both fused
 *       into the activation quantization kernel.
 *     Sec. 3 "Gradient Stability: The Chain-Rule Inconsistency" -- the dequantized backward uses
 *       DQ(Q(w)), the BF16 value of exactly what the quantizer encoded.
 *     Sec. 4 "The Four-Over-Six (4/6) Optimization" -- each block maps its max to +-6 or to +-4,
 *       whichever gives the lower block error; weights use the same scheme.
 *   "humans& Open-Sources the First Stable 4-Bit RL Training Recipe at 1.73x Speedup",
 *     "Three instabilities, three fixes" -- per-token activation scaling, dequantized backward,
 *     4/6 for weights and activations, bit-exact across training and inference.
 *   "TRACE FP4 RL -- Rollout-guided FP4 rounding", Jargon -- the E2M1 grid
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6} and round-to-nearest.
 *
 * The exact arithmetic (every FP32 rounding, the 4/6 error order, tie rules) is fixed in the
 * design notes; results are bit-identical to the CPU oracle that states it.
 *
 * Data layout (all row-major, all caller-owned DEVICE memory unless stated otherwise):
 *   x, y          BF16 [rows][cols], cols a multiple of 16, 16-byte aligned base.
 *   codes         uint8 [rows][cols/2]: E2M1 codes, element 2j in the low nibble of byte j,
 *                 16-byte aligned base.
 *   block_scales  uint8 [rows][cols/16]: one FP8 E4M3 byte per 16-element block.
 *   row scale     float [rows]: S_dec = amax_row / (6 * M) per row.
 *   tensor scale  float [1]:    S_dec = amax_tensor / (6 * M).
 *   M = 256 in modes FOUR_OVER_SIX and FOUR_OVER_SIX_FP16, 448 in mode SIX.
 *
 * Contract common to every call:
 *   - Asynchronous on `stream` (NULL = the legacy default stream); nothing synchronizes.
 *   - Arguments are validated on the host before anything is launched; a rejected call launches
 *     nothing and touches no memory.  rows == 0 is a valid no-op.
 *   - The library allocates no memory.  Inputs must not overlap outputs.
 *   - Errors detected on the device (invalid group offsets, a bounded wait that ran out) are
 *     recorded in a per-device status word read by nvfp4_get_device_status(); the first error
 *     recorded wins.
 *   - Non-finite inputs are outside the contract: they do not fault, their outputs are unspecified.
 *   - Results do not depend on the launch configuration, the stream or the rest of the batch.
 *   - Kernels are launched as programmatic dependents of the previous kernel on `stream` (they
 *     set up shared memory while it finishes, and wait for it before touching global memory) and
 *     let the next kernel start early.  A kernel the caller launches after a call with
 *     programmatic stream serialization must wait for its prerequisite grid
 *     (griddepcontrol.wait / cudaGridDependencySynchronize) before reading the call's outputs,
 *     as for any programmatic dependent; ordinary launches need nothing.
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st* nvfp4_stream_t;

typedef enum {
  NVFP4_MODE_SIX = 0,           /* block max always mapped to +-6 (ordinary NVFP4)           */
  NVFP4_MODE_FOUR_OVER_SIX = 1, /* block max mapped to +-6 or +-4, lower block error wins    */
  /* As FOUR_OVER_SIX, but the two block errors are taken from FP16 values (the fast path of
   * "NVFP4 RL" Sec. 4, "The optimization": the candidate q*s is exact in FP16 and the target is
   * scaled down by the inverse of the per-token scale instead): the target x * S_enc is cast to
   * FP16, each residual is one FP16 rounding of (target - q*s), and the squares are summed in
   * FP32 in element order.  Same candidates and codes as FOUR_OVER_SIX; only near-tie choices
   * differ (0.08-0.11% of the blocks of the synthetic workloads). */
  NVFP4_MODE_FOUR_OVER_SIX_FP16 = 2
} nvfp4_mode;

typedef enum {
  NVFP4_SCALE_ROW = 0,    /* one FP32 scale per row (token)    */
  NVFP4_SCALE_TENSOR = 1  /* one FP32 scale for the tensor     */
} nvfp4_scale_kind;

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,  /* null pointer, bad enum, negative count, overlapping buffers   */
  NVFP4_ERR_SHAPE = 2,        /* cols not a positive multiple of 16, or too large               */
  NVFP4_ERR_ALIGNMENT = 3,    /* a pointer below its required alignment                         */
  NVFP4_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed                    */
  NVFP4_ERR_TIMEOUT = 5,      /* device side: a bounded wait on a shared-memory barrier ran out */
  NVFP4_ERR_OFFSETS = 6,      /* device side: group offsets not 0 = o[0] <= ... <= o[G] = rows  */
  NVFP4_ERR_WORKSPACE = 7     /* workspace missing or smaller than nvfp4_tensor_workspace_bytes */
} nvfp4_status;

/* Per-token quantization ("NVFP4 RL" Sec. 2 and Sec. 4).
 *   x             BF16 [rows][cols] on the device.
 *   group_offsets optional device int32 [num_groups + 1] describing expert groups of rows
 *                 (MoE grouped layout).  Quantization never depends on the grouping; the offsets
 *                 are validated on the device (0 = o[0] <= o[1] <= ... <= o[num_groups] = rows)
 *                 and a violation records NVFP4_ERR_OFFSETS.  NULL (with num_groups == 0) skips it.
 *   mode          NVFP4_MODE_SIX or NVFP4_MODE_FOUR_OVER_SIX.
 *   codes, block_scales, row_scale   outputs as laid out above.
 * Supported cols: 16 <= cols <= 65536, cols % 16 == 0 (rows wider than 32768 are staged by all
 * 16 warps of a CTA in one shared-memory slot each, without copy/compute overlap: slower). */
nvfp4_status nvfp4_quantize_rowwise(const void* x, int64_t rows, int64_t cols,
                                    const int32_t* group_offsets, int32_t num_groups,
                                    nvfp4_mode mode, uint8_t* codes, uint8_t* block_scales,
                                    float* row_scale, nvfp4_stream_t stream);

/* Residual quantization in the manner of Rollout-ResQ ("HiFloat4 Format for End-To-End
 * Reinforcement Learning Post-Training of Large Language Models", Rollout-ResQ section: the
 * projection is computed as Q(X)Q(W) + Q(dX)Q(W) with dX = X - Q(X)), here with NVFP4 per-token
 * 4/6 quantization for both terms:
 *   (codes, block_scales, row_scale)             = Q(x), exactly as nvfp4_quantize_rowwise;
 *   dX = bf16(fp32(x) - fp32(DQ(Q(x))))          (the difference is exact in FP32; one BF16 rounding);
 *   (res_codes, res_block_scales, res_row_scale) = Q(dX) with dX's own per-token scale.
 * One pass over x.  The 2:4 sparsification of the residual on that page is not applied.  Buffers,
 * layouts and errors as nvfp4_quantize_rowwise; the two output sets must not overlap. */
nvfp4_status nvfp4_quantize_residual(const void* x, int64_t rows, int64_t cols, nvfp4_mode mode,
                                     uint8_t* codes, uint8_t* block_scales, float* row_scale,
                                     uint8_t* res_codes, uint8_t* res_block_scales,
                                     float* res_row_scale, nvfp4_stream_t stream);

/* Per-token amax: row_amax[r] = max_k |x[r][k]| (device float [rows]).  What a rollout records
 * so that a later nvfp4_quantize_guided reproduces its scales. */
nvfp4_status nvfp4_row_amax(const void* x, int64_t rows, int64_t cols, float* row_amax,
                            nvfp4_stream_t stream);

/* Rollout-guided rounding ("TRACE FP4 RL -- Rollout-guided FP4 rounding": between the two
 * neighbouring codewords of its own value the training engine picks the one closer to the
 * codeword the rollout recorded, under the rollout-side scale).  Inputs: the trainer's x, the
 * rollout's per-token amax (row_amax, device float [rows]), its codes and its E4M3 block scales
 * (layouts as nvfp4_quantize_rowwise).  Each element's scaled value t is formed as the quantizer
 * forms it from that amax and block scale; the output code is whichever of t's two neighbouring
 * E2M1 codewords (one if t is on the grid or beyond +-6) is closer to the rollout's codeword, with
 * the sign of t kept on zero.  The block scales and row scales stay the rollout's.  When x equals
 * the rollout's input the output equals the rollout's codes.  codes: device uint8 [rows][cols/2].
 * Any cols that is a positive multiple of 16. */
nvfp4_status nvfp4_quantize_guided(const void* x, int64_t rows, int64_t cols, nvfp4_mode mode,
                                   const float* row_amax, const uint8_t* ref_codes,
                                   const uint8_t* ref_block_scales, uint8_t* codes,
                                   nvfp4_stream_t stream);

/* Bytes of device workspace the per-tensor calls need (a few KB; it holds partial maxima). */
size_t nvfp4_tensor_workspace_bytes(void);

/* Per-tensor quantization for weights ("NVFP4 RL" Sec. 4: 4/6 applied to weights as well):
 * one amax over the whole tensor, then the same block/4-over-6 encoding as the row path.
 *   tensor_scale  device float [1], receives S_dec.
 *   workspace     device scratch of at least nvfp4_tensor_workspace_bytes() bytes, 16-byte
 *                 aligned; its contents on entry are ignored.  Two launches. */
nvfp4_status nvfp4_quantize_tensor(const void* x, int64_t rows, int64_t cols, nvfp4_mode mode,
                                   uint8_t* codes, uint8_t* block_scales, float* tensor_scale,
                                   void* workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* amax = max |x_i| over n BF16 elements (n >= 0; 0 for n == 0), written to the device float
 * *amax.  Used by sharded weights: each shard's amax, a max over ranks, then
 * nvfp4_quantize_tensor_with_amax. */
nvfp4_status nvfp4_tensor_amax(const void* x, int64_t n, float* amax, void* workspace,
                               size_t workspace_bytes, nvfp4_stream_t stream);

/* Per-tensor quantization with the amax supplied by the caller (device float [1]), e.g. the
 * max over shards.  Bit-identical to nvfp4_quantize_tensor when *amax is the tensor's amax. */
nvfp4_status nvfp4_quantize_tensor_with_amax(const void* x, int64_t rows, int64_t cols,
                                             nvfp4_mode mode, const float* amax, uint8_t* codes,
                                             uint8_t* block_scales, float* tensor_scale,
                                             nvfp4_stream_t stream);

/* Per-tensor quantization for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call; it exists for code that must not (or cannot) call cudaMalloc: an
 * allocator or memory-pool callback, a framework plugin that is handed only its input and output
 * tensors, or a path where an allocation's implicit synchronization is unacceptable.
 * Same arguments, outputs and results (bit for bit) as nvfp4_quantize_tensor, minus the
 * workspace: the partial maxima of the amax pass go to a fixed 2 KB array of device memory
 * inside the library, held on every GPU that loads the library until the process exits.
 *   - The first call on each device looks up that array's device address (cudaGetSymbolAddress,
 *     with the device current) and caches it; make that first call before any stream capture.
 *   - The array holds at most 512 partial maxima.  The amax pass needs 2 per SM (capped at 1024),
 *     i.e. 304 on a 152-SM GB300; a device that would need more is refused with
 *     NVFP4_ERR_WORKSPACE before anything is launched.  Any tensor size is accepted.
 *   - Every call shares the one array and it keeps the last call's contents; nothing in it has to
 *     start at zero.  Calls whose kernels overlap on the GPU (different streams with no ordering
 *     between them) race on the array: order them on one stream. */
nvfp4_status nvfp4_quantize_tensor_noalloc(const void* x, int64_t rows, int64_t cols,
                                           nvfp4_mode mode, uint8_t* codes,
                                           uint8_t* block_scales, float* tensor_scale,
                                           nvfp4_stream_t stream);

/* Dequantization for the dequantized backward ("NVFP4 RL" Sec. 3):
 * y = bf16_rne(fp32(fp32(q * s) * S_dec)) for every element -- exactly the value the quantizer
 * encoded, rounded once to FP32 and once to BF16.
 *   scale  device float [rows] for NVFP4_SCALE_ROW, [1] for NVFP4_SCALE_TENSOR.
 *   y      BF16 [rows][cols] output. */
nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* block_scales,
                              const float* scale, nvfp4_scale_kind kind, int64_t rows,
                              int64_t cols, void* y, nvfp4_stream_t stream);

/* Quantize and dequantize in one pass over x: emits codes, block scales, the scale(s) and the
 * BF16 round trip y = DQ(Q(x)) ("NVFP4 RL" Sec. 2-4).  Outputs are bit-identical to the
 * separate quantize and dequantize calls.  workspace is needed for NVFP4_SCALE_TENSOR only
 * (NULL / 0 allowed for NVFP4_SCALE_ROW). */
nvfp4_status nvfp4_fused_roundtrip(const void* x, int64_t rows, int64_t cols,
                                   nvfp4_scale_kind kind, nvfp4_mode mode, uint8_t* codes,
                                   uint8_t* block_scales, float* scale, void* y, void* workspace,
                                   size_t workspace_bytes, nvfp4_stream_t stream);

/* Bytes of device staging workspace nvfp4_fused_roundtrip_host needs for rows of `cols`
 * elements (three chunk buffers of ~32 MB of input each); 0 for an invalid cols. */
size_t nvfp4_roundtrip_host_workspace_bytes(int64_t cols);

/* nvfp4_fused_roundtrip with the row scale for a matrix in HOST memory ("NVFP4 RL" Sec. 6: the
 * same pipeline quantizes checkpoints online, from and to host memory).  x, codes, block_scales,
 * row_scale and y are host pointers (page-locked memory lets the copies overlap; pageable memory
 * works but serializes them); the layouts are those of the device calls.  Rows are streamed
 * through `workspace` (device memory of at least nvfp4_roundtrip_host_workspace_bytes(cols)
 * bytes, 256-byte aligned) in chunks on three internal streams, so host->device copies, kernels and
 * device->host copies overlap.  Ordered after the work already queued on `stream`; `stream` is
 * made to wait for all of it, so synchronize `stream` before reading the outputs.  Results are
 * bit-identical to nvfp4_fused_roundtrip. */
nvfp4_status nvfp4_fused_roundtrip_host(const void* x, int64_t rows, int64_t cols,
                                        nvfp4_mode mode, uint8_t* codes, uint8_t* block_scales,
                                        float* row_scale, void* y, void* workspace,
                                        size_t workspace_bytes, nvfp4_stream_t stream);

/* Bytes of the MMA-ready layout of the block scales of a [rows][cols] matrix: rows padded to 128
 * and scale columns (cols/16) padded to 4. */
size_t nvfp4_swizzled_scales_bytes(int64_t rows, int64_t cols);

/* Re-lays row-major E4M3 block scales [rows][cols/16] into the layout block-scaled tensor-core
 * GEMMs read: tiles of 128 rows x 4 scale columns (512 bytes), tiles row-major over
 * [ceil(rows/128)][ceil(cols/64)], the scale of (row r, scale column c) at byte
 * (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4) of its tile; padding is zero.
 * swizzled: 16-byte aligned device buffer of nvfp4_swizzled_scales_bytes(rows, cols) bytes
 * (NVFP4_ERR_ALIGNMENT otherwise). */
nvfp4_status nvfp4_swizzle_block_scales(const uint8_t* block_scales, int64_t rows, int64_t cols,
                                        uint8_t* swizzled, nvfp4_stream_t stream);

/* Scratch bytes nvfp4_gemm_nt needs: 0 (kept so callers that size a workspace keep working). */
size_t nvfp4_gemm_workspace_bytes(int64_t m, int64_t n);

/* The forward the quantized tensors feed ("NVFP4 RL" Sec. 3: y = x . Q(w); Sec. 2: x with per-token
 * FP32 scales): y[m][n] = bf16(fp32(fp32(D[m][n] * x_row_scale[m]) * w_tensor_scale[0])) with
 * D[m][n] = sum_k (qx[m][k] * sx[m][k/16]) * (qw[n][k] * sw[n][k/16]) accumulated in FP32 on the
 * tensor cores: one hand-written kernel (block-scaled FP4 tcgen05 products, the scales applied in
 * its epilogue; no library GEMM and no FP32 intermediate in memory).
 *   x_codes [m][k/2], w_codes [n][k/2]   E2M1 codes as the quantizer writes them (256-byte aligned)
 *   x_scales_swizzled, w_scales_swizzled block scales in the layout of nvfp4_swizzle_block_scales
 *                                        (256-byte aligned)
 *   x_row_scale [m], w_tensor_scale [1]  the quantizer's S_dec values
 *   y [m][n] BF16 (16-byte aligned).  workspace / workspace_bytes are unused (may be NULL / 0).
 * k must be a positive multiple of 64 and n of 16; m, n, k below 2^31 - 256.  Not bit-reproducible
 * against other GEMMs: the FP32 accumulation order is the tensor core's.  A bounded wait inside
 * the kernel that runs out records NVFP4_ERR_TIMEOUT in the device status word. */
nvfp4_status nvfp4_gemm_nt(const uint8_t* x_codes, const uint8_t* x_scales_swizzled,
                           const float* x_row_scale, const uint8_t* w_codes,
                           const uint8_t* w_scales_swizzled, const float* w_tensor_scale, int64_t m,
                           int64_t n, int64_t k, void* y, void* workspace, size_t workspace_bytes,
                           nvfp4_stream_t stream);

/* Reads (and, if clear != 0, resets to NVFP4_OK) the device status word of the current device.
 * Synchronizes the device.  *status_out receives NVFP4_OK or the first device-side error.
 * The library looks up the device addresses of its own device variables (this status word, the
 * allocation-free call's array) once per device and keeps them for the life of the process, so
 * it must not be used on a device after cudaDeviceReset or a teardown of its primary context. */
nvfp4_status nvfp4_get_device_status(int clear, nvfp4_status* status_out);

/* Static, NUL-terminated description of a status code. */
const char* nvfp4_status_string(nvfp4_status status);

/* Launch-shape override for tuning and for the launch-independence tests: warps per CTA, ring
 * stages per warp, and a cap on the grid size; 0 keeps the automatic choice.  Process-wide; the
 * results never depend on it.  Returns NVFP4_ERR_INVALID_ARG for negative or too-large values. */
nvfp4_status nvfp4_set_launch_config(int warps_per_cta, int stages, int max_ctas);

/* Self-test of the device-side failure path: launches one warp that waits on a shared-memory
 * barrier nothing arrives on, giving up after `timeout_ns` nanoseconds (1 ms default if 0) and
 * recording NVFP4_ERR_TIMEOUT in the device status word.  The wait always ends. */
nvfp4_status nvfp4_selftest_wait_timeout(uint64_t timeout_ns, nvfp4_stream_t stream);

/* Self-test of the quantize kernels' own failure path.  Until it is called again with row = -1,
 * every quantize call (row or tensor scale, plain, fused or residual) and every guided call whose
 * rows are staged through shared memory (cols a multiple of 1024) withholds the shared-memory
 * copies of row `row` of its input: the warps that own that row wait on their ring barrier in vain, give up after timeout_ns nanoseconds, record NVFP4_ERR_TIMEOUT in the device
 * status word, wait (within the library's usual 4 s bound) for their other copies still in
 * flight, and return, leaving their remaining rows unwritten; warps sharing a row leave together.
 * Every other wait keeps working, so every launch ends.  timeout_ns must be in (0, 4e9] when
 * row >= 0; row = -1 restores normal operation (timeout_ns ignored).  Process-wide, for tests
 * only: do not call it while other threads issue quantize calls. */
nvfp4_status nvfp4_selftest_withhold_row(int64_t row, uint64_t timeout_ns);

/* ABI version of this header (incremented on incompatible changes). */
int nvfp4_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
