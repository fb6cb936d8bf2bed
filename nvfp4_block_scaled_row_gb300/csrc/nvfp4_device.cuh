// nvfp4_device.cuh -- device-side building blocks for the sm_103a NVFP4 kernels: shared-memory
// barriers and bulk (TMA) copies, the hardware FP32 <-> E2M1 / E4M3 / BF16 conversions, packed
// FP32x2 arithmetic, and the launch-parameter structs shared by the kernel translation units.
//
// Every floating-point operation on the quantizer's data path is written as one explicit
// round-to-nearest instruction (inline PTX or __f*_rn intrinsics), and the library is compiled
// with --fmad=false, so no multiply-add is ever contracted behind the spec's back.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace nvfp4 {

constexpr int kBlockElems = 16;          // elements per E4M3-scaled block
constexpr int kMaxCols = 65536;          // widest row the shared-memory ring supports
constexpr int kMaxWarpsPerCta = 16;
constexpr int kMaxStages = 4;
constexpr int kMaxTeam = 16;             // warps that share one row (16: the whole CTA)
constexpr int kMaxBlocksPerLane = 8;     // 16-element blocks one lane owns per row (<= 8 KB slots)
constexpr int kAmaxMaxPartials = 1024;   // per-tensor amax: partial maxima in the workspace

// Shared-memory header of the quantize kernel, then the ring (128-byte aligned).
constexpr int kTableBytes = 256 * 8;                          // one ScaleEntry per E4M3 byte
constexpr int kXchBytes = 4 * kMaxWarpsPerCta * 4;            // row-amax partials: 2 parities x 2 tensors
constexpr int kAbortBytes = kMaxWarpsPerCta * 4;              // per-team abort flags
constexpr int kWorkQueue = 8;                                 // work requests in flight or unread
constexpr int kWorkQueueBytes = kWorkQueue * 16 + 2 * kWorkQueue * 8;  // answers, full/free barriers
constexpr int kFixedHeaderBytes = kTableBytes + kXchBytes + kAbortBytes + kWorkQueueBytes;

// Header bytes for `warps` warps with `stages` ring slots each (one copy barrier per slot).
__host__ __device__ constexpr int ring_header_bytes(int warps, int stages) {
  return ((kFixedHeaderBytes + warps * stages * 8 + 127) / 128) * 128;
}

// Device status codes (same numbers as nvfp4_status in include/nvfp4.h).
constexpr int kStatusTimeout = 5;
constexpr int kStatusOffsets = 6;

// Mode numbers (same as nvfp4_mode).
constexpr int kModeSix = 0;
constexpr int kModeFourOverSix = 1;
constexpr int kModeFourOverSixFp16 = 2;  // 4/6 with the block errors compared in FP16 arithmetic

// Per E4M3 byte: the correctly rounded reciprocal of its value s (0 for s == 0) and -s as an
// FP16 pair (E4M3 values are exact in FP16).
struct __align__(8) ScaleEntry {
  float inv;
  uint32_t neg_s_h2;
};

struct QuantParams {
  const uint16_t* x;        // BF16 bits [rows][cols]
  int64_t rows;
  int32_t cols;
  uint8_t* codes;           // [rows][cols/2]
  uint8_t* scales;          // [rows][cols/16]
  float* scale_out;         // S_dec: [rows] (row scale) or [1] (tensor scale)
  uint16_t* y;              // BF16 bits [rows][cols], fused round trip only
  uint8_t* res_codes;       // residual quantization outputs (residual kernels only)
  uint8_t* res_scales;
  float* res_scale_out;
  const float* amax_src;    // tensor scale: n_amax partial maxima (or one amax)
  int32_t n_amax;
  const int32_t* offsets;   // optional group offsets [num_groups + 1]
  int32_t num_groups;
  int32_t stages;           // ring slots per warp
  int32_t team;             // warps sharing one row
  int32_t blocks_per_warp;  // 16-element blocks each warp of a team owns
  uint32_t slot_bytes;      // bytes per ring slot (>= 32 * blocks_per_warp, multiple of 128)
  int32_t prologue_before_wait;  // 1: the first row copies may precede griddepcontrol.wait
  int* status;              // device status word
  uint64_t timeout_ns;      // bound on every ring-slot wait
  uint64_t drain_timeout_ns;  // bound on each wait for a copy still in flight before an early exit
  int64_t withhold_row;     // self-test only: the row whose copies are never issued (-1: none)
};

struct GuidedParams {
  const uint16_t* x;          // BF16 bits [rows][cols] (the trainer's values)
  int64_t rows;
  int32_t cols;
  const float* row_amax;      // the rollout's per-token amax [rows]
  const uint8_t* ref_codes;   // the rollout's codes [rows][cols/2]
  const uint8_t* ref_scales;  // the rollout's E4M3 block scales [rows][cols/16]
  uint8_t* codes;             // output codes [rows][cols/2]
  int* status;                // device status word
  uint64_t timeout_ns;        // bound on every ring-slot wait (ring variant)
  uint64_t drain_timeout_ns;  // bound on each wait for a copy still in flight before an early exit
  int64_t withhold_row;       // self-test only: the row whose copies are never issued (-1: none)
};

struct DequantParams {
  const uint8_t* codes;
  const uint8_t* scales;
  const float* scale;       // [rows] or [1]
  int64_t rows;
  int32_t cols;
  uint16_t* y;
};

// ------------------------------------------------------------------------------------------------
// Status word
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);  // first error wins
}

// ------------------------------------------------------------------------------------------------
// Shared-memory barriers and bulk copies (cp.async.bulk, the non-tensor TMA path)
// ------------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy (the bulk-copy engine).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the barrier phase with the given parity; gives up after timeout_ns nanoseconds.
// Returns false when it gave up.  Every wait in this library goes through here.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - start > timeout_ns) return false;
  }
}

// One arrival (count 1) on a shared-memory barrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Cluster launch control: asks the hardware to cancel one CTA of this grid that has not started
// yet; the 16-byte answer lands in `answer` and completes `bar` (16 transaction bytes, which the
// caller announces with mbar_arrive_expect_tx first).  One thread issues it.
__device__ __forceinline__ void launch_control_request(void* answer, uint64_t* bar) {
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128"
      " [%0], [%1];" ::"r"(smem_addr(answer)),
      "r"(smem_addr(bar))
      : "memory");
}

// Decodes an answer: returns true and the cancelled CTA's x index when the request succeeded
// (the index is only read from a successful answer).
__device__ __forceinline__ bool launch_control_answer(const void* answer, uint32_t& ctaid_x) {
  uint32_t ok, x;
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b128 h;\n\t"
      "ld.shared.b128 h, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, h;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t"
      "mov.u32 %1, 0;\n\t"
      "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, h;\n\t}"
      : "=r"(ok), "=r"(x)
      : "r"(smem_addr(answer))
      : "memory");
  ctaid_x = x;
  return ok != 0;
}

// Bulk prefetch of [gsrc, gsrc + bytes) into L2 (a hint: no data moves to this SM).
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  return policy;
}

// Bulk copy global -> shared, completing on `bar` (bytes: multiple of 16, both ends 16-aligned).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------------------------------------------------
// Packed FP32 pairs (.x in the low 32 bits)
// ------------------------------------------------------------------------------------------------

typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack2(f32x2 v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Two BF16 values (element 2j in the low half) widened exactly to an FP32 pair.
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w) {
  return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Two BF16 values widened to an FP32 pair on the FMA pipe: x * 1 + (-0) with BF16 operands and
// an FP32 result is exact and keeps the sign of zero (same result as bf16x2_to_f32x2).
__device__ __forceinline__ f32x2 bf16x2_to_f32x2_fma(uint32_t w, uint16_t one_bf16, float neg_zero) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "fma.rn.f32.bf16 %0, l, %3, %4;\n\t"
      "fma.rn.f32.bf16 %1, h, %3, %4;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w), "h"(one_bf16), "f"(neg_zero));
  return pack2(lo, hi);
}

// ------------------------------------------------------------------------------------------------
// Format conversions (hardware, round-to-nearest-even, saturating where named)
// ------------------------------------------------------------------------------------------------

// max(|a|, |b|) per BF16 half, sign bits = XOR of the inputs' (callers mask them off).
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Largest |value| of a BF16 pair word as FP32 (exact).
__device__ __forceinline__ float abs_max_of_pair(uint32_t m2) {
  const uint32_t h = m2 & 0x7FFF7FFFu;
  const uint32_t top = max(h >> 16, h & 0xFFFFu);
  return __uint_as_float(top << 16);
}

// E4M3 (RNE, satfinite) of two FP32 values: `hi` lands in bits 15..8, `lo` in bits 7..0.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float hi, float lo) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two E4M3 bytes (bits 15..8 and 7..0) to an FP16 pair (high half, low half); exact.
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t two_bytes) {
  uint32_t d;
  const uint16_t b = static_cast<uint16_t>(two_bytes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(b));
  return d;
}

// Eight FP32 targets (as four pairs, element 2j in .x) to eight E2M1 codes packed in a word,
// element i in nibble i (RNE, satfinite, sign kept).
__device__ __forceinline__ uint32_t e2m1x8_from_f32x2(f32x2 p0, f32x2 p1, f32x2 p2, f32x2 p3) {
  float a0, a1, b0, b1, c0, c1, d0, d1;
  unpack2(p0, a0, a1);
  unpack2(p1, b0, b1);
  unpack2(p2, c0, c1);
  unpack2(p3, d0, d1);
  uint32_t w;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(w)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1), "f"(d0), "f"(d1));
  return w;
}

// Eight FP32 targets (four pairs, element 2j in .x) rounded to E2M1 (RNE, satfinite, sign kept)
// and decoded back, in one step: returns the packed code word (element i in nibble i) and the
// four decoded FP16 pairs (element 2j in the low half).  The code bytes stay in registers between
// the two conversions.
__device__ __forceinline__ uint32_t e2m1x8_encode_decode(f32x2 p0, f32x2 p1, f32x2 p2, f32x2 p3,
                                                        uint32_t (&h)[4]) {
  float a0, a1, b0, b1, c0, c1, d0, d1;
  unpack2(p0, a0, a1);
  unpack2(p1, b0, b1);
  unpack2(p2, c0, c1);
  unpack2(p3, d0, d1);
  uint32_t w;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %8, %7;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %10, %9;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %12, %11;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, q0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, q1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, q2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %4, q3;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
      : "=r"(w), "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1), "f"(d0), "f"(d1));
  return w;
}

// Eight E2M1 codes (nibble i = element i) to four FP16 pairs (element 2j in the low half).
__device__ __forceinline__ void f16x2_from_e2m1x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Per half: a.h * b.h + c (FP16 operands widened exactly, one FP32 rounding) -> FP32 pair.
__device__ __forceinline__ f32x2 fma_f16x2_f32x2(uint32_t a, uint32_t b, f32x2 c) {
  float c0, c1, d0, d1;
  unpack2(c, c0, c1);
  asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %4;\n\t"
      "fma.rn.f32.f16 %1, ah, bh, %5;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "r"(a), "r"(b), "f"(c0), "f"(c1));
  return pack2(d0, d1);
}

// Residuals of two elements (2j, 2j+1) under two candidates at once: with a = the first
// candidate's decoded FP16 pair, b = the second's, and na / nb their negated scales (-s, -s) as
// FP16 pairs, returns even = (z0 - a.lo*s_a, z0 - b.lo*s_b) and odd = (z1 - a.hi*s_a,
// z1 - b.hi*s_b), each one FP32 rounding of the exact value (FP16 operands widen exactly).
__device__ __forceinline__ void residuals_two_candidates(uint32_t a, uint32_t na, uint32_t b,
                                                         uint32_t nb, f32x2 z, f32x2& even,
                                                         f32x2& odd) {
  float z0, z1, ae, be, ao, bo;
  unpack2(z, z0, z1);
  asm("{\n\t.reg .f16 a0, a1, b0, b1, sa, sb, xa, xb;\n\t"
      "mov.b32 {a0, a1}, %4;\n\t"
      "mov.b32 {b0, b1}, %6;\n\t"
      "mov.b32 {sa, xa}, %5;\n\t"
      "mov.b32 {sb, xb}, %7;\n\t"
      "fma.rn.f32.f16 %0, a0, sa, %8;\n\t"
      "fma.rn.f32.f16 %1, b0, sb, %8;\n\t"
      "fma.rn.f32.f16 %2, a1, sa, %9;\n\t"
      "fma.rn.f32.f16 %3, b1, sb, %9;\n\t}"
      : "=f"(ae), "=f"(be), "=f"(ao), "=f"(bo)
      : "r"(a), "r"(na), "r"(b), "r"(nb), "f"(z0), "f"(z1));
  even = pack2(ae, be);
  odd = pack2(ao, bo);
}

// FP32 pair to FP16 pair (RNE): .x to the low half.
__device__ __forceinline__ uint32_t f16x2_from_f32x2(f32x2 v) {
  float lo, hi;
  unpack2(v, lo, hi);
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Per half: a*b + c as one FP16 fused multiply-add (RNE).
__device__ __forceinline__ uint32_t fma_f16x2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// FP32 pair to BF16 pair (RNE): .x to the low half.
__device__ __forceinline__ uint32_t bf16x2_from_f32x2(f32x2 v) {
  float lo, hi;
  unpack2(v, lo, hi);
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// E4M3 byte -> table entry (built once per CTA).
__device__ __forceinline__ ScaleEntry make_scale_entry(uint32_t byte) {
  const uint32_t h2 = f16x2_from_e4m3x2(byte | (byte << 8));  // (s, s) in FP16
  const float s = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
  ScaleEntry e;
  e.inv = (s == 0.0f || !(s == s)) ? 0.0f : __frcp_rn(s);
  e.neg_s_h2 = h2 ^ 0x80008000u;
  return e;
}

// Orders this thread's earlier generic-proxy shared-memory writes before later async-proxy
// (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `threads` threads (a multiple of 32) of the CTA.
// Programmatic dependent launch.  pdl_wait: global memory written or read by the previous kernel
// on the stream is safe to use after it (it returns at once for an ordinary launch).
// pdl_trigger: the next kernel on the stream may start its own set-up.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace nvfp4
