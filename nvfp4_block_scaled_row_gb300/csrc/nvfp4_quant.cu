// nvfp4_quant.cu -- the NVFP4 quantize kernels for sm_103a: per-token ("NVFP4 RL" blog, Sec. 2)
// or per-tensor FP32 scale, E4M3 block scales with Four-Over-Six selection (Sec. 4), packed E2M1
// codes, and optionally the BF16 dequantized round trip (Sec. 3) in the same pass.
//
// Shape of the computation.  Every element is read once (2 B) and written once (0.5625 B, plus
// 2 B for the round trip).  CTAs of 16 warps, one per SM, walk the rows in teams of warps that
// share a row, each warp owning a contiguous part of it: the issue-bound quantize-only kernels in
// one static wave, the HBM-bound round trip in work units that running CTAs take over from CTAs
// not yet started (cluster launch control), in order.  Each warp owns a ring of shared-memory
// slots, one part-row per slot, filled by bulk asynchronous copies (cp.async.bulk, the non-tensor
// TMA path) that complete on per-slot mbarriers: while the warp encodes row k, its parts of the
// next rows are in flight.  Per row:
//   pass 1  row amax from shared memory (packed BF16x2 |max|, one redux over the warp, then the
//           team's partial maxima through shared memory);
//   pass 2  one lane per 16-element block: block amax, both candidate E4M3 scales, E2M1 codes
//           for both candidates, their block squared errors, the 4/6 choice, and the stores.
// Each launch is a programmatic dependent of the previous kernel on the stream: shared-memory
// set-up (and an L2 prefetch of the first rows) overlaps that kernel's tail.
// Each block's squared errors are summed in the spec's fixed order -- one FMA chain per
// candidate over the 16 elements in ascending order, the two candidates' chains side by side in
// one packed FP32 pair -- so the result is bit-identical to the CPU oracle and independent of the
// launch shape.
#include <atomic>
#include <cfloat>

#include "nvfp4_device.cuh"
#include "nvfp4_internal.h"

namespace nvfp4 {
namespace {

struct RowFactors {
  float S_enc;  // 6M / a: maps the amax to E2M1_MAXVAL * M
  float c6;     // M / a:   block amax -> scale-to-6 E4M3 scale
  float c4;     // 1.5M / a: block amax -> scale-to-4 E4M3 scale
  float S_dec;  // a / 6M:  the stored FP32 dequant multiplier
};

// "NVFP4 RL" Sec. 4, candidate = fp4 * fp8_scale * amax / (E2M1_MAXVAL * E4M3_4OVER6_MAXVAL),
// with E4M3_4OVER6_MAXVAL = M = 256 (448 in plain mode six).  Each factor is one IEEE division,
// clamped to FLT_MAX when it overflows; a zero amax gives all-zero factors.
template <int kMode>
__device__ __forceinline__ RowFactors row_factors(float a) {
  constexpr float M = (kMode == kModeSix) ? 448.0f : 256.0f;
  RowFactors f;
  if (a == 0.0f) {
    f.S_enc = f.c6 = f.c4 = f.S_dec = 0.0f;
    return f;
  }
  f.S_enc = fminf(__fdiv_rn(6.0f * M, a), FLT_MAX);
  f.c6 = fminf(__fdiv_rn(M, a), FLT_MAX);
  f.c4 = fminf(__fdiv_rn(1.5f * M, a), FLT_MAX);
  f.S_dec = __fdiv_rn(a, 6.0f * M);
  return f;
}

// The same four factors for a warp-uniform amax `a`, each division done once by its own lane
// (lanes 0-3) and broadcast; identical results to row_factors.
template <int kMode>
__device__ __forceinline__ RowFactors row_factors_warp(float a, int lane) {
  constexpr float M = (kMode == kModeSix) ? 448.0f : 256.0f;
  const float num = lane == 0 ? 6.0f * M : (lane == 1 ? M : (lane == 2 ? 1.5f * M : a));
  const float den = lane == 3 ? 6.0f * M : a;
  float q = __fdiv_rn(num, den);
  if (lane < 3) q = fminf(q, FLT_MAX);
  RowFactors f;
  f.S_enc = __shfl_sync(0xFFFFFFFFu, q, 0);
  f.c6 = __shfl_sync(0xFFFFFFFFu, q, 1);
  f.c4 = __shfl_sync(0xFFFFFFFFu, q, 2);
  f.S_dec = __shfl_sync(0xFFFFFFFFu, q, 3);
  if (a == 0.0f) f.S_enc = f.c6 = f.c4 = f.S_dec = 0.0f;
  return f;
}

// One candidate (scale-to-6 or scale-to-4) for a block whose 16 targets z are held as 8 FP32
// pairs in element order: the two packed code words (elements 0-7, then 8-15) and the 8 decoded
// FP16 pairs (element 2j in the low half of r[j]).
struct Codes {
  uint32_t cw[2];
  uint32_t r[8];
};

__device__ __forceinline__ Codes encode_codes(const f32x2 (&z)[8], float inv) {
  Codes c;
  const f32x2 inv2 = pack2(inv, inv);
  f32x2 t[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) t[j] = mul2(z[j], inv2);  // target scaled down by 1/s
  uint32_t lo[4], hi[4];
  c.cw[0] = e2m1x8_encode_decode(t[0], t[1], t[2], t[3], lo);
  c.cw[1] = e2m1x8_encode_decode(t[4], t[5], t[6], t[7], hi);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    c.r[j] = lo[j];
    c.r[4 + j] = hi[j];
  }
  return c;
}

// The block squared errors of both candidates ("NVFP4 RL" blog, Sec. 4: the blockwise error in
// FP32), each summed from +0 over the 16 elements in ascending order, e = fma(d_i, d_i, e), with
// d_i = z_i - r_i * s one rounding of the exact value (r * s is exact).  The two chains run side
// by side in one FP32 pair: .x the scale-to-6 error, .y the scale-to-4 error.
__device__ __forceinline__ f32x2 block_errors(const f32x2 (&z)[8], const Codes& c6, uint32_t ns6,
                                              const Codes& c4, uint32_t ns4) {
  f32x2 acc = pack2(0.0f, 0.0f);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    f32x2 even, odd;
    residuals_two_candidates(c6.r[j], ns6, c4.r[j], ns4, z[j], even, odd);
    acc = fma2(even, even, acc);  // element 2j
    acc = fma2(odd, odd, acc);    // element 2j + 1
  }
  return acc;
}

// The FP16 reading of the 4/6 fast path ("NVFP4 RL" blog, Sec. 4, "The optimization": cast
// losslessly to FP16 and scale the target down by its inverse instead of scaling the candidate
// up): per candidate, the residual of the FP16 target z_h = f16(z) against the exact FP16
// candidate q*s, d = f16(z_h - q*s) (one FP16 FMA of the decoded pair with -s), and its square
// summed in FP32 (exact: d has 11 significant bits) from +0 in ascending element order.  Returns
// (scale-to-6 error, scale-to-4 error).
__device__ __forceinline__ f32x2 block_errors_fp16(const f32x2 (&z)[8], const Codes& c6,
                                                   uint32_t ns6, const Codes& c4, uint32_t ns4) {
  float e6 = 0.0f, e4 = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t zh = f16x2_from_f32x2(z[j]);
    const uint32_t d6 = fma_f16x2(c6.r[j], ns6, zh);
    const uint32_t d4 = fma_f16x2(c4.r[j], ns4, zh);
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %2;\n\t"
        "mov.b32 {b0, b1}, %3;\n\t"
        "fma.rn.f32.f16 %0, a0, a0, %0;\n\t"
        "fma.rn.f32.f16 %1, b0, b0, %1;\n\t"
        "fma.rn.f32.f16 %0, a1, a1, %0;\n\t"
        "fma.rn.f32.f16 %1, b1, b1, %1;\n\t}"
        : "+f"(e6), "+f"(e4)
        : "r"(d6), "r"(d4));
  }
  return pack2(e6, e4);
}

// Encodes one 16-element block with block amax m: both candidates (scale-to-6 only in mode six),
// the 4/6 choice, then stores the 8 code bytes and the E4M3 scale byte.  lo holds elements 0-7
// of the block, hi elements 8-15.  With kWantY, `out` receives the block's dequantized BF16 pairs
// in element order = bf16(fp32(q*s) * S_dec).
template <int kMode, bool kWantY>
__device__ __forceinline__ void encode_block(const uint4 lo, const uint4 hi, float m,
                                             const RowFactors& f, const ScaleEntry* tab,
                                             uint8_t* codes_blk, uint8_t* scale_ptr,
                                             uint32_t (&out)[8]) {
  const f32x2 senc2 = pack2(f.S_enc, f.S_enc);
  const uint16_t one_bf16 = 0x3F80;
  const float neg_zero = -0.0f;
  const float u6 = __fmul_rn(m, f.c6);
  const float u4 = (kMode != kModeSix) ? __fmul_rn(m, f.c4) : 0.0f;
  const uint32_t sb = e4m3x2_from_f32(u4, u6);
  const uint32_t b6 = sb & 0xFFu, b4 = sb >> 8;

  f32x2 z[8];
  z[0] = mul2(bf16x2_to_f32x2_fma(lo.x, one_bf16, neg_zero), senc2);
  z[1] = mul2(bf16x2_to_f32x2_fma(lo.y, one_bf16, neg_zero), senc2);
  z[2] = mul2(bf16x2_to_f32x2_fma(lo.z, one_bf16, neg_zero), senc2);
  z[3] = mul2(bf16x2_to_f32x2_fma(lo.w, one_bf16, neg_zero), senc2);
  z[4] = mul2(bf16x2_to_f32x2_fma(hi.x, one_bf16, neg_zero), senc2);
  z[5] = mul2(bf16x2_to_f32x2_fma(hi.y, one_bf16, neg_zero), senc2);
  z[6] = mul2(bf16x2_to_f32x2_fma(hi.z, one_bf16, neg_zero), senc2);
  z[7] = mul2(bf16x2_to_f32x2_fma(hi.w, one_bf16, neg_zero), senc2);

  const ScaleEntry e6 = tab[b6];
  bool pick4 = false;
  ScaleEntry e4{};
  Codes c4{};
  const Codes c6 = encode_codes(z, e6.inv);
  if (kMode != kModeSix) {
    e4 = tab[b4];
    c4 = encode_codes(z, e4.inv);
    float err6, err4;
    unpack2(kMode == kModeFourOverSixFp16 ? block_errors_fp16(z, c6, e6.neg_s_h2, c4, e4.neg_s_h2)
                                          : block_errors(z, c6, e6.neg_s_h2, c4, e4.neg_s_h2),
            err6, err4);
    pick4 = err4 < err6;  // ties go to 6
  }
  const uint32_t w0 = pick4 ? c4.cw[0] : c6.cw[0];  // the chosen code words
  const uint32_t w1 = pick4 ? c4.cw[1] : c6.cw[1];
  const uint32_t* r = pick4 ? c4.r : c6.r;          // the chosen decoded pairs
  *reinterpret_cast<uint2*>(codes_blk) = make_uint2(w0, w1);
  *scale_ptr = static_cast<uint8_t>(pick4 ? b4 : b6);

  if (kWantY) {
    const uint32_t s_h2 = (pick4 ? e4.neg_s_h2 : e6.neg_s_h2) ^ 0x80008000u;
    const f32x2 sdec2 = pack2(f.S_dec, f.S_dec);
    const f32x2 nzero = pack2(-0.0f, -0.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const f32x2 qs = fma_f16x2_f32x2(r[j], s_h2, nzero);  // q*s, exact
      out[j] = bf16x2_from_f32x2(mul2(qs, sdec2));
    }
  }
}

// A block's two 16-byte halves in element order (lo = elements 0-7) from shared memory.
// kSwizzled: lanes of a quarter-warp read alternate halves first, so every 128-bit read is free
// of bank conflicts, and the halves are then put back in element order with selects; otherwise
// both reads are in element order (two-way bank conflicts, eight fewer instructions per block).
// Measured: the fused round trip, whose global stores share the memory pipe with these reads, is
// 2.5% faster swizzled; the issue-bound quantize-only kernels are 5% faster in element order.
template <bool kSwizzled>
__device__ __forceinline__ void load_block(const unsigned char* blk, uint4& lo, uint4& hi) {
  if (kSwizzled) {
    const int h0 = (threadIdx.x >> 2) & 1;
    const uint4 A = *reinterpret_cast<const uint4*>(blk + h0 * 16);
    const uint4 B = *reinterpret_cast<const uint4*>(blk + (h0 ^ 1) * 16);
    lo = make_uint4(h0 ? B.x : A.x, h0 ? B.y : A.y, h0 ? B.z : A.z, h0 ? B.w : A.w);
    hi = make_uint4(h0 ? A.x : B.x, h0 ? A.y : B.y, h0 ? A.z : B.z, h0 ? A.w : B.w);
  } else {
    lo = *reinterpret_cast<const uint4*>(blk);
    hi = *reinterpret_cast<const uint4*>(blk + 16);
  }
}

// BF16 residual pair bf16(fp32(x) - fp32(y)) of two BF16 pairs.  x - y is exact in FP32 (y is
// zero or within a few binades of x), so one BF16 FMA y * (-1) + x, which rounds the exact
// result once, gives the same bits.
__device__ __forceinline__ uint32_t bf16x2_residual(uint32_t xw, uint32_t yw) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(yw), "r"(0xBF80BF80u), "r"(xw));
  return d;
}

// E2M1 codes of eight BF16 zeros (+0 or -0): the sign of each element in bit 3 of its nibble.
__device__ __forceinline__ uint32_t sign_codes(const uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k)
    out |= (((w[k] >> 12) & 0x8u) | ((w[k] >> 24) & 0x80u)) << (8 * k);
  return out;
}

// Both halves of the result hold the largest |value| of a BF16 pair word (sign bits arbitrary).
__device__ __forceinline__ float abs_max_word(uint32_t mx) {
  const uint32_t mm = max_abs_bf16x2(mx, __byte_perm(mx, 0, 0x1032));
  return fabsf(__uint_as_float(mm << 16));
}

__device__ __forceinline__ uint32_t block_max_word(const uint4 A, const uint4 B) {
  return max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(A.x, A.y), max_abs_bf16x2(A.z, A.w)),
                        max_abs_bf16x2(max_abs_bf16x2(B.x, B.y), max_abs_bf16x2(B.z, B.w)));
}

// Shared-memory layout: [table | amax exchange | abort flags | work queue | copy barriers]
// (ring_header_bytes), then the ring: warp w owns `stages` slots of `slot_bytes`.
//
// Work split: a team of `team` warps shares each row; warp t of a team owns the blocks
// [t*bpw, min(nblk, (t+1)*bpw)) and stages only that part of the row.  Two schedules:
//  - dynamic (the fused round trip, bound by HBM): work unit u is the rows [u*T, u*T + T) of a
//    CTA with T teams, one row per team.  The grid has one CTA per unit (or gridDim.x < units
//    under a launch-shape override, when CTA c walks the units c, c + gridDim.x, ...); a CTA
//    starts with unit blockIdx.x, and when its walk ends it takes over the walk of a CTA of the
//    grid that has not started yet, by cluster launch control, until none is left.  The units go
//    to SMs in order as they free up, so the rows in flight stay one compact window of the
//    matrix and all SMs finish within about one unit of each other.  Thread 0 issues the
//    requests strictly one after another, each only after the previous one was answered with a
//    success (so none follows a failed one, and none can succeed after one failed); every warp
//    reads every answer in order and stops at the first failure.
//  - static (the issue-bound quantize-only and residual kernels, for which a request per unit
//    costs more than it balances): a persistent grid, team gt = team * gridDim.x + blockIdx.x
//    takes the rows gt, gt + NT, gt + 2NT, ... (NT = number of teams); consecutive teams sit on
//    different SMs, so uneven row counts put at most one extra row on an SM.
// With more than one warp per team the row amax is combined
// through shared memory behind a named barrier; if any member's copy times out, all members
// leave together after that barrier.
// kNB > 0: every lane owns exactly kNB blocks of each row (the row's blocks split evenly over the
// team, 32 * kNB per warp), so the block loops have a fixed trip count (residual kernels: only
// the third pass's loop); kNB = 0: any split.
template <int kMode, bool kTensor, bool kFused, bool kResidual, int kNB>
__global__ void __launch_bounds__(kMaxWarpsPerCta * 32, 1) quantize_kernel(const QuantParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  ScaleEntry* tab = reinterpret_cast<ScaleEntry*>(smem);
  float* xch = reinterpret_cast<float*>(smem + kTableBytes);
  int* abort_flag = reinterpret_cast<int*>(smem + kTableBytes + kXchBytes);
  unsigned char* answers = smem + kTableBytes + kXchBytes + kAbortBytes;  // kWorkQueue x 16 B
  uint64_t* q_full = reinterpret_cast<uint64_t*>(answers + kWorkQueue * 16);
  uint64_t* q_free = q_full + kWorkQueue;
  uint64_t* bars = q_free + kWorkQueue;

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int S = p.stages;
  const int TW = p.team;
  const int teams = nwarps / TW;
  const int team = warp / TW;
  const int tw = warp - team * TW;
  unsigned char* ring = smem + ring_header_bytes(nwarps, S);
  uint64_t* my_bars = bars + warp * S;
  unsigned char* my_ring = ring + static_cast<size_t>(warp) * S * p.slot_bytes;

  for (int i = threadIdx.x; i < 256; i += blockDim.x) tab[i] = make_scale_entry(i);
  if (threadIdx.x < kMaxWarpsPerCta) abort_flag[threadIdx.x] = 0;
  if (lane == 0)
    for (int s = 0; s < S; ++s) mbar_init(&my_bars[s], 1);
  if (threadIdx.x == 0)
    for (int i = 0; i < kWorkQueue; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_free[i], nwarps);
    }
  fence_barrier_init();
  __syncthreads();

  // ---- work units ----
  constexpr bool kDynamic = kFused;
  const int64_t units = (p.rows + teams - 1) / teams;
  const int64_t G = gridDim.x;
  const int64_t gt = static_cast<int64_t>(team) * G + blockIdx.x;  // static schedule
  const int64_t NT = G * teams;
  // The row of this team in unit u (dynamic) or step u (static); p.rows for none.
  auto row_of = [&](int64_t u) -> int64_t {
    if (u < 0) return p.rows;
    if constexpr (kDynamic) return u * teams + team;
    return gt + u * NT;
  };
  // When warp 0 reads answer j, thread 0 first makes sure requests up to j + kLead - 1 are out,
  // so the other warps rarely wait for one.
  constexpr int kLead = 3;
  // Thread 0: requests issued so far (request j >= 1 uses queue entry j % kWorkQueue for the
  // ((j - 1) / kWorkQueue)-th time), and whether it has stopped issuing.
  int requested = 0;
  bool stop_requests = false;
  auto request_next = [&]() {
    const int j = requested + 1;
    if (j >= 2) {  // the previous request must have been answered with a success
      const int q = (j - 1) % kWorkQueue;
      uint32_t unused;
      if (!mbar_wait_bounded(&q_full[q], static_cast<uint32_t>(((j - 2) / kWorkQueue) & 1),
                             p.timeout_ns)) {
        record_status(p.status, kStatusTimeout);
        stop_requests = true;
        return;
      }
      if (!launch_control_answer(answers + q * 16, unused)) {
        stop_requests = true;
        return;
      }
    }
    const int q = j % kWorkQueue;
    const int use = (j - 1) / kWorkQueue;
    // The entry's previous answer must have been read by every warp.
    if (use >= 1 && !mbar_wait_bounded(&q_free[q], static_cast<uint32_t>((use - 1) & 1),
                                       p.timeout_ns)) {
      record_status(p.status, kStatusTimeout);
      stop_requests = true;
      return;
    }
    mbar_arrive_expect_tx(&q_full[q], 16);
    launch_control_request(answers + q * 16, &q_full[q]);
    requested = j;
  };
  // Before thread 0 leaves early: wait (bounded) for its last request's answer, so that it does
  // not land after the CTA is gone.
  auto drain_requests = [&]() {
    if (requested >= 1)
      (void)mbar_wait_bounded(&q_full[requested % kWorkQueue],
                              static_cast<uint32_t>(((requested - 1) / kWorkQueue) & 1),
                              p.drain_timeout_ns);
  };
  // Warp-collective: the next answer in order (-1 once one failed; every warp reads each once).
  int answers_read = 0;
  bool ended = false;
  auto read_answer = [&]() -> int64_t {
    if (ended) return -1;
    int64_t u = -1;
    if (lane == 0) {
      const int j = answers_read + 1;
      if (threadIdx.x == 0)
        while (!stop_requests && requested < j + kLead - 1) request_next();
      const int q = j % kWorkQueue;
      if (mbar_wait_bounded(&q_full[q], static_cast<uint32_t>(((j - 1) / kWorkQueue) & 1),
                            p.timeout_ns)) {
        uint32_t x;
        if (launch_control_answer(answers + q * 16, x)) u = static_cast<int64_t>(x);
        mbar_arrive(&q_free[q]);
      } else {
        record_status(p.status, kStatusTimeout);
      }
      answers_read = j;
    }
    u = __shfl_sync(0xFFFFFFFFu, u, 0);
    if (u < 0 || u >= units) {
      ended = true;
      u = -1;
    }
    return u;
  };
  // The unit after `u` in this CTA's order (-1: none left).
  auto next_unit = [&](int64_t u) -> int64_t {
    if (u < 0) return -1;
    if constexpr (kDynamic) return u + G < units ? u + G : read_answer();
    return gt + (u + 1) * NT < p.rows ? u + 1 : -1;
  };
  // Lane s (s < S) holds the unit of the steps that use ring slot s; `last` is the unit of the
  // latest step assigned so far.
  int64_t slot_unit = -1;
  int64_t last = kDynamic ? static_cast<int64_t>(blockIdx.x) : (gt < p.rows ? 0 : -1);
  if (lane == 0) slot_unit = last;
  for (int s = 1; s < S; ++s) {
    last = next_unit(last);
    if (lane == s) slot_unit = last;
  }

  // Everything above touched only this CTA's shared memory, so it overlaps the previous kernel's
  // tail; global memory waits for that kernel (except the first row copies of a tensor-scale grid
  // that follows our amax kernel, see below).
  const int cols = p.cols;
  const int nblk = cols / kBlockElems;
  const int b0 = tw * p.blocks_per_warp;
  const int b1 = min(nblk, b0 + p.blocks_per_warp);
  const bool has_work = b1 > b0;
  const uint32_t chunk_bytes = has_work ? static_cast<uint32_t>(b1 - b0) * 32u : 0u;
  if (!p.prologue_before_wait) {
    // While the previous kernel finishes, pull this warp's first rows into L2 (coherent, so safe
    // even if that kernel writes them); the copies after the wait then hit L2.  Measured: the
    // fused round trip gains 2.3% prefetching all its ring's rows; quantize-only kernels lose 2%
    // doing the same but gain 0.5-2.5% prefetching only the first row.  Residual kernels skip it.
    const int np = kFused ? S : ((kResidual || !has_work) ? 0 : 1);
    for (int s = 0; s < np; ++s) {
      const int64_t r = row_of(__shfl_sync(0xFFFFFFFFu, slot_unit, s));
      if (lane == 0 && has_work && r < p.rows)
        bulk_prefetch_l2(p.x + r * cols + b0 * 16, chunk_bytes);
    }
    pdl_wait();
  }
  pdl_trigger();

  const uint64_t policy = l2_evict_first_policy();
  const int h0 = (lane >> 2) & 1;  // which 16-byte half of its block this lane reads first

  // Copies in flight (lane 0): bit s of `pending` is set while slot s has one; bit s of `phase`
  // is the parity of the slot barrier's next phase.  (The self-test's withheld row is never
  // copied, so its step's wait runs out.)
  uint32_t pending = 0, phase = 0;
  auto issue = [&](int slot_index, int64_t row) {
    if (row != p.withhold_row) {
      mbar_arrive_expect_tx(&my_bars[slot_index], chunk_bytes);
      bulk_load(my_ring + static_cast<size_t>(slot_index) * p.slot_bytes,
                p.x + row * cols + b0 * 16, chunk_bytes, &my_bars[slot_index], policy);
      pending |= 1u << slot_index;
    }
  };
  // Before an early exit (lane 0): wait (bounded) for this warp's copies still in flight, so that
  // none lands after the warp is gone; thread 0 also waits for its last request's answer.
  auto drain = [&]() {
    for (int s = 0; s < S; ++s)
      if ((pending >> s) & 1u)
        (void)mbar_wait_bounded(&my_bars[s], (phase >> s) & 1u, p.drain_timeout_ns);
    if (threadIdx.x == 0) drain_requests();
  };
  // Prologue: fill the ring with this warp's part of the team's first rows.
  for (int s = 0; s < S; ++s) {
    const int64_t r = row_of(__shfl_sync(0xFFFFFFFFu, slot_unit, s));
    if (lane == 0 && has_work && r < p.rows) issue(s, r);
  }

  RowFactors f{};
  if (kTensor) {
    // Tensor scale right after the amax kernel: x is not written there, so the copies above may
    // already run; the partial maxima need that grid complete.
    if (p.prologue_before_wait) pdl_wait();
    float a = 0.0f;
    for (int i = lane; i < p.n_amax; i += 32) a = fmaxf(a, p.amax_src[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    f = row_factors<kMode>(a);
  }

  // Once per grid, by the first warp of the team that has row 0 (dynamic: whichever CTA got unit
  // 0; static: CTA 0): the tensor scale, and the group offsets, which only need validating (every
  // row is quantized independently of its group).
  auto grid_once = [&]() {
    if (kTensor && lane == 0) p.scale_out[0] = f.S_dec;
    if (p.offsets != nullptr) {
      bool bad = false;
      for (int i = lane; i <= p.num_groups; i += 32) {
        const int32_t v = p.offsets[i];
        if (i == 0 && v != 0) bad = true;
        if (i == p.num_groups && static_cast<int64_t>(v) != p.rows) bad = true;
        if (i > 0 && p.offsets[i - 1] > v) bad = true;
      }
      if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) record_status(p.status, kStatusOffsets);
    }
  };
  if (!kDynamic && gt == 0 && tw == 0) grid_once();

  // Step k uses ring slot k mod S (advanced incrementally); its row comes from the unit held by
  // lane `slot` (dynamic) or advances by NT (static).
  int slot = 0;
  int64_t row = gt;
  for (int64_t k = 0;; ++k) {
    if constexpr (kDynamic) {
      const int64_t unit = __shfl_sync(0xFFFFFFFFu, slot_unit, slot);
      if (unit < 0) break;
      row = row_of(unit);
    } else {
      if (row >= p.rows) break;
    }
    if (kDynamic && row == 0 && tw == 0) grid_once();
    if (row < p.rows) {
      int ok = 1;
      if (lane == 0 && has_work) {
        ok = mbar_wait_bounded(&my_bars[slot], (phase >> slot) & 1u, p.timeout_ns) ? 1 : 0;
        if (ok) {
          phase ^= 1u << slot;
          pending &= ~(1u << slot);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      const bool team_sync = !kTensor && TW > 1;
      if (!ok && lane == 0) record_status(p.status, kStatusTimeout);
      if (!ok && !team_sync) {
        // A copy did not land in time: wait for the copies still in flight, and stop.
        if (lane == 0) drain();
        return;
      }
      unsigned char* xs = my_ring + static_cast<size_t>(slot) * p.slot_bytes;

      // Pass 1 (row scale): block maxima (kept in registers for pass 2) and the row amax.
      uint32_t bmax[kMaxBlocksPerLane];
      if (!kTensor) {
        uint32_t m2 = 0;
#pragma unroll
        for (int j = 0; j < kMaxBlocksPerLane; ++j) {
          const int b = b0 + lane + 32 * j;
          bmax[j] = 0;
          if ((kNB > 0 && !kResidual) ? j < kNB : (ok && b < b1)) {
            const unsigned char* blk = xs + (b - b0) * 32;
            const uint4 A = *reinterpret_cast<const uint4*>(blk + h0 * 16);
            const uint4 B = *reinterpret_cast<const uint4*>(blk + (1 - h0) * 16);
            bmax[j] = block_max_word(A, B);
            m2 = max_abs_bf16x2(m2, bmax[j]);
          }
        }
        // Row amax: the largest BF16 magnitude of the warp (as its bit pattern, which orders like
        // the magnitude), then the team's.
        const uint32_t mh = m2 & 0x7FFF7FFFu;
        const uint32_t mtop = __reduce_max_sync(0xFFFFFFFFu, max(mh >> 16, mh & 0xFFFFu));
        float a = __uint_as_float(mtop << 16);
        if (team_sync) {
          float* part = xch + (k & 1) * kMaxWarpsPerCta;
          if (lane == 0) {
            part[warp] = a;
            if (!ok) abort_flag[team] = 1;
          }
          named_barrier(1 + team, TW * 32);
          if (abort_flag[team]) {
            if (lane == 0) drain();
            return;
          }
          a = 0.0f;
          for (int j = 0; j < TW; ++j) a = fmaxf(a, part[team * TW + j]);
        }
        f = row_factors_warp<kMode>(a, lane);
        if (lane == 0 && tw == 0) p.scale_out[row] = f.S_dec;
      }

      // Pass 2: encode this warp's blocks (residual kernels also turn each block into its BF16
      // residual x - DQ(Q(x)) in place, with the residual's block maxima kept for pass 3).
      uint8_t* codes_row = p.codes + row * (cols / 2);
      uint8_t* scales_row = p.scales + row * nblk;
      uint32_t rmax[kMaxBlocksPerLane];
      uint32_t rm2 = 0;
      if (!kResidual && f.S_dec == 0.0f) {
        // Zero amax (a padding row, or an all-zero tensor): every element is +-0, so every scale
        // is 0, every code is the sign of its element (0x0 or 0x8) and y = x, bit for bit.
#pragma unroll
        for (int j = 0; j < (kNB > 0 ? kNB : kMaxBlocksPerLane); ++j) {
          const int b = b0 + lane + 32 * j;
          if (kNB == 0 && b >= b1) break;
          const unsigned char* blk = xs + (b - b0) * 32;
          const uint4 A = *reinterpret_cast<const uint4*>(blk + h0 * 16);
          const uint4 B = *reinterpret_cast<const uint4*>(blk + (1 - h0) * 16);
          uint32_t* cw = reinterpret_cast<uint32_t*>(codes_row + b * 8);
          cw[h0] = sign_codes(A);
          cw[1 - h0] = sign_codes(B);
          scales_row[b] = 0;
          if (kFused) {
            uint16_t* y_blk = p.y + row * cols + b * kBlockElems;
            *reinterpret_cast<uint4*>(y_blk + h0 * 8) = A;
            *reinterpret_cast<uint4*>(y_blk + (1 - h0) * 8) = B;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < ((kNB > 0 && !kResidual) ? kNB : kMaxBlocksPerLane); ++j) {
          const int b = b0 + lane + 32 * j;
          if ((kNB == 0 || kResidual) && b >= b1) break;
          unsigned char* blk = xs + (b - b0) * 32;
          uint4 lo, hi;
          load_block<kFused>(blk, lo, hi);
          const float m = abs_max_word(kTensor ? block_max_word(lo, hi) : bmax[j]);
          uint32_t out[8];
          encode_block<kMode, kFused || kResidual>(lo, hi, m, f, tab, codes_row + b * 8,
                                                   scales_row + b, out);
          if (kFused) {
            uint16_t* y_blk = p.y + row * cols + b * kBlockElems;
            *reinterpret_cast<uint4*>(y_blk) = make_uint4(out[0], out[1], out[2], out[3]);
            *reinterpret_cast<uint4*>(y_blk + 8) = make_uint4(out[4], out[5], out[6], out[7]);
          }
          if (kResidual) {
            const uint4 RL =
                make_uint4(bf16x2_residual(lo.x, out[0]), bf16x2_residual(lo.y, out[1]),
                           bf16x2_residual(lo.z, out[2]), bf16x2_residual(lo.w, out[3]));
            const uint4 RH =
                make_uint4(bf16x2_residual(hi.x, out[4]), bf16x2_residual(hi.y, out[5]),
                           bf16x2_residual(hi.z, out[6]), bf16x2_residual(hi.w, out[7]));
            *reinterpret_cast<uint4*>(blk) = RL;
            *reinterpret_cast<uint4*>(blk + 16) = RH;
            rmax[j] = block_max_word(RL, RH);
            rm2 = max_abs_bf16x2(rm2, rmax[j]);
          }
        }
      }

      if (kResidual) {
        // Pass 3: the residual's own per-token scale, then its blocks.
        const uint32_t rh = rm2 & 0x7FFF7FFFu;
        const uint32_t rtop = __reduce_max_sync(0xFFFFFFFFu, max(rh >> 16, rh & 0xFFFFu));
        float a = __uint_as_float(rtop << 16);
        if (TW > 1) {
          float* part = xch + (2 + (k & 1)) * kMaxWarpsPerCta;
          if (lane == 0) part[warp] = a;
          named_barrier(1 + team, TW * 32);
          a = 0.0f;
          for (int j = 0; j < TW; ++j) a = fmaxf(a, part[team * TW + j]);
        }
        const RowFactors g = row_factors_warp<kMode>(a, lane);
        if (lane == 0 && tw == 0) p.res_scale_out[row] = g.S_dec;
        uint8_t* rcodes_row = p.res_codes + row * (cols / 2);
        uint8_t* rscales_row = p.res_scales + row * nblk;
#pragma unroll
        for (int j = 0; j < (kNB > 0 ? kNB : kMaxBlocksPerLane); ++j) {
          const int b = b0 + lane + 32 * j;
          if (kNB == 0 && b >= b1) break;
          uint4 lo, hi;
          load_block<false>(xs + (b - b0) * 32, lo, hi);
          uint32_t unused[8];
          encode_block<kMode, false>(lo, hi, abs_max_word(rmax[j]), g, tab, rcodes_row + b * 8,
                                     rscales_row + b, unused);
        }
        fence_proxy_async_smem();  // the residual writes above precede the slot's next bulk copy
      }

    }  // row < p.rows

    // Slot consumed: refill it with this warp's part of the row `stages` steps ahead.
    __syncwarp();
    int64_t next;
    if constexpr (kDynamic) {
      last = next_unit(last);
      if (lane == slot) slot_unit = last;
      next = row_of(last);
    } else {
      next = row + static_cast<int64_t>(S) * NT;
      row += NT;
    }
    if (lane == 0 && has_work && next < p.rows) issue(slot, next);
    if (++slot == S) slot = 0;
  }
  // Every request thread 0 issued has been answered: the warps read them all up to the first
  // failure, which is the last one issued.
}

constexpr int kGuidedUnroll = 4;  // 8-element groups per lane per step of the guided encoder

// Sign masks of eight FP32 values as nibbles: nibble i of the result is 0xF when v[i] has its
// sign bit set, else 0.  prmt's sign-replicating selectors (selector msb set) copy the top bit of
// byte 3 of each value into a whole byte; two bytes per element pair are then merged into nibbles.
__device__ __forceinline__ uint32_t sign_nibbles(const float (&v)[8]) {
  uint32_t a, b, even, p02, p46, p13, p57, odd;
  asm("prmt.b32 %0, %1, %2, 0x00FB;" : "=r"(p02) : "f"(v[0]), "f"(v[2]));
  asm("prmt.b32 %0, %1, %2, 0xFB00;" : "=r"(p46) : "f"(v[4]), "f"(v[6]));
  asm("prmt.b32 %0, %1, %2, 0x7610;" : "=r"(a) : "r"(p02), "r"(p46));
  asm("prmt.b32 %0, %1, %2, 0x00FB;" : "=r"(p13) : "f"(v[1]), "f"(v[3]));
  asm("prmt.b32 %0, %1, %2, 0xFB00;" : "=r"(p57) : "f"(v[5]), "f"(v[7]));
  asm("prmt.b32 %0, %1, %2, 0x7610;" : "=r"(b) : "r"(p13), "r"(p57));
  even = a & 0x0F0F0F0Fu;  // byte k: element 2k -> low nibble
  odd = b & 0xF0F0F0F0u;   // byte k: element 2k+1 -> high nibble
  return even | odd;
}

// TRACE rollout-guided rounding ("TRACE FP4 RL -- Rollout-guided FP4 rounding"): with the
// rollout's per-token amax and block scales, each element's scaled value t is formed exactly as
// the quantizer forms it; of its two neighbouring codewords the one closer to the rollout's
// recorded codeword is kept.  Elementwise: warps walk rows, lane l owns 8-element group l of each
// 256-element chunk.  The neighbours come from the hardware round-to-nearest code m of t: if the
// rounding went away from zero they are (m-1, m), towards zero (m, m+1), none if t is on the grid
// or saturated.  Of two adjacent magnitudes the larger is closer to the rollout's codeword exactly
// when that codeword lies on t's side of zero with magnitude >= it.
//
// The decision runs on all eight nibbles of a code word at once.  With u = r - t and v = t - r
// (both exact in sign; both +0 when t is on the grid), rounding went away from zero where
// t >= 0 and v < 0, or t < 0 and u < 0; towards zero where t >= 0 and u < 0, or t < 0 and v < 0.
// Magnitude comparisons of the rollout's codes R with m use borrow-free nibble subtraction
// ((R | 8) - m keeps bit 3 exactly when R >= m).  The magnitude then moves by -1 (away, unless the
// rollout's code is on the same side with R >= m) or +1 (towards, when it is with R > m).
// One 8-element group of the guided encoder: xw = the trainer's eight BF16 values, ref = the
// rollout's eight codes (element i in nibble i), e = the rollout's block scale.  Returns the
// eight output codes.
__device__ __forceinline__ uint32_t guided_group(const uint4 xw, uint32_t ref, const ScaleEntry e,
                                                 f32x2 senc2) {
  const uint32_t one_h2 = 0x3C003C00u;   // FP16 (1, 1)
  const uint32_t mone_h2 = 0xBC00BC00u;  // FP16 (-1, -1)
  const f32x2 inv2 = pack2(e.inv, e.inv);
  const f32x2 ninv2 = pack2(-e.inv, -e.inv);
  f32x2 z[4], t[4];
  z[0] = mul2(bf16x2_to_f32x2(xw.x), senc2);
  z[1] = mul2(bf16x2_to_f32x2(xw.y), senc2);
  z[2] = mul2(bf16x2_to_f32x2(xw.z), senc2);
  z[3] = mul2(bf16x2_to_f32x2(xw.w), senc2);
#pragma unroll
  for (int j = 0; j < 4; ++j) t[j] = mul2(z[j], inv2);
  uint32_t r[4];
  const uint32_t rtn = e2m1x8_encode_decode(t[0], t[1], t[2], t[3], r);
  float uu[8], vv[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const f32x2 nt = mul2(z[j], ninv2);                     // -t, exactly
    const f32x2 uj = fma_f16x2_f32x2(r[j], one_h2, nt);     // r - t, one rounding
    const f32x2 vj = fma_f16x2_f32x2(r[j], mone_h2, t[j]);  // t - r, one rounding
    unpack2(uj, uu[2 * j], uu[2 * j + 1]);
    unpack2(vj, vv[2 * j], vv[2 * j + 1]);
  }
  const uint32_t su = sign_nibbles(uu), sv = sign_nibbles(vv);
  const uint32_t st = rtn & 0x88888888u;                        // sign of t (bit 3)
  const uint32_t away = (st & su) | (~st & sv);                 // bit 3 meaningful
  const uint32_t toward = (st & sv) | (~st & su);
  const uint32_t mag = rtn & 0x77777777u;
  const uint32_t rg = ref | 0x88888888u;
  const uint32_t ge = rg - mag;                                 // bit 3: R >= m
  const uint32_t gt = rg - mag - 0x11111111u;                   // bit 3: R > m
  const uint32_t other = rtn ^ ref;                             // bit 3: R on the other side
  const uint32_t down = away & (~ge | other) & 0x88888888u;
  const uint32_t up = toward & gt & ~other & 0x88888888u;
  return rtn + (up >> 3) - (down >> 3);
}

template <int kMode>
__global__ void __launch_bounds__(256) guided_kernel(const GuidedParams p) {
  __shared__ ScaleEntry tab[256];
  for (int i = threadIdx.x; i < 256; i += blockDim.x) tab[i] = make_scale_entry(i);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t NW = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int cols = p.cols;
  const int ngroups = cols / 8;
  // Work units: kGuidedUnroll * 32 consecutive 8-element groups of one row, so a lane has
  // kGuidedUnroll independent loads in flight.  Each warp takes a contiguous range of units (the
  // row factors are recomputed only when the row changes), which balances rows across warps.
  const int units_per_row = (ngroups + 32 * kGuidedUnroll - 1) / (32 * kGuidedUnroll);
  const int64_t total = p.rows * units_per_row;
  const int64_t per_warp = (total + NW - 1) / NW;
  const int64_t u_begin = gw * per_warp;
  const int64_t u_end = min(total, u_begin + per_warp);
  if (lane == 0 && u_begin < u_end) {  // this warp's first x bytes into L2 while the wait runs
    const int64_t r0 = u_begin / units_per_row;
    const int g0 = static_cast<int>(u_begin - r0 * units_per_row) * 32 * kGuidedUnroll;
    const int n = min(ngroups - g0, 32 * kGuidedUnroll);
    bulk_prefetch_l2(p.x + r0 * cols + g0 * 8, static_cast<uint32_t>(n) * 16u);
  }
  pdl_wait();  // global memory only after the previous kernel on the stream
  pdl_trigger();
  int64_t cur_row = -1;
  f32x2 senc2 = pack2(0.0f, 0.0f);
  int64_t row = u_begin / units_per_row;  // walked forward below, without further divisions
  int unit = static_cast<int>(u_begin - row * units_per_row);
  for (int64_t u = u_begin; u < u_end; ++u, ++unit) {
    if (unit == units_per_row) {
      unit = 0;
      ++row;
    }
    if (row != cur_row) {
      const RowFactors f = row_factors_warp<kMode>(p.row_amax[row], lane);
      senc2 = pack2(f.S_enc, f.S_enc);
      cur_row = row;
    }
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + row * cols);
    const uint32_t* rr = reinterpret_cast<const uint32_t*>(p.ref_codes + row * (cols / 2));
    const uint8_t* sr = p.ref_scales + row * (cols / kBlockElems);
    uint32_t* out = reinterpret_cast<uint32_t*>(p.codes + row * (cols / 2));
    const int g0 = unit * 32 * kGuidedUnroll + lane;
    uint4 xw[kGuidedUnroll];
    uint32_t ref[kGuidedUnroll], sb[kGuidedUnroll];
#pragma unroll
    for (int k = 0; k < kGuidedUnroll; ++k) {
      const int g = g0 + 32 * k;
      if (g < ngroups) {
        xw[k] = __ldcs(xr + g);
        ref[k] = __ldcs(rr + g);
        sb[k] = sr[g >> 1];
      }
    }
#pragma unroll
    for (int k = 0; k < kGuidedUnroll; ++k) {
      const int g = g0 + 32 * k;
      if (g >= ngroups) break;
      __stcs(out + g, guided_group(xw[k], ref[k], tab[sb[k]], senc2));
    }
  }
}

// The guided encoder with its inputs staged through shared memory: rows whose width is a multiple
// of kGuidedChunk (and 16-byte aligned tensors).  Work unit = one kGuidedChunk-element piece of a
// row: its BF16 values, the rollout's codes and block scales, moved by three bulk copies into
// one slot of the warp's ring (completing on the slot's mbarrier), so each warp keeps
// kGuidedStages units of loads in flight instead of one per lane.  Lane l then encodes groups
// l, l + 32, ... of the unit from shared memory exactly as guided_kernel does.
constexpr int kGuidedChunk = 32 * kGuidedUnroll * 8;                  // 1024 elements
constexpr int kGuidedXBytes = kGuidedChunk * 2;
constexpr int kGuidedCodeBytes = kGuidedChunk / 2;
constexpr int kGuidedScaleBytes = kGuidedChunk / kBlockElems;
constexpr int kGuidedSlotBytes =
    ((kGuidedXBytes + kGuidedCodeBytes + kGuidedScaleBytes + 127) / 128) * 128;
constexpr int kGuidedStages = 4;
constexpr int kGuidedWarps = 16;
constexpr int kGuidedBarBytes = ((kGuidedWarps * kGuidedStages * 8 + 127) / 128) * 128;
constexpr size_t kGuidedSmem = kTableBytes + kGuidedBarBytes +
                               static_cast<size_t>(kGuidedWarps) * kGuidedStages * kGuidedSlotBytes;

template <int kMode>
__global__ void __launch_bounds__(kGuidedWarps * 32, 1) guided_ring_kernel(const GuidedParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  ScaleEntry* tab = reinterpret_cast<ScaleEntry*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTableBytes);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  uint64_t* my_bars = bars + warp * kGuidedStages;
  unsigned char* my_ring = smem + kTableBytes + kGuidedBarBytes +
                           static_cast<size_t>(warp) * kGuidedStages * kGuidedSlotBytes;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) tab[i] = make_scale_entry(i);
  if (lane == 0)
    for (int s = 0; s < kGuidedStages; ++s) mbar_init(&my_bars[s], 1);
  fence_barrier_init();
  __syncthreads();

  const int cols = p.cols;
  const int upr = cols / kGuidedChunk;  // units per row
  const int64_t total = p.rows * upr;
  const int64_t NW = static_cast<int64_t>(gridDim.x) * nwarps;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
  const int64_t per_warp = (total + NW - 1) / NW;
  const int64_t u_begin = min(total, gw * per_warp);
  const int64_t u_end = min(total, u_begin + per_warp);
  const uint64_t policy = l2_evict_first_policy();

  // Copy cursor (lane 0): the row and chunk of the next unit to copy, walked without divisions.
  int64_t c_row = u_begin / upr;
  int c_chunk = static_cast<int>(u_begin - c_row * upr);
  int64_t copied = u_begin;
  uint32_t pending = 0, phase = 0;
  if (lane == 0 && u_begin < u_end)  // the first unit's values into L2 while the wait runs
    bulk_prefetch_l2(p.x + c_row * cols + c_chunk * kGuidedChunk, kGuidedXBytes);
  pdl_wait();  // global memory only after the previous kernel on the stream
  pdl_trigger();
  // (The self-test's withheld row is never copied, so the wait for its units runs out.)
  auto issue = [&](int slot) {
    if (c_row != p.withhold_row) {
      unsigned char* dst = my_ring + slot * kGuidedSlotBytes;
      const int64_t e0 = c_row * cols + static_cast<int64_t>(c_chunk) * kGuidedChunk;
      mbar_arrive_expect_tx(&my_bars[slot], kGuidedXBytes + kGuidedCodeBytes + kGuidedScaleBytes);
      bulk_load(dst, p.x + e0, kGuidedXBytes, &my_bars[slot], policy);
      bulk_load(dst + kGuidedXBytes, p.ref_codes + e0 / 2, kGuidedCodeBytes, &my_bars[slot],
                policy);
      bulk_load(dst + kGuidedXBytes + kGuidedCodeBytes, p.ref_scales + e0 / kBlockElems,
                kGuidedScaleBytes, &my_bars[slot], policy);
      pending |= 1u << slot;
    }
    ++copied;
    if (++c_chunk == upr) {
      c_chunk = 0;
      ++c_row;
    }
  };
  if (lane == 0)
    for (int s = 0; s < kGuidedStages && copied < u_end; ++s) issue(s);

  int64_t row = u_begin / upr;
  int chunk = static_cast<int>(u_begin - row * upr);
  int64_t cur_row = -1;
  f32x2 senc2 = pack2(0.0f, 0.0f);
  int slot = 0;
  for (int64_t u = u_begin; u < u_end; ++u) {
    int ok = 1;
    if (lane == 0) {
      ok = mbar_wait_bounded(&my_bars[slot], (phase >> slot) & 1u, p.timeout_ns) ? 1 : 0;
      if (ok) {
        phase ^= 1u << slot;
        pending &= ~(1u << slot);
      }
    }
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) {
      // A copy did not land in time: wait (bounded) for the copies still in flight, and stop.
      if (lane == 0) {
        record_status(p.status, kStatusTimeout);
        for (int s = 0; s < kGuidedStages; ++s)
          if ((pending >> s) & 1u)
            (void)mbar_wait_bounded(&my_bars[s], (phase >> s) & 1u, p.drain_timeout_ns);
      }
      return;
    }
    if (row != cur_row) {
      const RowFactors f = row_factors_warp<kMode>(p.row_amax[row], lane);
      senc2 = pack2(f.S_enc, f.S_enc);
      cur_row = row;
    }
    const unsigned char* xs = my_ring + slot * kGuidedSlotBytes;
    uint32_t* out = reinterpret_cast<uint32_t*>(p.codes + row * (cols / 2)) +
                    chunk * (kGuidedChunk / 8);
#pragma unroll
    for (int k = 0; k < kGuidedUnroll; ++k) {
      const int g = lane + 32 * k;  // 8-element group of the unit
      const uint4 xw = *reinterpret_cast<const uint4*>(xs + g * 16);
      const uint32_t ref = *reinterpret_cast<const uint32_t*>(xs + kGuidedXBytes + g * 4);
      const uint32_t sb = xs[kGuidedXBytes + kGuidedCodeBytes + (g >> 1)];
      __stcs(out + g, guided_group(xw, ref, tab[sb], senc2));
    }
    // Slot consumed: refill it with this warp's unit kGuidedStages ahead.
    __syncwarp();
    if (lane == 0 && copied < u_end) issue(slot);
    if (++slot == kGuidedStages) slot = 0;
    if (++chunk == upr) {
      chunk = 0;
      ++row;
    }
  }
}

// Per-row amax max |x| over each row of `cols` BF16 values (warp per row).
__global__ void __launch_bounds__(256) row_amax_kernel(const uint16_t* x, int64_t rows, int cols,
                                                       float* amax) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t NW = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = gw; row < rows; row += NW) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * cols);
    const int nvec = cols / 8;
    uint32_t m2 = 0;
    int g = lane;
    for (; g + 96 < nvec; g += 128) {  // four independent 16-byte loads in flight per lane
      uint4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = __ldcs(xr + g + 32 * k);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        m2 = max_abs_bf16x2(m2, max_abs_bf16x2(max_abs_bf16x2(v[k].x, v[k].y),
                                               max_abs_bf16x2(v[k].z, v[k].w)));
    }
    for (; g < nvec; g += 32) {
      const uint4 v = __ldcs(xr + g);
      m2 = max_abs_bf16x2(m2, max_abs_bf16x2(max_abs_bf16x2(v.x, v.y), max_abs_bf16x2(v.z, v.w)));
    }
    float a = abs_max_of_pair(m2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
    if (lane == 0) amax[row] = a;
  }
}

struct RingShape {
  int warps;
  int stages;
  int team;
  int blocks_per_warp;
  uint32_t slot_bytes;
  size_t smem;
};

constexpr size_t kSmemLimit = 227 * 1024;
constexpr uint32_t kTargetSlotBytes = 8192;  // split rows wider than this across a team

// Team size, ring depth and warps per CTA for rows of `cols` elements: as many warps as shared
// memory allows (up to 16), then as many stages as fit (up to 4, at least 2 when possible).
bool choose_ring(int64_t cols, RingShape* out, int warps_cap = 0) {
  if (cols <= 0 || cols % kBlockElems != 0 || cols > kMaxCols) return false;
  const int nblk = static_cast<int>(cols / kBlockElems);
  int team = 1;
  while (team < kMaxTeam && ((nblk + team - 1) / team) * 32u > kTargetSlotBytes) team *= 2;
  while (team > 1 && (team - 1) * ((nblk + team - 1) / team) >= nblk) team /= 2;
  const int bpw = (nblk + team - 1) / team;
  const uint32_t slot = static_cast<uint32_t>(((bpw * 32 + 127) / 128) * 128);
  const LaunchOverride ov = launch_override();
  int max_warps = kMaxWarpsPerCta;
  if (ov.warps_per_cta > 0) max_warps = ov.warps_per_cta < team ? team : ov.warps_per_cta;
  else if (warps_cap > 0 && warps_cap < max_warps) max_warps = warps_cap < team ? team : warps_cap;
  max_warps -= max_warps % team;
  for (int min_stages : {2, 1}) {
    for (int warps = max_warps; warps >= team; warps -= team) {
      for (int stages = kMaxStages; stages >= min_stages; --stages) {
        if (ov.stages > 0 && stages != ov.stages) continue;
        const size_t smem = static_cast<size_t>(ring_header_bytes(warps, stages)) +
                            static_cast<size_t>(warps) * stages * slot;
        if (smem > kSmemLimit) continue;
        out->warps = warps;
        out->stages = stages;
        out->team = team;
        out->blocks_per_warp = bpw;
        out->slot_bytes = slot;
        out->smem = smem;
        return true;
      }
    }
  }
  return false;
}

// Per kernel instantiation and device: whether the shared-memory limit has been raised, and the
// resident CTAs per SM for each launch shape seen (looked up once, then reused).
struct LaunchCache {
  static constexpr int kDevices = 64;
  static constexpr int kShapes = 32;
  std::atomic<int> attr_set[kDevices];
  struct Entry {
    std::atomic<long long> key;  // warps | stages << 8 | slot_bytes << 16, 0 = empty
    std::atomic<int> per_sm;
  } entries[kDevices][kShapes];
};

template <int kMode, bool kTensor, bool kFused, bool kResidual, int kNB>
cudaError_t launch_impl(QuantParams p, cudaStream_t stream, bool after_amax_kernel) {
  static LaunchCache cache;
  RingShape rs;
  if (!choose_ring(p.cols, &rs)) return cudaErrorInvalidValue;
  auto kern = quantize_kernel<kMode, kTensor, kFused, kResidual, kNB>;
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  {
    // Too few rows to give every SM a full CTA: spread them over all SMs with smaller CTAs, so
    // each SM runs few warps (fast per row) instead of some SMs running 16 and the rest idling.
    const int64_t sms = sm_count(device);
    const int64_t teams_full = rs.warps / rs.team;
    if ((p.rows + teams_full - 1) / teams_full < sms) {
      const int64_t teams_needed = (p.rows + sms - 1) / sms;
      if (!choose_ring(p.cols, &rs, static_cast<int>(teams_needed * rs.team)))
        return cudaErrorInvalidValue;
    }
  }
  const bool cached_dev = device >= 0 && device < LaunchCache::kDevices;
  if (!cached_dev || cache.attr_set[device].load() == 0) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemLimit));
    if (err != cudaSuccess) return err;
    if (cached_dev) cache.attr_set[device].store(1);
  }
  // Dynamic schedule (fused): one CTA per work unit (a row per team); the hardware starts as many
  // as fit and the running ones take over the rest as they free up.  A launch-shape override (or
  // more units than a grid holds) caps the grid, and each CTA then walks every gridDim.x-th unit
  // from its own.  Static schedule: one wave of resident CTAs.
  const int teams = rs.warps / rs.team;
  int64_t grid = (p.rows + teams - 1) / teams;
  if (!kFused) {
    const long long key = static_cast<long long>(rs.warps) |
                          (static_cast<long long>(rs.stages) << 8) |
                          (static_cast<long long>(rs.slot_bytes) << 16);
    int per_sm = 0;
    if (cached_dev)
      for (auto& e : cache.entries[device])
        if (e.key.load() == key) {
          per_sm = e.per_sm.load();
          break;
        }
    if (per_sm == 0) {
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, rs.warps * 32, rs.smem);
      if (err != cudaSuccess) return err;
      if (per_sm < 1) per_sm = 1;
      if (cached_dev)
        for (auto& e : cache.entries[device]) {
          long long empty = 0;
          if (e.key.load() == key) break;
          if (e.key.compare_exchange_strong(empty, key)) {
            e.per_sm.store(per_sm);
            break;
          }
        }
    }
    const int64_t cap = static_cast<int64_t>(sm_count(device)) * per_sm;
    if (grid > cap) grid = cap;
  }
  const LaunchOverride ov = launch_override();
  if (ov.max_ctas > 0 && grid > ov.max_ctas) grid = ov.max_ctas;
  if (grid > 0x7FFFFFFF) grid = 0x7FFFFFFF;
  if (grid < 1) grid = 1;
  p.stages = rs.stages;
  p.team = rs.team;
  p.blocks_per_warp = rs.blocks_per_warp;
  p.slot_bytes = rs.slot_bytes;
  // Every launch is a programmatic dependent of the previous kernel on the stream, so its set-up
  // overlaps that kernel's tail.  Only a tensor-scale launch right after our amax kernel issues
  // its first row copies before the wait: that grid only reads x, and it started after
  // everything before it on the stream had finished.
  p.prologue_before_wait = (kTensor && after_amax_kernel) ? 1 : 0;
  return launch_programmatic(kern, dim3(static_cast<unsigned>(grid)), dim3(rs.warps * 32),
                             rs.smem, stream, p);
}

// Picks the fixed-trip-count instantiation when the row's blocks split evenly into 4, 7 or 8 per
// lane (widths 2048, 7168, 4096, 8192, 16384, ...).  Quantize-only kernels are issue-bound and
// gain 2-6% from it (measured); the fused round trip (bound by HBM) is unchanged by it and keeps
// the general form; the residual kernel uses it for its third pass only (+1.5%; with it in the
// first two passes as well it measured 3.6% slower).
template <int kMode, bool kTensor, bool kFused, bool kResidual>
cudaError_t launch_nb(QuantParams p, cudaStream_t stream, bool after_amax_kernel = false) {
  if constexpr (!kFused) {  // quantize-only and residual kernels
    RingShape rs;
    if (!choose_ring(p.cols, &rs)) return cudaErrorInvalidValue;
    const int nblk = p.cols / kBlockElems;
    if (rs.blocks_per_warp % 32 == 0 && nblk == rs.team * rs.blocks_per_warp) {
      const bool after = after_amax_kernel;
      switch (rs.blocks_per_warp / 32) {
        case 4: return launch_impl<kMode, kTensor, kFused, kResidual, 4>(p, stream, after);
        case 7: return launch_impl<kMode, kTensor, kFused, kResidual, 7>(p, stream, after);
        case 8: return launch_impl<kMode, kTensor, kFused, kResidual, 8>(p, stream, after);
        default: break;
      }
    }
  }
  return launch_impl<kMode, kTensor, kFused, kResidual, 0>(p, stream, after_amax_kernel);
}

}  // namespace

bool quantize_cols_supported(int64_t cols) {
  RingShape rs;
  return cols > 0 && cols <= kMaxCols && cols % kBlockElems == 0 && choose_ring(cols, &rs);
}

template <int kMode>
cudaError_t launch_mode(bool tensor_scale, bool fused, QuantParams p, cudaStream_t stream,
                        bool after_amax_kernel) {
  if (tensor_scale)
    return fused ? launch_nb<kMode, true, true, false>(p, stream, after_amax_kernel)
                 : launch_nb<kMode, true, false, false>(p, stream, after_amax_kernel);
  return fused ? launch_nb<kMode, false, true, false>(p, stream)
               : launch_nb<kMode, false, false, false>(p, stream);
}

cudaError_t launch_quantize(int mode, bool tensor_scale, bool fused, QuantParams p,
                            cudaStream_t stream, bool after_amax_kernel) {
  switch (mode) {
    case kModeFourOverSix:
      return launch_mode<kModeFourOverSix>(tensor_scale, fused, p, stream, after_amax_kernel);
    case kModeFourOverSixFp16:
      return launch_mode<kModeFourOverSixFp16>(tensor_scale, fused, p, stream, after_amax_kernel);
    default: return launch_mode<kModeSix>(tensor_scale, fused, p, stream, after_amax_kernel);
  }
}

cudaError_t launch_quantize_guided(int mode, const GuidedParams& p, cudaStream_t stream) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  // Rows that split into whole units over 16-byte aligned tensors go through the staged ring.
  const bool ring = p.cols % kGuidedChunk == 0 &&
                    (reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.ref_codes) |
                     reinterpret_cast<uintptr_t>(p.ref_scales)) % 16 == 0;
  if (ring) {
    auto rkern = mode == kModeSix ? guided_ring_kernel<kModeSix>
                                  : guided_ring_kernel<kModeFourOverSix>;
    static std::atomic<int> attr_set[64];
    const bool cached_dev = device >= 0 && device < 64;
    if (!cached_dev || attr_set[device].load() == 0) {
      err = cudaFuncSetAttribute(guided_ring_kernel<kModeSix>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kGuidedSmem));
      if (err == cudaSuccess)
        err = cudaFuncSetAttribute(guided_ring_kernel<kModeFourOverSix>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   static_cast<int>(kGuidedSmem));
      if (err != cudaSuccess) return err;
      if (cached_dev) attr_set[device].store(1);
    }
    const int64_t units = p.rows * (p.cols / kGuidedChunk);
    int64_t grid = (units + kGuidedWarps - 1) / kGuidedWarps;
    const int64_t cap = sm_count(device);
    if (grid > cap) grid = cap;
    const LaunchOverride ov = launch_override();
    if (ov.max_ctas > 0 && grid > ov.max_ctas) grid = ov.max_ctas;
    if (grid < 1) grid = 1;
    return launch_programmatic(rkern, dim3(static_cast<unsigned>(grid)), dim3(kGuidedWarps * 32),
                               kGuidedSmem, stream, p);
  }
  // The guided encoder keeps the rollout's scales: only M (mode six or not) matters.
  auto kern = mode == kModeSix ? guided_kernel<kModeSix> : guided_kernel<kModeFourOverSix>;
  // One wave of resident blocks; the kernel spreads the work units over its warps.
  static std::atomic<int> per_sm_cache[2] = {{0}, {0}};
  std::atomic<int>& cached = per_sm_cache[mode == kModeSix ? 0 : 1];
  int per_sm = cached.load();
  if (per_sm == 0) {
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    cached.store(per_sm);
  }
  const int64_t units = p.rows * ((p.cols / 8 + 32 * kGuidedUnroll - 1) / (32 * kGuidedUnroll));
  int64_t grid = (units + 7) / 8;  // 8 warps per block
  const int64_t cap = static_cast<int64_t>(sm_count(device)) * per_sm;
  if (grid > cap) grid = cap;
  const LaunchOverride ov = launch_override();
  if (ov.max_ctas > 0 && grid > ov.max_ctas) grid = ov.max_ctas;
  if (grid < 1) grid = 1;
  return launch_programmatic(kern, dim3(static_cast<unsigned>(grid)), dim3(256), 0, stream, p);
}

cudaError_t launch_row_amax(const uint16_t* x, int64_t rows, int cols, float* amax,
                            cudaStream_t stream) {
  int device = 0;
  cudaError_t err = cudaGetDevice(&device);
  if (err != cudaSuccess) return err;
  int64_t grid = (rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sm_count(device)) * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  row_amax_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(x, rows, cols, amax);
  return cudaGetLastError();
}

cudaError_t launch_quantize_residual(int mode, QuantParams p, cudaStream_t stream) {
  switch (mode) {
    case kModeFourOverSix: return launch_nb<kModeFourOverSix, false, false, true>(p, stream);
    case kModeFourOverSixFp16:
      return launch_nb<kModeFourOverSixFp16, false, false, true>(p, stream);
    default: return launch_nb<kModeSix, false, false, true>(p, stream);
  }
}

}  // namespace nvfp4
