// nvfp4_gemm.cu -- the consumer side of the quantizer: the MMA-ready block-scale layout and an
// NVFP4 x NVFP4 GEMM for the forward y = x . Q(w) ("NVFP4 RL" blog, Sec. 3: the forward executed
// is y = x . Q(w); Sec. 2: activations carry a per-token FP32 scale).
//
// Block-scaled tensor-core products read E4M3 block scales in tiles of 128 rows x 4 scale
// columns (512 bytes each, tiles row-major over [ceil(rows/128)][ceil(cols/64)]): inside a tile
// the scale of (row r, scale column c) sits at byte (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4),
// so the 16-byte line r % 32 holds the four scales of rows r % 32, +32, +64 and +96.  The
// quantizer writes scales row-major; nvfp4_swizzle_block_scales re-lays them (zero padding).
//
// nvfp4_gemm_nt is one hand-written tcgen05 kernel.  A persistent grid (one CTA per SM) walks the
// 128 x 256 output tiles (128 rows of x, 256 rows of w); per CTA:
//   warp 0      (one thread) TMA: per stage the 128-byte (256 FP4 values) K slab of the tile's
//               128 rows of x and 256 rows of w (128-byte swizzle, cp.async.bulk.tensor) and the
//               stage's 512-byte scale tiles (cp.async.bulk), into a 4-stage shared-memory ring
//               completing on mbarriers;
//   warps 10-13 write each stage's scale tiles into a TMEM slot with tcgen05.st (every lane
//               quarter holds a whole tile, the layout the block-scaled product reads);
//   warp 1      owns the tensor memory (TMEM); one thread issues the block-scaled FP4 products
//               (tcgen05.mma kind::mxf4nvf4, scale_vec::4X: E2M1 x E2M1 with one UE4M3 scale per
//               16 values along K, M = 128, N = 256, K = 64, FP32 accumulation in TMEM), releases
//               each stage with tcgen05.commit and hands the finished accumulator over;
//   warps 2-9   epilogue: warp w reads TMEM lanes 32*(w % 4) .. +31 (its 32 rows) and 128 of the
//               256 accumulator columns with tcgen05.ld, forms
//               y[m][n] = bf16(fp32(fp32(D[m][n] * S_x[m]) * S_w)) in registers, hands the
//               accumulator back (the next tile's products start), then writes y straight to
//               global memory.
// Measured on GB300 (16384 x 2048 x 7168): consecutive products into one accumulator run about
// 250 cycles apart whatever N is, so each product takes the widest N (256) the accumulator and
// the scale slots leave room for in TMEM (512 columns); products into independent accumulators
// overlap, but two 256-column accumulators leave no columns for the scales.  Scale copies issued
// by the product thread (tcgen05.cp) wait in the same in-order pipe as the products (measured
// 286 -> 164 us without them), hence the separate scale warps.
// Every mbarrier wait is bounded; a wait that runs out records NVFP4_ERR_TIMEOUT, tells the other
// roles to stop, and the CTA waits for its own copies and products in flight and frees its TMEM
// before it returns.
#include <atomic>
#include <cstdint>
#include <cuda.h>          // CUtensorMap and its enums; the encoder is looked up at run time
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "nvfp4.h"
#include "nvfp4_internal.h"

namespace {

using nvfp4::global_ns;
using nvfp4::mbar_try_wait;
using nvfp4::smem_addr;

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

// ------------------------------------------------------------------------------------------------
// The tcgen05 block-scaled FP4 GEMM
// ------------------------------------------------------------------------------------------------

constexpr int kTileM = 128;                // output rows per tile (x rows)
constexpr int kTileN = 256;                // output columns per tile (w rows)
constexpr int kHalfN = kTileN / 2;         // columns one epilogue warp drains
constexpr int kStageK = 256;               // FP4 values along K per stage (128 bytes per row)
constexpr int kMmaK = 64;                  // K of one kind::mxf4nvf4 instruction
constexpr int kSteps = kStageK / kMmaK;    // products per chain per stage
constexpr int kStages = 4;
constexpr int kSlabA = kTileM * (kStageK / 2);          // 16 KB of x codes per stage
constexpr int kSlabB = kTileN * (kStageK / 2);          // 32 KB of w codes per stage
constexpr int kSfTileBytes = 512;                       // 128 rows x 4 scales
constexpr int kSfA = kSteps * kSfTileBytes;             // 2 KB of x scales per stage
constexpr int kSfB = 2 * kSteps * kSfTileBytes;         // 4 KB of w scales per stage
constexpr int kSfColsA = kSteps * 4;                    // TMEM columns of x's scales per stage
constexpr int kSfColsB = kSteps * 8;                    // TMEM columns of w's scales per stage
constexpr int kSfColsPerStage = kSfColsA + kSfColsB;    // 48
constexpr int kTmemCols = 512;             // accumulators (256) + the scale ring (192)
constexpr int kEpiWarps = 8;               // two per TMEM lane quarter, one per 128 columns
constexpr int kSfWarps = 4;                // one per TMEM lane quarter
constexpr int kFirstEpiWarp = 2;
constexpr int kFirstSfWarp = kFirstEpiWarp + kEpiWarps;
constexpr int kGemmThreads = (kFirstSfWarp + kSfWarps) * 32;
constexpr int kBarrierCount = 3 * kStages + 3;
constexpr size_t kGemmSmem = 1024 /* alignment slack */ +
                             kStages * (kSlabA + kSlabB + kSfA + kSfB) + kBarrierCount * 8 + 16;
static_assert(kTileN + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
static_assert(kGemmSmem <= 227 * 1024, "shared-memory budget");

// Instruction descriptor of tcgen05.mma kind::mxf4nvf4: A and B both E2M1 (type code 1, bits
// 7-9 and 10-12), both K-major (bits 15, 16 = 0), N >> 3 in bits 17-22, UE4M3 scales (bit 23 = 0),
// M >> 4 in bits 24-28, scale-factor ids 0, dense.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (static_cast<uint32_t>(kTileN >> 3) << 17) |
                            (static_cast<uint32_t>(kTileM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand slab with 128-byte swizzle: start address
// >> 4 (bits 0-13), leading byte offset 16 (unused for swizzled K-major; bits 16-29), stride byte
// offset 1024 = 8 rows of 128 bytes (bits 32-45), the fixed 0b001 of bits 46-48, swizzle mode 2
// = 128-byte (bits 61-63).  Slabs are 1024-byte aligned; a K step of 64 values advances the start
// address by 32 bytes inside the swizzle row.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(holder)),
               "r"(cols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The mbarrier receives one arrival once every tcgen05 operation this thread issued before has
// completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// D (+)= (A . scale_A) x (B . scale_B)^T for one K step of 64 FP4 values.
__device__ __forceinline__ void tc_mma_nvfp4(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa,
                                             uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

// 32 consecutive FP32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_load_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_store16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_store_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 2-D tiled TMA load (x = byte offset along the row, y = row) completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

struct GemmParams {
  const uint8_t* sfa;   // swizzled x scales
  const uint8_t* sfb;   // swizzled w scales
  const float* sx;      // x row scales [m]
  const float* sw;      // w tensor scale [1]
  uint16_t* y;          // BF16 [m][n]
  int m, n, k;
  int tiles_n;          // ceil(n / 256)
  int tiles;            // ceil(m / 128) * tiles_n
  int w_row_tiles;      // ceil(n / 128): 128-row bands of w's scales
  int kstages;          // ceil(k / 256)
  int sf_tiles_c;       // k / 64: scale tiles per 128-row band
  int* status;
  uint64_t timeout_ns;
};

// Waits for the barrier phase of the given parity; gives up when another role has stopped the
// CTA (abort flag) or after timeout_ns (then it records the timeout and stops the others).
// Roles whose events are far apart poll with a pause of sleep_ns between rounds, which leaves
// the issue slots and shared-memory port to the roles on the critical path (measured: 4% faster).
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                           volatile int* abort_flag, int* status,
                                           int sleep_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t start = global_ns();
  while (true) {
    for (int i = 0; i < 4; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (sleep_ns > 0) __nanosleep(sleep_ns);
    if (*abort_flag) return false;
    if (global_ns() - start > timeout_ns) {
      *abort_flag = 1;
      nvfp4::record_status(status, nvfp4::kStatusTimeout);
      return false;
    }
  }
}

// The same, for a whole warp: lane 0 waits and the warp follows its answer, so warp-wide
// tcgen05 instructions after it run on all 32 lanes or on none.
__device__ __forceinline__ bool warp_wait_phase(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                                volatile int* abort_flag, int* status, int lane,
                                                int sleep_ns = 0) {
  int ok = 0;
  if (lane == 0) ok = wait_phase(bar, parity, timeout_ns, abort_flag, status, sleep_ns) ? 1 : 0;
  return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// Number of the tile's two 128-row bands of w that exist (the last tile may have one; the other's
// rows are zero-filled by TMA and its scales are never read for a stored output).
__device__ __forceinline__ int live_halves(const GemmParams& p, int nt) {
  return min(2, p.w_row_tiles - 2 * nt);
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_b, const GemmParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* slab_a = smem;                                  // [kStages][16 KB]
  unsigned char* slab_b = slab_a + kStages * kSlabA;             // [kStages][32 KB]
  unsigned char* sf_a = slab_b + kStages * kSlabB;               // [kStages][2 KB]
  unsigned char* sf_b = sf_a + kStages * kSfA;                   // [kStages][2][2 KB]
  uint64_t* full = reinterpret_cast<uint64_t*>(sf_b + kStages * kSfB);
  uint64_t* empty = full + kStages;
  uint64_t* sf_ready = empty + kStages;
  uint64_t* acc_full = sf_ready + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* done = acc_empty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      nvfp4::mbar_init(&full[s], 1);
      nvfp4::mbar_init(&empty[s], 1);
      nvfp4::mbar_init(&sf_ready[s], kSfWarps);
    }
    nvfp4::mbar_init(acc_full, 1);
    nvfp4::mbar_init(acc_empty, kEpiWarps);
    nvfp4::mbar_init(done, 1);
    *abort_flag = 0;
    nvfp4::fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t sf_tmem = tmem + kTileN;  // the scale ring
  const uint64_t tmo = p.timeout_ns;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
      int g = 0;  // stages issued
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
        const int mt = tile / p.tiles_n, nt = tile - (tile / p.tiles_n) * p.tiles_n;
        const int hv = live_halves(p, nt);
        for (int ks = 0; ks < p.kstages; ++ks, ++g) {
          const int s = g % kStages;
          if (!wait_phase(&empty[s], ((g / kStages) & 1) ^ 1, tmo, abort_flag, p.status, 64)) {
            ok = false;
            break;
          }
          const int nk = min(kSteps, (p.k - ks * kStageK) / kMmaK);
          const uint32_t sf_bytes = static_cast<uint32_t>(nk) * kSfTileBytes;
          nvfp4::mbar_arrive_expect_tx(&full[s], kSlabA + kSlabB + (1u + hv) * sf_bytes);
          tma_load_2d(slab_a + s * kSlabA, &map_a, ks * (kStageK / 2), mt * kTileM, &full[s]);
          tma_load_2d(slab_b + s * kSlabB, &map_b, ks * (kStageK / 2), nt * kTileN, &full[s]);
          const int64_t tc = static_cast<int64_t>(ks) * kSteps;
          bulk_copy(sf_a + s * kSfA,
                    p.sfa + (static_cast<int64_t>(mt) * p.sf_tiles_c + tc) * kSfTileBytes,
                    sf_bytes, &full[s]);
          for (int h = 0; h < hv; ++h)
            bulk_copy(sf_b + s * kSfB + h * (kSfB / 2),
                      p.sfb + (static_cast<int64_t>(2 * nt + h) * p.sf_tiles_c + tc) * kSfTileBytes,
                      sf_bytes, &full[s]);
        }
      }
      // Whatever happened, the copies issued land before the CTA goes: wait for the last phase
      // each stage was filled for.
      for (int s = 0; s < kStages; ++s) {
        const int n_s = g > s ? (g - s + kStages - 1) / kStages : 0;
        if (n_s > 0)
          (void)nvfp4::mbar_wait_bounded(&full[s], static_cast<uint32_t>((n_s - 1) & 1), tmo);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issue: one 128 x 256 accumulation chain per tile ----
      int g = 0, it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x, ++it) {
        if (!wait_phase(acc_empty, (it & 1) ^ 1, tmo, abort_flag, p.status)) break;
        tc_fence_after();
        for (int ks = 0; ks < p.kstages; ++ks, ++g) {
          const int s = g % kStages;
          const uint32_t par = (g / kStages) & 1;
          if (!wait_phase(&full[s], par, tmo, abort_flag, p.status) ||
              !wait_phase(&sf_ready[s], par, tmo, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nk = min(kSteps, (p.k - ks * kStageK) / kMmaK);
          const uint32_t sf = sf_tmem + static_cast<uint32_t>(s * kSfColsPerStage);
          const uint32_t a0 = smem_addr(slab_a + s * kSlabA);
          const uint32_t b0 = smem_addr(slab_b + s * kSlabB);
          for (int kk = 0; kk < nk; ++kk)
            tc_mma_nvfp4(tmem, desc_sw128(a0 + kk * (kMmaK / 2)), desc_sw128(b0 + kk * (kMmaK / 2)),
                         sf + kk * 4, sf + kSfColsA + kk * 8, (ks | kk) != 0 ? 1u : 0u);
          tc_commit(&empty[s]);  // the stage (and its scale slot) is free once these are done
        }
        if (!ok) break;
        tc_commit(acc_full);  // the accumulators are complete once every product is done
      }
      // Every product issued has finished before the TMEM is freed.
      tc_commit(done);
      (void)nvfp4::mbar_wait_bounded(done, 0, tmo);
    }
  } else if (warp < kFirstSfWarp) {
    // ---- epilogue: warp w reads TMEM lanes 32*(w % 4) .. +31 (its 32 rows of the tile) and
    // accumulator columns half * 128 .. +127, half = (w - 2) / 4 ----
    const int quarter = warp & 3;
    const int half = (warp - kFirstEpiWarp) / 4;
    const int r_in_tile = quarter * 32 + lane;
    const float sw = p.sw[0];
    int it = 0;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++it) {
      if (!warp_wait_phase(acc_full, it & 1, tmo, abort_flag, p.status, lane, 1000)) break;
      tc_fence_after();
      const int mt = tile / p.tiles_n, nt = tile - (tile / p.tiles_n) * p.tiles_n;
      const int row = mt * kTileM + r_in_tile;
      const bool live = row < p.m;
      const float sx = live ? p.sx[row] : 0.0f;
      uint16_t* yrow = p.y + static_cast<int64_t>(live ? row : 0) * p.n;
      const uint32_t t0 = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                          static_cast<uint32_t>(half * kHalfN);
      // Drain this warp's 128 accumulator columns into registers as BF16 pairs first, release the
      // accumulator (the next tile's products start), then store.
      uint32_t packed[kHalfN / 2];
#pragma unroll
      for (int c = 0; c < kHalfN; c += 32) {
        uint32_t v[32];
        tmem_load32(t0 + c, v);
        tmem_load_wait();
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float lo = __fmul_rn(__fmul_rn(__uint_as_float(v[2 * q]), sx), sw);
          const float hi = __fmul_rn(__fmul_rn(__uint_as_float(v[2 * q + 1]), sx), sw);
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(packed[c / 2 + q]) : "f"(hi), "f"(lo));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      const int col0 = nt * kTileN + half * kHalfN;
      if (live) {
#pragma unroll
        for (int g8 = 0; g8 < kHalfN / 8; ++g8) {
          if (col0 + 8 * g8 >= p.n) break;
          *reinterpret_cast<uint4*>(yrow + col0 + 8 * g8) =
              make_uint4(packed[4 * g8], packed[4 * g8 + 1], packed[4 * g8 + 2], packed[4 * g8 + 3]);
        }
      }
    }
  } else {
    // ---- scales into TMEM: warp w fills lanes 32*(w % 4) .. +31 of the stage's scale slot.
    // Lane r takes line r (16 bytes) of each 512-byte scale tile -- the four scales of rows r,
    // r+32, r+64 and r+96 -- into four consecutive columns: every lane quarter holds the whole
    // tile, and the product reads row m's scales at lane m % 128, column (tile's first column +
    // m / 32).  x: K step t's tile at columns 4t.  w (256 rows = two 128-row bands): K step t's
    // tiles at columns 8t (band 0) and 8t + 4 (band 1), so row n of w is read at column 8t + n/32.
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int g = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < p.tiles; tile += gridDim.x) {
      const int hv = live_halves(p, tile - (tile / p.tiles_n) * p.tiles_n);
      for (int ks = 0; ks < p.kstages; ++ks, ++g) {
        const int s = g % kStages;
        if (!warp_wait_phase(&full[s], (g / kStages) & 1, tmo, abort_flag, p.status, lane, 128)) {
          ok = false;
          break;
        }
        const int nk = min(kSteps, (p.k - ks * kStageK) / kMmaK);
        const uint32_t slot = sf_tmem + lane_base + static_cast<uint32_t>(s * kSfColsPerStage);
        uint32_t va[16];
        uint32_t vb[32];
#pragma unroll
        for (int t = 0; t < kSteps; ++t) {
          uint4 la = make_uint4(0, 0, 0, 0), lb0 = la, lb1 = la;
          if (t < nk) {
            la = *reinterpret_cast<const uint4*>(sf_a + s * kSfA + t * kSfTileBytes + lane * 16);
            lb0 = *reinterpret_cast<const uint4*>(sf_b + s * kSfB + t * kSfTileBytes + lane * 16);
            if (hv > 1)
              lb1 = *reinterpret_cast<const uint4*>(sf_b + s * kSfB + kSfB / 2 +
                                                     t * kSfTileBytes + lane * 16);
          }
          va[4 * t] = la.x; va[4 * t + 1] = la.y; va[4 * t + 2] = la.z; va[4 * t + 3] = la.w;
          vb[8 * t] = lb0.x; vb[8 * t + 1] = lb0.y; vb[8 * t + 2] = lb0.z; vb[8 * t + 3] = lb0.w;
          vb[8 * t + 4] = lb1.x; vb[8 * t + 5] = lb1.y; vb[8 * t + 6] = lb1.z;
          vb[8 * t + 7] = lb1.w;
        }
        tmem_store16(slot, va);
        tmem_store32(slot + kSfColsA, vb);
        tmem_store_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sf_ready[s]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// The driver's tensor-map encoder, looked up once through the runtime (no link-time dependency
// on the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load();
  if (f == nullptr) {
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || f == nullptr)
      return nullptr;
    fn.store(f);
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// Tensor map of packed E2M1 codes [rows][k/2] bytes: boxes of 128 bytes x box_rows rows, 128-byte
// swizzle, zero fill past the edges.
bool encode_codes_map(CUtensorMap* map, const uint8_t* codes, int64_t rows, int64_t k,
                      uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(k / 2), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(k / 2)};
  const cuuint32_t box[2] = {kStageK / 2, box_rows};
  const cuuint32_t elem_strides[2] = {1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides,
                box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  (void)m;
  (void)n;
  return 0;  // the product needs no scratch memory
}

extern "C" nvfp4_status nvfp4_gemm_nt(const uint8_t* x_codes, const uint8_t* x_scales_swizzled,
                                      const float* x_row_scale, const uint8_t* w_codes,
                                      const uint8_t* w_scales_swizzled, const float* w_tensor_scale,
                                      int64_t m, int64_t n, int64_t k, void* y, void* workspace,
                                      size_t workspace_bytes, nvfp4_stream_t stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (m < 0 || n < 0 || k < 0) return NVFP4_ERR_INVALID_ARG;
  if (k == 0 || k % 64 != 0 || n % 16 != 0) return NVFP4_ERR_SHAPE;
  if (m > (int64_t{1} << 31) - kTileM || n > (int64_t{1} << 31) - kTileN ||
      k > (int64_t{1} << 31) - kStageK)
    return NVFP4_ERR_SHAPE;
  if (m == 0 || n == 0) return NVFP4_OK;
  if (!x_codes || !x_scales_swizzled || !x_row_scale || !w_codes || !w_scales_swizzled ||
      !w_tensor_scale || !y)
    return NVFP4_ERR_INVALID_ARG;
  if (!aligned(x_codes, 256) || !aligned(w_codes, 256) || !aligned(x_scales_swizzled, 256) ||
      !aligned(w_scales_swizzled, 256) || !aligned(y, 16) || !aligned(x_row_scale, 4) ||
      !aligned(w_tensor_scale, 4))
    return NVFP4_ERR_ALIGNMENT;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return NVFP4_ERR_CUDA;
  int* status = nullptr;
  if (nvfp4::device_status_word(&status) != cudaSuccess) return NVFP4_ERR_CUDA;
  CUtensorMap map_a, map_b;
  if (!encode_codes_map(&map_a, x_codes, m, k, kTileM) ||
      !encode_codes_map(&map_b, w_codes, n, k, kTileN))
    return NVFP4_ERR_CUDA;
  static std::atomic<int> attr_set[64];
  if (device < 0 || device >= 64 || attr_set[device].load() == 0) {
    if (cudaFuncSetAttribute(gemm_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemmSmem)) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    if (device >= 0 && device < 64) attr_set[device].store(1);
  }
  GemmParams p{};
  p.sfa = x_scales_swizzled;
  p.sfb = w_scales_swizzled;
  p.sx = x_row_scale;
  p.sw = w_tensor_scale;
  p.y = static_cast<uint16_t*>(y);
  p.m = static_cast<int>(m);
  p.n = static_cast<int>(n);
  p.k = static_cast<int>(k);
  p.tiles_n = static_cast<int>((n + kTileN - 1) / kTileN);
  p.tiles = static_cast<int>((m + kTileM - 1) / kTileM) * p.tiles_n;
  p.w_row_tiles = static_cast<int>((n + 127) / 128);
  p.kstages = static_cast<int>((k + kStageK - 1) / kStageK);
  p.sf_tiles_c = static_cast<int>(k / 64);
  p.status = status;
  p.timeout_ns = nvfp4::kWaitTimeoutNs;
  int grid = nvfp4::sm_count(device);
  if (grid > p.tiles) grid = p.tiles;
  gemm_nvfp4_kernel<<<grid, kGemmThreads, kGemmSmem, reinterpret_cast<cudaStream_t>(stream)>>>(
      map_a, map_b, p);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}
