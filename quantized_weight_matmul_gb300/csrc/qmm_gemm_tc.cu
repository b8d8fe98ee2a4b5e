// qmm_gemm_tc.cu -- MMQ on the sm_103a tensor cores (tcgen05, TMEM, TMA).
//
// What it computes ("llama.cpp MMQ", sec. 4-6; "The quantized GEMM",
// "The GPU path"):
//   Q4_K: out[t][r] = sum_b sum_j ( d_b*sc_j*dx_tj*D_trj - dmin_b*m_j*s_tj ),
//         D = sum over the 32 values of sub-block j of nibble * q
//   Q6_K: out[t][r] = sum_b sum_g d_b*sc_g*dx_t(g/2)*D_trg,
//         D = sum over the 16 values of group g of (q6 - 32) * q
//
// GB300 design.  tcgen05 has no int8 kind on sm_103a and the legacy int8
// warp MMA is slow, so the integer dots run on the f16 kind with operands
// that are small integers f16 holds exactly; the f32 accumulation of one
// 32-value block stays below 2^24 in magnitude, so TMEM holds the exact
// integer sum.  The weight operand carries its integer group scale:
//   Q4_K  sc_j * nibble (<= 945);
//   Q6_K  sc_g * (q - 32) split exactly into two operands, hi = sgn*16*(|sc|>>4)
//         *(q-32) and lo = sgn*(|sc|&15)*(q-32), both dotted with the same
//         activation codes and accumulated into the same sum, so one
//         accumulator holds sum_g sc_g*D_g of a whole 32-value block.
// One accumulator per 32-value block is then rescaled once per output in
// fp32 by the token's dx (and the row's d, factored out of the running sum).
//
// One CTA computes a 128-row x BN-token tile with 16 warps:
//   warp 0      TMA producer: raw weight super-blocks (128 rows x 144 B, or
//               240 B windows around the 2-byte-aligned 210-byte Q6_K
//               blocks), the f16 activation tile (BN x 64 k, 128-byte
//               swizzle) with the token-contiguous dx rows of the same 64 k,
//               and for Q4_K the three bf16 parts of s of each super-block.
//   warp 1      TMEM allocation and the single MMA-issuing thread: per
//               32-value block an MMA chain into one of NBUF accumulators of
//               BN columns, committed to an mbarrier; Q4_K's min term
//               sum_j m_j*s_tj of each super-block is one more entry of the
//               same accumulator ring (bf16 operands, exact products).
//   warps 4-7   unpack, one TMEM lane quarter each, one weight row per
//               thread: raw codes -> the f16 weight operand of a 64-k stage,
//               written straight into TMEM (tcgen05.st), where the MMA reads
//               it as its A operand -- the operand never touches shared
//               memory, whose bandwidth the MMAs' activation reads need.
//               The 64-token Q6_K tile has eight (warps 4-11), two per lane
//               quarter, each unpacking one 32-value block of every stage.
//   8 warps     epilogue (warps 8-15, or 12-19), two per lane quarter
//               (BN/2 token columns each):
//               per accumulator the TMEM loads of its columns, the
//               accumulator handed back after the last of them, the fp32
//               rescale into register accumulators; one store at the end.
// Stages that a role reads with ordinary loads and the producer refills with
// TMA (raw weights, the dx rows) go back through release_stage, which fences
// the reads against the async-proxy refill.  Every wait is bounded: a wait
// that runs past its deadline raises the CTA's abort flag and QMM_ETIMEOUT in
// the status word, all roles leave their loops, in-flight copies and MMAs
// are drained, and TMEM is freed.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kQ4 = 0, kQ6 = 1;

template <int QT, int BN>
struct Cfg {
  static constexpr int BM = 128;                // weight rows per CTA = TMEM lanes
  static constexpr int KS = 64;                 // k per operand stage
  // first unpack warp; epilogue warps per TMEM lane quarter, all epilogue
  // warps, the first of them
  // Q6_K's unpack (two operands per code, realigned 2-byte blocks) costs
  // several times Q4_K's, so the 64-token Q6_K tile, whose epilogue is light,
  // gets two unpack warps per lane quarter, one per 32-value block of a stage
  static constexpr int UW = (QT == kQ6 && BN == 64) ? 8 : 4;  // unpack warps
  static constexpr int U0 = 4, EPQ = 2, NE = 4 * EPQ, E0 = U0 + UW;
  static constexpr int THREADS = 32 * (E0 + NE);
  static constexpr int CPW = BN / EPQ;  // token columns per epilogue warp
  static_assert(CPW % 32 == 0, "whole 32-column TMEM loads");
  // register budgets per warpgroup: producers / MMA (warps 0-3), unpack
  // (U0 .. E0-1), epilogue (E0 ..).  The block is launched with 65536 /
  // THREADS per thread, rounded down to a multiple of 8 (128 for 512
  // threads, 96 for 640); the budgets add up to no more than that.
  static constexpr uint32_t REG_LAUNCH = (65536 / THREADS) & ~7u;
  static constexpr uint32_t REG_CTL = 56, REG_UNPACK = THREADS == 512 ? 96 : 80;
  static constexpr uint32_t REG_EPI =
      ((REG_LAUNCH * THREADS - 128 * REG_CTL - 32 * UW * REG_UNPACK) / (32 * NE)) & ~7u;
  static_assert(128 * REG_CTL + 32 * UW * REG_UNPACK + 32 * NE * REG_EPI <= REG_LAUNCH * THREADS, "register split");
  static_assert(REG_EPI >= REG_LAUNCH, "the epilogue gains registers");
  // ring depths: raw weight super-blocks, activation stages, dx stages,
  // operand stages in TMEM.  The activation ring is as deep as shared memory
  // allows: its stages are released by the MMAs alone, so all of them are
  // prefetch depth against the TMA latency.
  static constexpr int RS = (QT == kQ6 && BN == 64) ? 4 : 3;
  static constexpr int BS = BN == 128 ? 6 : 8;
  static constexpr int DS = 8, AS = 4;
  // raw bytes per row and super-block in shared memory (Q6_K: a window around
  // the 2-byte-aligned 210-byte block; 240 rather than 224 bytes, so that a
  // warp's 32-bit loads of 32 rows hit 8 bank offsets instead of 4)
  static constexpr int RAW_ROW = QT == kQ4 ? 144 : 240;
  static constexpr int BLK = QT == kQ4 ? kQ4KBytes : kQ6KBytes;
  static constexpr int RAW_BYTES = BM * RAW_ROW;
  static constexpr bool MINT = QT == kQ4;                // Q4_K min term
  static constexpr int MINB_BYTES = MINT ? BN * 64 : 0;  // 4 chunks x BN tokens x 8 bf16
  static constexpr int AMIN_BYTES = MINT ? BM * 64 : 0;  // 4 chunks x BM rows x 8 bf16
  static constexpr int B_BYTES = BN * KS * 2;
  static constexpr int SC_BYTES = 2 * BN * 4;  // dx of a stage's two 32-value blocks
  // TMEM: NBUF accumulators of BN columns, then AS operand stages of ACOLS
  // columns (Q4_K: 32, the codes of 64 k; Q6_K: 64, the hi and lo operands of
  // two 32-value blocks).  A barrier hop costs ~150 cycles and an MMA's
  // completion is seen ~250 cycles after its work, so both rings need depth:
  // four operand stages, and accumulators for 256-512 cycles of tensor work
  // (a Q6_K block, with its hi and lo operands, is twice a Q4_K block's).
  static constexpr int ACOLS = QT == kQ4 ? 32 : 64;
  static constexpr int NBUF = (512 - AS * ACOLS) / BN;
  // Q6_K with the 64-token tile: the two 32-value blocks of a stage share one
  // accumulator pair, one commit and one release (NBUF / 2 pairs), so each
  // MMA -> epilogue -> MMA round trip carries a whole stage
  static constexpr bool PAIRED = QT == kQ6 && BN == 64;
  static constexpr int A_COL0 = NBUF * BN;
  static_assert(NBUF >= 2 && NBUF <= 8, "accumulator ring");
  static_assert(A_COL0 % 16 == 0 && ACOLS % 16 == 0, "TMEM column alignment");
  static constexpr int RAW_OFF = 0;
  static constexpr int B_OFF = RAW_OFF + RS * RAW_BYTES;
  static constexpr int MINB_OFF = B_OFF + BS * B_BYTES;
  // Q4_K: the min term's weight operand m[r][j] (bf16, canonical K-major),
  // one per raw stage: written by the unpack warps, read by the min MMA
  static constexpr int AMIN_OFF = MINB_OFF + RS * MINB_BYTES;
  static constexpr int SC_OFF = AMIN_OFF + RS * AMIN_BYTES;
  static constexpr int BAR_OFF = SC_OFF + DS * SC_BYTES;
  // barriers: raw full/empty, b full/empty, dx full/empty, a full/empty,
  // acc full/empty, done
  static constexpr int NBARS = 2 * RS + 2 * BS + 2 * DS + 2 * AS + 2 * NBUF + 1;
  static_assert(BAR_OFF + NBARS * 8 + 16 + 1024 <= 227 * 1024, "shared memory");
  static constexpr int SMEM = BAR_OFF + NBARS * 8 + 16 + 1024;  // + slack for 1 KB alignment
  static_assert(RAW_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "128-byte swizzle needs 1 KB aligned stages");
  static_assert(SC_BYTES % 16 == 0 && MINB_BYTES % 16 == 0, "bulk copy alignment");
};

template <int QT, int BN>
struct Bars {
  using C = Cfg<QT, BN>;
  uint32_t base;
  __device__ uint32_t raw_full(int i) const { return base + 8 * i; }
  __device__ uint32_t raw_empty(int i) const { return base + 8 * (C::RS + i); }
  __device__ uint32_t b_full(int i) const { return base + 8 * (2 * C::RS + i); }
  __device__ uint32_t b_empty(int i) const { return base + 8 * (2 * C::RS + C::BS + i); }
  static constexpr int X0 = 2 * C::RS + 2 * C::BS;  // after the raw and activation rings
  __device__ uint32_t dx_full(int i) const { return base + 8 * (X0 + i); }
  __device__ uint32_t dx_empty(int i) const { return base + 8 * (X0 + C::DS + i); }
  static constexpr int A0 = X0 + 2 * C::DS;
  __device__ uint32_t a_full(int i) const { return base + 8 * (A0 + i); }
  __device__ uint32_t a_empty(int i) const { return base + 8 * (A0 + C::AS + i); }
  __device__ uint32_t acc_full(int i) const { return base + 8 * (A0 + 2 * C::AS + i); }
  __device__ uint32_t acc_empty(int i) const { return base + 8 * (A0 + 2 * C::AS + C::NBUF + i); }
  __device__ uint32_t done() const { return base + 8 * (A0 + 2 * C::AS + 2 * C::NBUF); }
};

// Wait used while draining: ignores the abort flag, gives up at `deadline`.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t deadline) {
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 63u && global_ns() > deadline) return;
  }
}

// Bounded wait of one thread.  (Waits that park the thread with a suspend
// hint were measured 3-8 % slower here than polling try_wait.)
__device__ __forceinline__ bool gwait(uint32_t bar, uint32_t parity, const Guard& g) {
  return wait_bar(bar, parity, g);
}

// Warp-uniform bounded wait: every lane waits, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Guard& g) {
  const bool ok = gwait(bar, parity, g);
  return __all_sync(0xffffffffu, ok);
}

// f16x2 of (1024 + a, 1024 + b) for two codes held in bits 0-5 and 16-21.
__device__ __forceinline__ uint32_t magic_pair(uint32_t two_codes, uint32_t mask) {
  return and_or(two_codes, mask, 0x64006400u);
}

__device__ __forceinline__ uint32_t f16x2_of(float v) {
  const __half2 h = __float2half2_rn(v);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---------------------------------------------------------------- unpack --
// Q4_K: stage p of one row (qs bytes 32p..32p+31, i.e. sub-blocks 2p and
// 2p+1) -> 32 TMEM columns of f16 pairs in k order: column c holds k = 2c and
// 2c+1; the low nibbles are k 0..31, the high ones k 32..63.  Each value is
// sc * nibble (an exact f16 integer <= 945), the 1024-magic conversion with
// the scale folded into the FMA: (1024 + n) * sc - 1024 * sc.
__device__ __forceinline__ void unpack_q4k_stage(uint4 q0, uint4 q1, uint32_t sc2, bool d_zero,
                                                 uint32_t (&a)[32]) {
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  const float sl = d_zero ? 0.0f : (float)(sc2 & 0xFFu), sh = d_zero ? 0.0f : (float)(sc2 >> 8);
  const uint32_t mul_lo = f16x2_of(sl), off_lo = f16x2_of(-1024.0f * sl);
  const uint32_t mul_hi = f16x2_of(sh), off_hi = f16x2_of(-1024.0f * sh);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t t01 = prmt(w[i], 0u, 0x4140u), t23 = prmt(w[i], 0u, 0x4342u);
    a[2 * i] = hfma2_bits(magic_pair(t01, 0x000F000Fu), mul_lo, off_lo);
    a[2 * i + 1] = hfma2_bits(magic_pair(t23, 0x000F000Fu), mul_lo, off_lo);
    a[16 + 2 * i] = hfma2_bits(magic_pair(t01 >> 4, 0x000F000Fu), mul_hi, off_hi);
    a[16 + 2 * i + 1] = hfma2_bits(magic_pair(t23 >> 4, 0x000F000Fu), mul_hi, off_hi);
  }
}

// Q6_K: one 32-value block of stage s of one row -> 32 TMEM columns: the hi
// and lo operands of its two 16-value groups, [hi g0 | lo g0 | hi g1 | lo g1],
// 8 columns (16 k) each.  Stage s holds elements 64s..64s+63 of the
// super-block: half n = s/2, quads 2(s%2) and 2(s%2)+1 (block `blk` = quad
// 2(s%2)+blk).  Element 128n + 32*quad + l takes its low 4 bits from
// ql[64n + l] (quads 0, 2) or ql[64n + 32 + l] (quads 1, 3) -- the low nibble
// for quads 0-1, the high one for quads 2-3 -- and its top 2 bits from bits
// 2*quad..2*quad+1 of qh[32n + l].  L: the 8 ql words of this quad's l range,
// H: the 8 qh words of the half; mh / ml: f16x2 multipliers of the two groups.
__device__ __forceinline__ void unpack_q6k_block(const uint32_t (&L)[8], const uint32_t (&H)[8], int s, int blk,
                                                 const uint32_t (&mh)[2], const uint32_t (&ml)[2],
                                                 uint32_t (&a)[32]) {
  const uint32_t upper = (uint32_t)(s & 1);
  const uint32_t quad = 2u * upper + (uint32_t)blk;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int g = w >> 2;  // group of values l = 4w..4w+3
    const uint32_t codes = ((L[w] >> (4u * upper)) & 0x0F0F0F0Fu) | (((H[w] >> (2u * quad)) << 4) & 0x30303030u);
    const uint32_t t01 = prmt(codes, 0u, 0x4140u), t23 = prmt(codes, 0u, 0x4342u);
    // (q - 32) as f16: (1024 + q) - 1056
    const uint32_t v01 = hfma2_bits(magic_pair(t01, 0x003F003Fu), 0x3C003C00u, 0xE420E420u);
    const uint32_t v23 = hfma2_bits(magic_pair(t23, 0x003F003Fu), 0x3C003C00u, 0xE420E420u);
    const int c = 16 * g + 2 * (w & 3);
    a[c] = hmul2_bits(v01, mh[g]);
    a[c + 1] = hmul2_bits(v23, mh[g]);
    a[c + 8] = hmul2_bits(v01, ml[g]);
    a[c + 9] = hmul2_bits(v23, ml[g]);
  }
}

// The exact split of a signed int8 group scale into the two f16 operand
// multipliers: hi = sgn * 16 * (|sc| >> 4), lo = sgn * (|sc| & 15), so that
// hi + lo = sc and every product with q - 32 in [-32, 31] is an exact f16
// integer.  Both are zero when the super-block's d is zero.
__device__ __forceinline__ void q6k_split(int sc, bool d_zero, uint32_t& mh, uint32_t& ml) {
  const int a = sc < 0 ? -sc : sc;
  const float sg = sc < 0 ? -1.0f : 1.0f;
  mh = f16x2_of(d_zero ? 0.0f : sg * (float)(16 * (a >> 4)));
  ml = f16x2_of(d_zero ? 0.0f : sg * (float)(a & 15));
}

// --------------------------------------------------------------- kernel --
template <int QT, int BN, bool DOTS>
__global__ void __launch_bounds__(Cfg<QT, BN>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const float* __restrict__ scl, const uint8_t* __restrict__ W, float* __restrict__ out,
                   int32_t* __restrict__ dots, int od, int K, int nt, int ntp, int* status, int limit_ms,
                   int skip_first_weight_load, int row_copy) {
  using C = Cfg<QT, BN>;
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t s0 = smem_addr(smem_dyn);
  const uint32_t pad = (1024u - (s0 & 1023u)) & 1023u;
  uint8_t* smem = smem_dyn + pad;
  const uint32_t sb = s0 + pad;
  const Bars<QT, BN> bars{sb + C::BAR_OFF};
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + C::NBARS * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + C::NBARS * 8 + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * C::BM, tok0 = blockIdx.y * BN;
  // split-K: CTA z of gridDim.z takes super-blocks [b_off, b_off + nsb); all
  // ring indices below are relative to the slice, addresses absolute
  const int nsb_all = K >> 8, per = (nsb_all + (int)gridDim.z - 1) / (int)gridDim.z;
  const int b_off = (int)blockIdx.z * per;
  const int nsb = min(per, nsb_all - b_off);
  const Guard g{abort_flag, status, global_ns() + (uint64_t)limit_ms * 1000000ull};
  constexpr bool MIN = C::MINT && !DOTS;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RS; ++i) {
      mbar_init(bars.raw_full(i), 1);
      mbar_init(bars.raw_empty(i), C::UW + (MIN ? 1 : 0));  // unpack warps (+ the min-term MMAs)
    }
    for (int i = 0; i < C::BS; ++i) {
      mbar_init(bars.b_full(i), 1);
      mbar_init(bars.b_empty(i), 1);  // the MMAs that read the stage have completed
    }
    for (int i = 0; i < C::DS; ++i) {
      mbar_init(bars.dx_full(i), 1);
      mbar_init(bars.dx_empty(i), C::NE);  // the epilogue warps read the stage's dx rows
    }
    for (int i = 0; i < C::AS; ++i) {
      mbar_init(bars.a_full(i), C::UW);
      mbar_init(bars.a_empty(i), 1);
    }
    for (int i = 0; i < C::NBUF; ++i) {
      mbar_init(bars.acc_full(i), 1);
      mbar_init(bars.acc_empty(i), C::NE);
    }
    mbar_init(bars.done(), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    if (!row_copy) prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t raw_s = sb + C::RAW_OFF, b_s = sb + C::B_OFF, sc_s = sb + C::SC_OFF, minb_s = sb + C::MINB_OFF;
  const uint32_t amin_s = sb + C::AMIN_OFF;
  // the bf16 parts of s: [K/256][4][ntp][8] after the dx plane [K/32][ntp]
  const uint8_t* smin = reinterpret_cast<const uint8_t*>(scl + (size_t)(K >> 5) * ntp);

  // Each warpgroup sets its register budget at the top of its own branch, so
  // that the budget covers all of the role's code.
  if (warp < C::U0) {
    regs_release<C::REG_CTL>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane 0 waits for free stages and issues the copies.  Raw weights come
    // as one 2-D TMA box of 128 rows, or -- when the row pitch is not a
    // multiple of 16 bytes (Q6_K with K % 2048 != 0), which a tensor map
    // cannot describe -- as one bulk copy per row of the 16-byte-aligned
    // window around the row's 210-byte block, issued by all 32 lanes.
    const size_t row_bytes = (size_t)nsb_all * (QT == kQ4 ? kQ4KBytes : kQ6KBytes);
    const size_t w_bytes = (size_t)od * row_bytes;
    // everything loaded below may be written by the preceding kernel
    griddep_wait();
    int raw_issued = 0, b_issued = 0;
    bool ok = true;
    for (int b = 0; b < nsb && ok; ++b) {
      const int rs = b % C::RS;
      bool okw = true;
      if (lane == 0) okw = gwait(bars.raw_empty(rs), ((b / C::RS) & 1) ^ 1, g);
      if (!__shfl_sync(0xffffffffu, okw, 0)) break;
      if (!(skip_first_weight_load && b == 0)) {
        if (!row_copy) {
          if (lane == 0) {
            mbar_arrive_expect_tx(bars.raw_full(rs), C::RAW_BYTES + (MIN ? C::MINB_BYTES : 0));
            const int x = QT == kQ4 ? (b + b_off) * kQ4KBytes : ((b + b_off) * kQ6KBytes) & ~15;
            tma_load_2d(raw_s + rs * C::RAW_BYTES, &tmW, x, row0, bars.raw_full(rs));
          }
        } else {
          // rows lane + 32i: window [start & ~15, (end + 15) & ~15) of the
          // block's bytes [start, end), capped at the matrix's last 16-byte
          // boundary; the at most 14 bytes past it (last row only) are copied
          // with ordinary loads before the barrier is armed
          uint32_t bytes = 0;
          size_t a0[4], a1[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = lane + 32 * i;
            a0[i] = a1[i] = 0;
            if (row0 + r >= od) continue;
            const size_t start = (size_t)(row0 + r) * row_bytes + (size_t)(b + b_off) * C::BLK;
            const size_t end = start + C::BLK;
            a0[i] = start & ~(size_t)15;
            a1[i] = (end + 15) & ~(size_t)15;
            const size_t cap = w_bytes & ~(size_t)15;
            if (a1[i] > cap) {
              uint8_t* dst = smem + C::RAW_OFF + rs * C::RAW_BYTES + r * C::RAW_ROW;
              for (size_t o = cap; o < end; o += 2)
                *reinterpret_cast<uint16_t*>(dst + (o - a0[i])) = __ldg(reinterpret_cast<const uint16_t*>(W + o));
              a1[i] = cap;
            }
            bytes += (uint32_t)(a1[i] - a0[i]);
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
          __syncwarp();
          if (lane == 0) mbar_arrive_expect_tx(bars.raw_full(rs), bytes + (MIN ? C::MINB_BYTES : 0));
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (a1[i] > a0[i])
              bulk_load(raw_s + rs * C::RAW_BYTES + (lane + 32 * i) * C::RAW_ROW, W + a0[i], (uint32_t)(a1[i] - a0[i]),
                        bars.raw_full(rs));
        }
        if (MIN && lane == 0) {
#pragma unroll
          for (int kc = 0; kc < 4; ++kc)
            bulk_load(minb_s + rs * C::MINB_BYTES + kc * BN * 16,
                      smin + (((size_t)(b + b_off) * 4 + kc) * ntp + tok0) * 16, BN * 16, bars.raw_full(rs));
        }
      }
      ++raw_issued;
      if (lane == 0) {
        for (int s = 0; s < 4; ++s) {
          const int gs = 4 * b + s, bs = gs % C::BS;
          if (!gwait(bars.b_empty(bs), ((gs / C::BS) & 1) ^ 1, g)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bars.b_full(bs), (uint32_t)C::B_BYTES);
          const int gk = gs + 4 * b_off;  // absolute 64-k stage
          tma_load_2d(b_s + bs * C::B_BYTES, &tmX, C::KS * gk, tok0, bars.b_full(bs));
          ++b_issued;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    // drain: every copy still in flight lands before the CTA may exit
    if (lane == 0) {
      const uint64_t dl = global_ns() + 1000000000ull;
      for (int i = raw_issued - C::RS; i < raw_issued; ++i)
        if (i >= 0 && !(skip_first_weight_load && i == 0))
          drain_wait(bars.raw_full(i % C::RS), (i / C::RS) & 1, dl);
      for (int i = b_issued - C::BS; i < b_issued; ++i)
        if (i >= 0) drain_wait(bars.b_full(i % C::BS), (i / C::BS) & 1, dl);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------- dx producer
    // the token-contiguous dx rows of each stage's two 32-value blocks, in
    // their own ring: the epilogue releases them, the MMAs do not wait on it
    if (lane == 0) {
      griddep_wait();
      int issued = 0;
      for (int gs = 0; gs < 4 * nsb; ++gs) {
        const int ds = gs % C::DS;
        if (!gwait(bars.dx_empty(ds), ((gs / C::DS) & 1) ^ 1, g)) break;
        mbar_arrive_expect_tx(bars.dx_full(ds), (uint32_t)C::SC_BYTES);
        const int gk = gs + 4 * b_off;
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
          bulk_load(sc_s + ds * C::SC_BYTES + gi * BN * 4, scl + ((size_t)(2 * gk + gi) * ntp + tok0), BN * 4,
                    bars.dx_full(ds));
        ++issued;
      }
      const uint64_t dl = global_ns() + 1000000000ull;
      for (int i = issued - C::DS; i < issued; ++i)
        if (i >= 0) drain_wait(bars.dx_full(i % C::DS), (i / C::DS) & 1, dl);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA
    // One thread issues every MMA of the CTA, so its loop is kept lean: the
    // stage structure of a super-block is unrolled, ring positions are
    // counters, and the shared-memory descriptors are advanced by constant
    // offsets (a single issuing thread would otherwise spend several times
    // an MMA's duration on index arithmetic between two MMAs).
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(C::BM, BN);
      constexpr uint32_t idesc_bf = idesc | (1u << 7) | (1u << 10);  // A and B bf16
      // descriptor start addresses are in 16-byte units in the low bits
      const uint64_t bdesc0 = smem_desc(b_s, 16, 1024, 2);
      const uint64_t mdesc0 = smem_desc(minb_s, BN * 16, 128, 0);
      const uint64_t adesc0 = smem_desc(amin_s, 2048, 128, 0);
      uint32_t slot = 0, ph = 0;  // accumulator ring position and the parity of its round
      int bs = 0, rs = 0;
      uint32_t bph = 0;
      bool ok = true;
      // the next accumulator, once the epilogue has read it: its TMEM address
      auto acquire = [&](uint32_t& d_t) -> bool {
        if (!gwait(bars.acc_empty(slot), ph ^ 1u, g)) return false;
        tc_fence_after();
        d_t = tmem + slot * (uint32_t)BN;
        return true;
      };
      auto advance = [&]() {
        if (++slot == (uint32_t)C::NBUF) {
          slot = 0;
          ph ^= 1u;
        }
      };
      for (int b = 0; b < nsb && ok; ++b) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const int as = s;  // stage 4b + s uses operand slot s in round b
          if (!gwait(bars.a_full(as), (uint32_t)b & 1u, g) || !gwait(bars.b_full(bs), bph, g)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_t = tmem + (uint32_t)(C::A_COL0 + as * C::ACOLS);
          const uint64_t bd = bdesc0 + (uint64_t)(bs * (C::B_BYTES >> 4));
          uint32_t d_t;
          if (MIN && s == 0) {
            // super-block b: D_min[r][t] = sum over its 8 sub-blocks j of
            // m[r][j] * s[t][j], with s split into three bf16 parts (exact
            // products, f32 sums)
            if (!acquire(d_t)) {
              ok = false;
              break;
            }
            const uint64_t md = mdesc0 + (uint64_t)(rs * (C::MINB_BYTES >> 4));
            const uint64_t ad = adesc0 + (uint64_t)(rs * (C::AMIN_BYTES >> 4));
            tc_mma_f16(d_t, ad, md, idesc_bf, 0u);
            tc_mma_f16(d_t, ad + (uint64_t)((2 * 2048) >> 4), md + (uint64_t)((2 * BN * 16) >> 4), idesc_bf, 1u);
            tc_commit(bars.acc_full(slot));
            tc_commit(bars.raw_empty(rs));  // the raw stage's min operands were read
            advance();
          }
          if constexpr (C::PAIRED) {
            // both blocks into one accumulator pair, one commit: the ring's
            // slots are pairs here (slot < NBUF / 2, BN columns apart)
            if (!gwait(bars.acc_empty(slot), ph ^ 1u, g)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t dp = tmem + slot * (uint32_t)(2 * BN);
#pragma unroll
            for (int gi = 0; gi < 2; ++gi)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                tc_mma_f16_tmem_a(dp + (uint32_t)(gi * BN), a_t + 32 * gi + 8 * i,
                                  bd + (uint64_t)(2 * (2 * gi + (i >> 1))), idesc, i > 0 ? 1u : 0u);
            tc_commit(bars.acc_full(slot));
            if (++slot == (uint32_t)(C::NBUF / 2)) {
              slot = 0;
              ph ^= 1u;
            }
          } else
#pragma unroll
          for (int gi = 0; gi < 2; ++gi) {
            if (!acquire(d_t)) {
              ok = false;
              break;
            }
            if constexpr (QT == kQ4) {
              // sub-block 2p + gi: k 32gi..32gi+31 of the stage, two K=16 MMAs
#pragma unroll
              for (int i = 0; i < 2; ++i)
                tc_mma_f16_tmem_a(d_t, a_t + 16 * gi + 8 * i, bd + (uint64_t)(2 * (2 * gi + i)), idesc,
                                  i > 0 ? 1u : 0u);
            } else {
              // block gi: hi and lo operands of its groups g0 (k 0..15) and g1
              // (k 16..31), each against the group's activation codes
#pragma unroll
              for (int i = 0; i < 4; ++i)
                tc_mma_f16_tmem_a(d_t, a_t + 32 * gi + 8 * i, bd + (uint64_t)(2 * (2 * gi + (i >> 1))), idesc,
                                  i > 0 ? 1u : 0u);
            }
            tc_commit(bars.acc_full(slot));
            advance();
          }
          if (!ok) break;
          tc_commit(bars.a_empty(as));  // the operand stage in TMEM may be rewritten
          tc_commit(bars.b_empty(bs));  // and the activation stage refilled
          if (++bs == C::BS) {
            bs = 0;
            bph ^= 1u;
          }
        }
        if (++rs == C::RS) rs = 0;
      }
      tc_commit(bars.done());
      drain_wait(bars.done(), 0, global_ns() + 1000000000ull);
    }
  }
  } else if (warp < C::E0) {
    if constexpr (C::REG_UNPACK < C::REG_LAUNCH) regs_release<C::REG_UNPACK>();
    // ----------------------------------------------------------- unpack
    const int q = warp & 3;       // TMEM lane quarter
    const int r = 32 * q + lane;  // the thread's weight row within the tile
    // Q6_K: the 32-value block of each stage this warp unpacks (both when
    // there is one unpack warp per lane quarter)
    const int blk0 = C::UW == 8 ? (warp - C::U0) >> 2 : 0, nblk = C::UW == 8 ? 1 : 2;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    int rs = 0;
    uint32_t rph = 0;  // parity of the raw ring's round
    bool ok = true;
    for (int b = 0; b < nsb && ok; ++b) {
      if (!warp_wait(bars.raw_full(rs), rph, g)) break;
      const uint8_t* row = smem + C::RAW_OFF + rs * C::RAW_BYTES + r * C::RAW_ROW;
      // per super-block: Q4_K header (d, dmin, scales); Q6_K scales and d
      uint4 hdr = make_uint4(0, 0, 0, 0);
      uint32_t d6 = 0;
      int blk_off = 0;
      if constexpr (QT == kQ4) {
        hdr = *reinterpret_cast<const uint4*>(row);
      } else {
        // the block's offset in its row's window: the same for every row when
        // the row pitch is a multiple of 16 (one TMA box), per row otherwise
        blk_off = (int)(((size_t)(row0 + r) * ((size_t)nsb_all * kQ6KBytes) + (size_t)(b + b_off) * kQ6KBytes) & 15);
        d6 = *reinterpret_cast<const uint16_t*>(row + blk_off + 208);
      }
      // a rolled loop: the unpack, epilogue and MMA roles run different code
      // at the same time, and unrolled copies of these bodies would not fit
      // the instruction cache together
#pragma unroll 1
      for (int s = 0; s < 4; ++s) {
        const int as = s;
        // the operand stage in TMEM is free again
        if (!warp_wait(bars.a_empty(as), ((uint32_t)b & 1u) ^ 1u, g)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_t = tmem + lane_base + (uint32_t)(C::A_COL0 + as * C::ACOLS);
        if constexpr (QT == kQ4) {
          const uint4 q0 = *reinterpret_cast<const uint4*>(row + 16 + 32 * s);
          const uint4 q1 = *reinterpret_cast<const uint4*>(row + 32 + 32 * s);
          uint32_t sc2, m2;
          q4k_pair_codes(hdr.y, hdr.z, hdr.w, s, sc2, m2);
          uint32_t a[32];
          unpack_q4k_stage(q0, q1, sc2, (hdr.x & 0x7FFFu) == 0, a);
          tc_st_32x32_x32(a_t, a);
          if (MIN && s == 0) {
            // m[r][j] of the 8 sub-blocks as bf16 (exact small integers): k =
            // 8*part + j for the three parts of s, zeros for the fourth chunk
            // (shared memory: the raw stage's min operand)
            uint32_t mv[16];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              uint32_t sc2p, m2p;
              q4k_pair_codes(hdr.y, hdr.z, hdr.w, p, sc2p, m2p);
              const uint32_t pr = (__float_as_uint((float)(m2p & 0xFFu)) >> 16) |
                                  (__float_as_uint((float)(m2p >> 8)) & 0xFFFF0000u);
              mv[p] = mv[4 + p] = mv[8 + p] = pr;
              mv[12 + p] = 0u;
            }
            // chunk p of the canonical K-major layout at p * 2048, row r at r * 16
            uint8_t* am = smem + C::AMIN_OFF + rs * C::AMIN_BYTES + r * 16;
#pragma unroll
            for (int p = 0; p < 4; ++p)
              *reinterpret_cast<uint4*>(am + p * 2048) = make_uint4(mv[4 * p], mv[4 * p + 1], mv[4 * p + 2], mv[4 * p + 3]);
            fence_proxy_async();  // generic writes, read by the MMA through the async proxy
          }
        } else {
          const int n = s >> 1;
          uint32_t H[8], sw[1];
          // TMA rows share one block offset (a warp-uniform branch); rows
          // staged as windows each have their own, so their lanes' words
          // differ in alignment: branch-free reads there (the extra word read
          // ends by byte 224 of the 240-byte row)
          if (!row_copy) {
            load_words_even<8>(row, blk_off + 128 + 32 * n, H);
            load_words_even<1>(row, blk_off + 192 + 4 * s, sw);  // the scales of groups 4s..4s+3
          } else {
            load_words_even_bf<8>(row, blk_off + 128 + 32 * n, H);
            load_words_even_bf<1>(row, blk_off + 192 + 4 * s, sw);
          }
          const bool dz = (d6 & 0x7FFFu) == 0;
#pragma unroll
          for (int bi = 0; bi < 2; ++bi) {
            if (bi >= nblk) break;
            const int blk = blk0 + bi;
            uint32_t L[8];
            if (!row_copy)
              load_words_even<8>(row, blk_off + 64 * n + 32 * blk, L);
            else
              load_words_even_bf<8>(row, blk_off + 64 * n + 32 * blk, L);
            // groups 4s + 2blk and 4s + 2blk + 1: bytes 2blk, 2blk+1 of scale word s
            uint32_t mh[2], ml[2];
#pragma unroll
            for (int h = 0; h < 2; ++h)
              q6k_split((int)(int8_t)((sw[0] >> (8 * (2 * blk + h))) & 0xFFu), dz, mh[h], ml[h]);
            uint32_t a[32];
            unpack_q6k_block(L, H, s, blk, mh, ml, a);
            tc_st_32x32_x32(a_t + 32 * blk, a);
          }
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.a_full(as));
      }
      if (!ok) break;
      release_stage(bars.raw_empty(rs));  // the super-block's raw words were read
      if (++rs == C::RS) {
        rs = 0;
        rph ^= 1u;
      }
    }
  } else {
    if constexpr (C::REG_EPI > C::REG_LAUNCH) regs_take<C::REG_EPI>();
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int cb = (warp - C::E0) >> 2;  // column block: tokens cb*CPW .. + CPW
    const int r = 32 * q + lane;         // tile row
    const int row_g = row0 + r;
    const bool row_ok = row_g < od;
    const int row_c = row_ok ? row_g : od - 1;
    constexpr int CPW = C::CPW, CH = CPW / 32;
    const size_t row_bytes = (size_t)nsb_all * (QT == kQ4 ? kQ4KBytes : kQ6KBytes);
    const uint8_t* wrow = W + (size_t)row_c * row_bytes;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    // the running sums as packed f32 pairs (columns 2i, 2i+1): one FMA-pipe
    // instruction per two outputs
    f2 acc[CPW / 2];
#pragma unroll
    for (int i = 0; i < CPW / 2; ++i) acc[i] = pk2(0.0f, 0.0f);
    float sigma = 1.0f;  // acc holds (partial sum) / sigma
    uint32_t slot = 0, ph = 0;
    int bs = 0;
    uint32_t bph = 0;
    bool ok = true;
    // the weights (scale words) and the outputs may be touched by the
    // preceding kernel
    griddep_wait();
    // the next super-block's scale words are fetched one super-block ahead,
    // so their global-load latency is off the epilogue's critical path
    uint32_t h_next = 0;  // Q4_K: d | dmin << 16; Q6_K: d
    auto fetch = [&](int bb) {
      if (DOTS || bb >= nsb) return;
      if (QT == kQ4)
        h_next = __ldg(reinterpret_cast<const uint32_t*>(wrow + (size_t)(bb + b_off) * kQ4KBytes));
      else
        h_next = __ldg(reinterpret_cast<const uint16_t*>(wrow + (size_t)(bb + b_off) * kQ6KBytes + 208));
    };
    // acc[16c .. 16c+15] += dx[32c .. 32c+31] * P: the chunk's 32 dx values
    // are all loaded first (broadcast shared-memory loads), so their latency
    // is paid once per chunk
    auto fma_chunk = [&](int c, const float* dxp, const uint32_t(&P)[32]) {
      float4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = *reinterpret_cast<const float4*>(dxp + 32 * c + 4 * q);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        f2& a0 = acc[16 * c + 2 * q];
        f2& a1 = acc[16 * c + 2 * q + 1];
        a0 = fma2(pk2(v[q].x, v[q].y), pk2(__uint_as_float(P[4 * q]), __uint_as_float(P[4 * q + 1])), a0);
        a1 = fma2(pk2(v[q].z, v[q].w), pk2(__uint_as_float(P[4 * q + 2]), __uint_as_float(P[4 * q + 3])), a1);
      }
    };
    // acc[16c ..] += m * P (the min-term entry; m is the same for every column)
    auto fma_chunk_scalar = [&](int c, float m, const uint32_t(&P)[32]) {
      const f2 m2 = pk2(m, m);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        acc[16 * c + q] = fma2(m2, pk2(__uint_as_float(P[2 * q]), __uint_as_float(P[2 * q + 1])), acc[16 * c + q]);
    };
    // one accumulator entry: wait, read this warp's CPW columns 32 at a time,
    // hand the accumulator back right after the last read, apply f(chunk, P)
    // to each chunk as soon as it is in registers
    auto entry = [&](auto&& f) -> bool {
      if (!warp_wait(bars.acc_full(slot), ph, g)) return false;
      tc_fence_after();
      const uint32_t t_acc = tmem + lane_base + slot * (uint32_t)BN + (uint32_t)(cb * CPW);
      const uint32_t bar_empty = bars.acc_empty(slot);
      if (++slot == (uint32_t)C::NBUF) {
        slot = 0;
        ph ^= 1u;
      }
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        uint32_t P[32];
        __syncwarp();
        tc_ld_32x32_sync(t_acc + 32 * c, P);
        if (c == CH - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_empty);
        }
        f(c, P);
      }
      return true;
    };
    fetch(0);
    for (int b = 0; b < nsb && ok; ++b) {
      float mc = 0.0f;  // Q4_K: -dmin / sigma
      if (!DOTS) {
        const uint32_t h = h_next;
        fetch(b + 1);
        // the rescaling factors only feed the fp32 sums, so a reciprocal
        // within an ulp or two (instead of an IEEE division) is enough
        const float d = half_bits_to_float(h);
        if (d != 0.0f) {
          const float ratio = sigma * __fdividef(1.0f, d);
          sigma = d;
          if (b > 0) {
            const f2 r2 = pk2(ratio, ratio);
#pragma unroll
            for (int i = 0; i < CPW / 2; ++i) acc[i] = mul2(acc[i], r2);
          }
        }
        if (QT == kQ4) mc = -half_bits_to_float(h >> 16) * __fdividef(1.0f, sigma);
      }
#pragma unroll 1
      for (int s = 0; s < 4 && ok; ++s) {
        if (!warp_wait(bars.dx_full(bs), bph, g)) {
          ok = false;
          break;
        }
        if (MIN && s == 0) {
          ok = entry([&](int c, const uint32_t(&P)[32]) { fma_chunk_scalar(c, mc, P); });
          if (!ok) break;
        }
        const float* scp = reinterpret_cast<const float*>(smem + C::SC_OFF + bs * C::SC_BYTES);
        if constexpr (C::PAIRED) {
          // the stage's two blocks: one wait, both loads, one release
          if (!warp_wait(bars.acc_full(slot), ph, g)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t t_acc = tmem + lane_base + slot * (uint32_t)(2 * BN) + (uint32_t)(cb * CPW);
          const uint32_t bar_empty = bars.acc_empty(slot);
          if (++slot == (uint32_t)(C::NBUF / 2)) {
            slot = 0;
            ph ^= 1u;
          }
#pragma unroll
          for (int gi = 0; gi < 2; ++gi) {
            uint32_t P[32];
            __syncwarp();
            tc_ld_32x32_sync(t_acc + (uint32_t)(gi * BN), P);
            if (gi == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_empty);
            }
            if constexpr (DOTS) {
              const int grp = 8 * (b + b_off) + 2 * s + gi;
              const size_t ng = (size_t)(K >> 5), tstride = (size_t)od * ng;
              const int t0 = tok0 + cb * CPW;
              int32_t* dpp = dots + ((size_t)t0 * od + row_g) * ng + grp;
              const int nv = row_ok ? min(32, nt - t0) : 0;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < nv) dpp[i * tstride] = __float2int_rn(__uint_as_float(P[i]));
            } else {
              fma_chunk(0, scp + gi * BN + cb * CPW, P);
            }
          }
        } else
#pragma unroll
        for (int gi = 0; gi < 2 && ok; ++gi) {
          const float* dxp = scp + gi * BN + cb * CPW;  // dx of this block's tokens
          const int grp = 8 * (b + b_off) + 2 * s + gi;  // the 32-value block within the row
          ok = entry([&](int c, const uint32_t(&P)[32]) {
            if constexpr (DOTS) {
              const size_t ng = (size_t)(K >> 5), tstride = (size_t)od * ng;
              const int t0 = tok0 + cb * CPW + 32 * c;
              int32_t* dp = dots + ((size_t)t0 * od + row_g) * ng + grp;
              const int nv = row_ok ? min(32, nt - t0) : 0;
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (i < nv) dp[i * tstride] = __float2int_rn(__uint_as_float(P[i]));
            } else {
              fma_chunk(c, dxp, P);
            }
          });
        }
        if (!ok) break;
        release_stage(bars.dx_empty(bs));  // the stage's dx rows were read
        if (++bs == C::DS) {
          bs = 0;
          bph ^= 1u;
        }
      }
    }
    if (!DOTS && ok && row_ok) {
#pragma unroll
      for (int i = 0; i < CPW / 2; ++i) {
        const float2 v = upk2(acc[i]);
        const int t = tok0 + cb * CPW + 2 * i;  // slice z's partials
        float* o = out + ((size_t)blockIdx.z * nt + t) * od + row_g;
        if (t < nt) o[0] = sigma * v.x;
        if (t + 1 < nt) o[od] = sigma * v.y;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// ----------------------------------------------------------------- host --
bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// out[i] = sum over the slices z = 0..S-1 of part[z][i], in that order.
__global__ void __launch_bounds__(256) split_reduce_kernel(const float* __restrict__ part, int S, int64_t n,
                                                           float* __restrict__ out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float a = part[i];
    for (int z = 1; z < S; ++z) a += part[(size_t)z * n + i];
    out[i] = a;
  }
}

template <int QT, int BN, bool DOTS>
int launch_cfg(const void* W, const __half* xh, const float* scl, float* out, int32_t* dots, float* part,
               int64_t od, int64_t K, int64_t nt, int* status, int stall_ms, cudaStream_t stream) {
  using C = Cfg<QT, BN>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QMM_EDEVICE;
  int optin = 0;
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (C::SMEM > optin) return QMM_ESMEM;
  static PerDevice<bool> attr_done;
  if (int rc = smem_attr_once(gemm_tc_kernel<QT, BN, DOTS>, C::SMEM, attr_done, dev)) return rc;
  const uint64_t row_bytes = (uint64_t)(K / 256) * (QT == kQ4 ? kQ4KBytes : kQ6KBytes);
  // a tensor map needs a row pitch that is a multiple of 16 bytes; other
  // pitches (Q6_K with K % 2048 != 0) are copied row by row instead
  const int row_copy = row_bytes % 16 ? 1 : 0;
  CUtensorMap mw = {}, mx;
  if (!row_copy && !make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, row_bytes, (uint64_t)od, row_bytes,
                                (uint32_t)C::RAW_ROW, (uint32_t)C::BM, CU_TENSOR_MAP_SWIZZLE_NONE))
    return QMM_ELAUNCH;
  if (!make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, (uint64_t)K, (uint64_t)nt, (uint64_t)K * 2, 64,
                   (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return QMM_ELAUNCH;
  // the block-dot hook writes every block once and needs no slicing
  const int S = DOTS ? 1 : gemm_splits(od, K, nt);
  if (S > 1 && !part) return QMM_EWORKSPACE;
  const dim3 grid((unsigned)((od + C::BM - 1) / C::BM), (unsigned)((nt + BN - 1) / BN), (unsigned)S);
  const int limit_ms = stall_ms > 0 ? stall_ms : 4000;
  // a programmatic dependent of the kernel before it (the quantizer or the
  // operand prepass): barrier set-up, TMEM allocation and the tensor-map
  // prefetch overlap its tail; every load waits for it
  int rc = launch_ex(gemm_tc_kernel<QT, BN, DOTS>, grid, dim3(C::THREADS), (size_t)C::SMEM, stream, true, mw, mx,
                     scl, static_cast<const uint8_t*>(W), S > 1 ? part : out, dots, (int)od, (int)K, (int)nt,
                     (int)gemm_ntp(nt), status, limit_ms, stall_ms > 0 ? 1 : 0, row_copy);
  if (rc) return rc;
  if (S > 1) {
    const int64_t n = nt * od;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    split_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(part, S, n, out);
    if (cudaGetLastError() != cudaSuccess) return QMM_ELAUNCH;
  }
  return QMM_OK;
}

template <int QT, bool DOTS>
int launch_qt(const void* W, const __half* xh, const float* scl, float* out, int32_t* dots, float* part, int64_t od,
              int64_t K, int64_t nt, int* status, int stall_ms, cudaStream_t stream) {
  // the block-dot hook runs the same tile choice as the product path
  if (nt > 64) return launch_cfg<QT, 128, DOTS>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
  return launch_cfg<QT, 64, DOTS>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
}

}  // namespace

int launch_gemm_tc(int qtype, const void* W, const __half* xh, const float* scl, float* out, int32_t* dots,
                   float* part, int64_t od, int64_t K, int64_t nt, int* status, int stall_ms, cudaStream_t stream) {
  if (qtype == QMM_Q4_K)
    return dots ? launch_qt<kQ4, true>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream)
                : launch_qt<kQ4, false>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
  if (qtype == QMM_Q6_K) {
    return dots ? launch_qt<kQ6, true>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream)
                : launch_qt<kQ6, false>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
  }
  return QMM_EINVAL_QTYPE;
}

}  // namespace qmm
