// qmm_gemm_tc.cu -- MMQ on the sm_103a tensor cores (tcgen05, TMEM, TMA).
//
// What it computes ("llama.cpp MMQ", sec. 4-6; "The quantized GEMM",
// "The GPU path"):
//   Q4_K: out[t][r] = sum_b sum_j ( d_b*sc_j*dx_tj*D_trj - dmin_b*m_j*s_tj ),
//         D = sum over the 32 values of sub-block j of nibble * q
//   Q6_K: out[t][r] = sum_b sum_g d_b*sc_g*dx_t(g/2)*D_trg,
//         D = sum over the 16 values of group g of (q6 - 32) * q
//
// GB300 design.  The int8 MMA of this part is slow (the legacy warp-level
// path) and tcgen05 has no int8 kind on sm_103a, so the integer dots run on
// the f16 kind: every operand is a small integer that f16 holds exactly
// (nibble*sc <= 945, q6-32 in [-32,31], q8 in [-127,127]) and the f32
// accumulation of one scale group (|D| < 2^24) is exact, so the TMEM
// accumulator holds the exact integer dot.
//
// One CTA computes a 128-row x BN-token tile with 12 warps:
//   warp 0      TMA producer: raw weight super-blocks (128 rows x 144 B, or
//               240 B windows for the 2-byte-aligned Q6_K blocks), the f16
//               activation tile (BN x 64, 128-byte swizzle) and the
//               token-contiguous (dx, s) rows of the same 64 k.
//   warp 1      TMEM allocation and the single MMA-issuing thread: per scale
//               group an MMA chain into one of NBUF TMEM accumulators (3 to 8
//               of the 512 columns; round robin by group), committed to an
//               mbarrier.
//   warps 2-3   unpack: raw nibbles / 6-bit codes -> f16 operand tiles in the
//               canonical no-swizzle K-major layout (Q4_K folds the 6-bit scale
//               into the operand: sc*nibble is exact), one 64-k stage at a time.
//   warps 4-11  epilogue: TMEM -> registers per group, fp32 rescale into
//               register accumulators, one fp32 store at the end.  A TMEM
//               accumulator is handed back to the MMA thread only after the
//               epilogue has finished the arithmetic on the values it read
//               from it.
// Stages that a role reads with ordinary loads and the producer refills with
// TMA (raw weights, the per-token scale rows) are handed back through
// release_stage, which fences the reads against the async-proxy refill.
// Every wait is bounded: a wait that runs past its deadline raises the CTA's
// abort flag and QMM_ETIMEOUT in the status word, all roles leave their
// loops, in-flight copies and MMAs are drained, and TMEM is freed.
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
  static constexpr int BM = 128;
  // unpack warps.  A 14-warp layout with four caps a thread at 128 registers
  // and was measured no faster for Q6_K (it also exposed, before the stages
  // were handed back through release_stage, the cross-proxy refill race that
  // release_stage closes).
  static constexpr int NU = 2;
  static constexpr int UROWS = BM / (32 * NU);  // rows each unpack thread converts per stage
  static constexpr int EPI0 = 2 + NU;           // first of the 8 epilogue warps
  static constexpr int THREADS = 32 * (EPI0 + 8);
  static constexpr int KS = 64;  // k per operand stage
  static constexpr int RS = 2, AS = 3, BS = 4;
  // raw bytes per row and super-block in shared memory (Q6_K: a window
  // around the 2-byte-aligned 210-byte block; 240 rather than 224 bytes, so
  // that a warp's 32-bit loads of 32 rows hit 8 bank offsets instead of 4)
  static constexpr int RAW_ROW = QT == kQ4 ? 144 : 240;
  static constexpr int GPS = QT == kQ4 ? 2 : 4;  // scale groups per stage
  static constexpr int MPG = QT == kQ4 ? 2 : 1;  // K=16 MMAs per group
  static constexpr int RAW_BYTES = BM * RAW_ROW;
  static constexpr int A_BYTES = BM * KS * 2;
  static constexpr int B_BYTES = BN * KS * 2;
  static constexpr int SC_BYTES = 2 * BN * 4;  // dx of the stage's two 32-k groups
  // Q4_K min term: per super-block the MMA operands m[row][8p + j] (A) and
  // s_p[token][8p + j] (B, the three bf16 parts of s), k = 32: 4 chunks of 8
  static constexpr bool MINMMA = QT == kQ4;
  static constexpr int AMIN_BYTES = MINMMA ? BM * 64 : 0;
  static constexpr int BMIN_BYTES = MINMMA ? BN * 64 : 0;
  // TMEM (all 512 columns): NBUF group accumulators of BN columns, then the
  // min-term accumulator
  static constexpr int TMEM_COLS = 512;
  static constexpr int NBUF = TMEM_COLS / BN - (MINMMA ? 1 : 0);
  static_assert(NBUF <= 8, "accumulator barriers");
  static constexpr int RAW_OFF = 0;
  static constexpr int A_OFF = RAW_OFF + RS * RAW_BYTES;
  static constexpr int B_OFF = A_OFF + AS * A_BYTES;
  static constexpr int SC_OFF = B_OFF + BS * B_BYTES;
  static constexpr int AMIN_OFF = SC_OFF + BS * SC_BYTES;
  static constexpr int BMIN_OFF = AMIN_OFF + RS * AMIN_BYTES;
  static constexpr int BAR_OFF = BMIN_OFF + RS * BMIN_BYTES;
  // barriers: raw full/empty, a full/empty, b full/empty, acc full/empty, done, min full/empty
  static constexpr int NBARS = 2 * RS + 2 * AS + 2 * BS + 16 + 1 + 2;
  static constexpr int SMEM = BAR_OFF + NBARS * 8 + 16 + 1024;  // + slack for 1 KB alignment
  static_assert(RAW_BYTES % 1024 == 0 && A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "align");
  static_assert(SC_BYTES % 16 == 0, "align");
};

struct Bars {
  uint32_t base;
  int RS, AS, BS;
  __device__ uint32_t raw_full(int i) const { return base + 8 * i; }
  __device__ uint32_t raw_empty(int i) const { return base + 8 * (RS + i); }
  __device__ uint32_t a_full(int i) const { return base + 8 * (2 * RS + i); }
  __device__ uint32_t a_empty(int i) const { return base + 8 * (2 * RS + AS + i); }
  __device__ uint32_t b_full(int i) const { return base + 8 * (2 * RS + 2 * AS + i); }
  __device__ uint32_t b_empty(int i) const { return base + 8 * (2 * RS + 2 * AS + BS + i); }
  __device__ uint32_t acc_full(int i) const { return base + 8 * (2 * RS + 2 * AS + 2 * BS + i); }
  __device__ uint32_t acc_empty(int i) const { return base + 8 * (2 * RS + 2 * AS + 2 * BS + 8 + i); }
  __device__ uint32_t done() const { return base + 8 * (2 * RS + 2 * AS + 2 * BS + 16); }
  __device__ uint32_t min_full() const { return base + 8 * (2 * RS + 2 * AS + 2 * BS + 17); }
  __device__ uint32_t min_empty() const { return base + 8 * (2 * RS + 2 * AS + 2 * BS + 18); }
};

// Wait used while draining: ignores the abort flag, gives up at `deadline`.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t deadline) {
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return;
    if ((it & 63u) == 63u && global_ns() > deadline) return;
  }
}

// Warp-uniform bounded wait: every lane polls, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const Guard& g) {
  const bool ok = wait_bar(bar, parity, g);
  return __all_sync(0xffffffffu, ok);
}

// f16x2 of (1024 + a, 1024 + b) for two 4..6-bit codes held in bits 0-5 and 16-21.
__device__ __forceinline__ uint32_t magic_pair(uint32_t two_codes, uint32_t mask) {
  return and_or(two_codes, mask, 0x64006400u);
}

// ---------------------------------------------------------------- unpack --
// Q4_K: pair p of one row (qs bytes 32p..32p+31) -> 64 f16 operand values in
// k order: the low nibbles are k 0..31 (sub-block 2p), the high ones k 32..63
// (sub-block 2p+1).  Each value is sc*nibble (FOLD) or the nibble itself.
// Output: row-major 8-k chunks at dst + kc*2048 (kc = k/8), 16 bytes each.
// The 12 words of pair p of one row: the 16-byte header, then qs bytes
// 32p..32p+31.
struct Q4Raw {
  uint4 hdr, q0, q1;
};
__device__ __forceinline__ Q4Raw load_q4k_pair(const uint8_t* raw_row, int p) {
  return {*reinterpret_cast<const uint4*>(raw_row), *reinterpret_cast<const uint4*>(raw_row + 16 + 32 * p),
          *reinterpret_cast<const uint4*>(raw_row + 16 + 32 * p + 16)};
}

template <bool FOLD>
__device__ __forceinline__ void unpack_q4k_pair(const Q4Raw& rw, int p, uint8_t* dst) {
  const uint4 hdr = rw.hdr, q0 = rw.q0, q1 = rw.q1;
  const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
  uint32_t mul_lo, off_lo, mul_hi, off_hi;
  if (FOLD) {
    int sc_lo, m_lo, sc_hi, m_hi;
    q4k_scale_min_words(hdr.y, hdr.z, hdr.w, 2 * p, sc_lo, m_lo);
    q4k_scale_min_words(hdr.y, hdr.z, hdr.w, 2 * p + 1, sc_hi, m_hi);
    if ((hdr.x & 0x7FFFu) == 0) sc_lo = sc_hi = 0;  // d == 0: the main term vanishes
    const __half2 a = __float2half2_rn((float)sc_lo), b = __float2half2_rn((float)sc_hi);
    const __half2 na = __float2half2_rn(-1024.0f * (float)sc_lo), nb = __float2half2_rn(-1024.0f * (float)sc_hi);
    mul_lo = *reinterpret_cast<const uint32_t*>(&a);
    mul_hi = *reinterpret_cast<const uint32_t*>(&b);
    off_lo = *reinterpret_cast<const uint32_t*>(&na);
    off_hi = *reinterpret_cast<const uint32_t*>(&nb);
  } else {
    mul_lo = mul_hi = 0x3C003C00u;  // 1.0
    off_lo = off_hi = 0xE400E400u;  // -1024.0
  }
#pragma unroll
  for (int kc = 0; kc < 4; ++kc) {
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t wd = w[2 * kc + e];
      const uint32_t t01 = prmt(wd, 0u, 0x4140u), t23 = prmt(wd, 0u, 0x4342u);
      lo[2 * e] = hfma2_bits(magic_pair(t01, 0x000F000Fu), mul_lo, off_lo);
      lo[2 * e + 1] = hfma2_bits(magic_pair(t23, 0x000F000Fu), mul_lo, off_lo);
      hi[2 * e] = hfma2_bits(magic_pair(t01 >> 4, 0x000F000Fu), mul_hi, off_hi);
      hi[2 * e + 1] = hfma2_bits(magic_pair(t23 >> 4, 0x000F000Fu), mul_hi, off_hi);
    }
    *reinterpret_cast<uint4*>(dst + kc * 2048) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(dst + (kc + 4) * 2048) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  }
}

// Q6_K: stage s (elements 64s..64s+63 of the super-block) of one row -> 64
// f16 values q - 32.  Element 128n + 32*quad + l takes its low 4 bits from
// ql[64n + l] (quads 0, 2) or ql[64n + 32 + l] (quads 1, 3) -- the low nibble
// for quads 0-1, the high one for quads 2-3 -- and its top 2 bits from bits
// 2*quad..2*quad+1 of qh[32n + l].  Stage s covers half n = s/2, quads
// 2(s%2) and 2(s%2)+1.
struct Q6Raw {
  uint32_t L[16], H[8];  // ql bytes 64n..64n+63, qh bytes 32n..32n+31 of half n = s/2
};
__device__ __forceinline__ void load_q6k_stage(const uint8_t* row_window, int blk_off, int s, Q6Raw& rw) {
  const int n = s >> 1;
  load_words_even<16>(row_window, blk_off + 64 * n, rw.L);
  load_words_even<8>(row_window, blk_off + 128 + 32 * n, rw.H);
}

__device__ __forceinline__ void unpack_q6k_stage(const Q6Raw& rw, int s, uint8_t* dst) {
  const uint32_t* L = rw.L;
  const uint32_t* H = rw.H;
  const bool upper = s & 1;
  const uint32_t mul = 0x3C003C00u, off = 0xE420E420u;  // 1.0, -1056.0 (= -1024 - 32)
#pragma unroll
  for (int kc = 0; kc < 8; ++kc) {
    // kc 0..3: first quad of the stage, l = 8kc..; kc 4..7: second quad, l = 8(kc-4)..
    const int quad1 = kc >> 2;
    const int i0 = 2 * (kc & 3);  // word index of l
    uint32_t v[4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t lw = L[i0 + e + 8 * quad1];
      const uint32_t hw = H[i0 + e];
      uint32_t codes;
      if (!upper) {
        codes = (lw & 0x0F0F0F0Fu) | ((quad1 ? (hw << 2) : (hw << 4)) & 0x30303030u);
      } else {
        codes = ((lw >> 4) & 0x0F0F0F0Fu) | ((quad1 ? (hw >> 2) : hw) & 0x30303030u);
      }
      const uint32_t t01 = prmt(codes, 0u, 0x4140u), t23 = prmt(codes, 0u, 0x4342u);
      v[2 * e] = hfma2_bits(magic_pair(t01, 0x003F003Fu), mul, off);
      v[2 * e + 1] = hfma2_bits(magic_pair(t23, 0x003F003Fu), mul, off);
    }
    *reinterpret_cast<uint4*>(dst + kc * 2048) = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

// --------------------------------------------------------------- kernel --
template <int QT, int BN, bool DOTS>
__global__ void __launch_bounds__(Cfg<QT, BN>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const float* __restrict__ scl, const uint8_t* __restrict__ W, float* __restrict__ out,
                   int32_t* __restrict__ dots, int od, int K, int nt, int ntp, int* status, int limit_ms,
                   int skip_first_weight_load) {
  using C = Cfg<QT, BN>;
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t s0 = smem_addr(smem_dyn);
  const uint32_t pad = (1024u - (s0 & 1023u)) & 1023u;
  uint8_t* smem = smem_dyn + pad;
  const uint32_t sb = s0 + pad;
  const Bars bars{sb + C::BAR_OFF, C::RS, C::AS, C::BS};
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::BAR_OFF + C::NBARS * 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::BAR_OFF + C::NBARS * 8 + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * C::BM, tok0 = blockIdx.y * BN;
  // split-K: CTA z of gridDim.z takes super-blocks [b_off, b_off + nsb); all
  // ring indices below are relative to the slice, addresses absolute
  const int nsb_all = K >> 8, per = (nsb_all + (int)gridDim.z - 1) / (int)gridDim.z;
  const int b_off = (int)blockIdx.z * per;
  const int nsb = min(per, nsb_all - b_off), NS = 4 * nsb;
  const Guard g{abort_flag, status, global_ns() + (uint64_t)limit_ms * 1000000ull};

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RS; ++i) {
      mbar_init(bars.raw_full(i), 1);
      mbar_init(bars.raw_empty(i), C::NU + (C::MINMMA && !DOTS ? 1 : 0));  // unpack warps (+ the min-term MMAs)
    }
    for (int i = 0; i < C::AS; ++i) {
      mbar_init(bars.a_full(i), C::NU);
      mbar_init(bars.a_empty(i), 1);
    }
    for (int i = 0; i < C::BS; ++i) {
      mbar_init(bars.b_full(i), 1);
      mbar_init(bars.b_empty(i), 1 + 8);
    }
    for (int i = 0; i < C::NBUF; ++i) {
      mbar_init(bars.acc_full(i), 1);
      mbar_init(bars.acc_empty(i), 8);
    }
    mbar_init(bars.done(), 1);
    mbar_init(bars.min_full(), 1);
    mbar_init(bars.min_empty(), 8);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(C::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t raw_s = sb + C::RAW_OFF, a_s = sb + C::A_OFF, b_s = sb + C::B_OFF, sc_s = sb + C::SC_OFF;
  const uint32_t amin_s = sb + C::AMIN_OFF, bmin_s = sb + C::BMIN_OFF;
  // the bf16 parts of s: [K/256][4][ntp][8] after the dx plane [K/32][ntp]
  const uint8_t* smin = reinterpret_cast<const uint8_t*>(scl + (size_t)(K >> 5) * ntp);
  constexpr bool MIN = C::MINMMA && !DOTS;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t nbytes_b = (uint64_t)C::B_BYTES + C::SC_BYTES;
      int raw_issued = 0, b_issued = 0;
      bool ok = true;
      for (int b = 0; b < nsb && ok; ++b) {
        const int rs = b % C::RS;
        if (!wait_bar(bars.raw_empty(rs), ((b / C::RS) & 1) ^ 1, g)) break;
        if (!(skip_first_weight_load && b == 0)) {
          mbar_arrive_expect_tx(bars.raw_full(rs), C::RAW_BYTES + (MIN ? 4 * BN * 16 : 0));
          const int x = QT == kQ4 ? (b + b_off) * kQ4KBytes : ((b + b_off) * kQ6KBytes) & ~15;
          tma_load_2d(raw_s + rs * C::RAW_BYTES, &tmW, x, row0, bars.raw_full(rs));
          if (MIN) {
#pragma unroll
            for (int kc = 0; kc < 4; ++kc)
              bulk_load(bmin_s + rs * C::BMIN_BYTES + kc * BN * 16,
                        smin + (((size_t)(b + b_off) * 4 + kc) * ntp + tok0) * 16, BN * 16, bars.raw_full(rs));
          }
        }
        ++raw_issued;
        for (int s = 0; s < 4; ++s) {
          const int gs = 4 * b + s, bs = gs % C::BS;
          if (!wait_bar(bars.b_empty(bs), ((gs / C::BS) & 1) ^ 1, g)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bars.b_full(bs), (uint32_t)nbytes_b);
          const int gk = gs + 4 * b_off;  // absolute 64-k stage
          tma_load_2d(b_s + bs * C::B_BYTES, &tmX, C::KS * gk, tok0, bars.b_full(bs));
#pragma unroll
          for (int gi = 0; gi < 2; ++gi)
            bulk_load(sc_s + bs * C::SC_BYTES + gi * BN * 4, scl + ((size_t)(2 * gk + gi) * ntp + tok0),
                      BN * 4, bars.b_full(bs));
          ++b_issued;
        }
      }
      // drain: every copy still in flight lands before the CTA may exit
      const uint64_t dl = global_ns() + 1000000000ull;
      for (int i = raw_issued - C::RS; i < raw_issued; ++i)
        if (i >= 0 && !(skip_first_weight_load && i == 0))
          drain_wait(bars.raw_full(i % C::RS), (i / C::RS) & 1, dl);
      for (int i = b_issued - C::BS; i < b_issued; ++i)
        if (i >= 0) drain_wait(bars.b_full(i % C::BS), (i / C::BS) & 1, dl);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(C::BM, BN);
      int u = 0;
      bool ok = true;
      for (int gs = 0; gs < NS && ok; ++gs) {
        const int as = gs % C::AS, bs = gs % C::BS;
        if (!wait_bar(bars.a_full(as), (gs / C::AS) & 1, g)) break;
        if (!wait_bar(bars.b_full(bs), (gs / C::BS) & 1, g)) break;
        tc_fence_after();
        for (int gi = 0; gi < C::GPS; ++gi, ++u) {
          const int buf = u % C::NBUF;
          if (!wait_bar(bars.acc_empty(buf), ((u / C::NBUF) & 1) ^ 1, g)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int i = 0; i < C::MPG; ++i) {
            const int kk = gi * C::MPG + i;  // K=16 chunk within the 64-k stage
            const uint64_t ad = smem_desc(a_s + as * C::A_BYTES + kk * 4096, 2048, 128, 0);
            const uint64_t bd = smem_desc(b_s + bs * C::B_BYTES + kk * 32, 16, 1024, 2);
            tc_mma_f16(tmem + (uint32_t)(buf * BN), ad, bd, idesc, i > 0 ? 1u : 0u);
          }
          tc_commit(bars.acc_full(buf));
        }
        if (!ok) break;
        tc_commit(bars.a_empty(as));
        tc_commit(bars.b_empty(bs));
        if (MIN && (gs & 3) == 3) {
          // super-block b: D_min[r][t] = sum over its 8 sub-blocks j of
          // m[r][j] * s[t][j], with s split into three bf16 parts (exact
          // products, f32 sums); then the raw stage (and these operands) may go
          const int b = gs >> 2, rs = b % C::RS;
          if (!wait_bar(bars.min_empty(), (b & 1) ^ 1, g)) break;
          tc_fence_after();
          const uint32_t idesc_bf = idesc_f16(C::BM, BN) | (1u << 7) | (1u << 10);  // A and B bf16
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t ad = smem_desc(amin_s + rs * C::AMIN_BYTES + kk * 4096, 2048, 128, 0);
            const uint64_t bd = smem_desc(bmin_s + rs * C::BMIN_BYTES + kk * 2 * BN * 16, BN * 16, 128, 0);
            tc_mma_f16(tmem + (uint32_t)(C::NBUF * BN), ad, bd, idesc_bf, kk > 0 ? 1u : 0u);
          }
          tc_commit(bars.min_full());
          tc_commit(bars.raw_empty(rs));
        }
      }
      tc_commit(bars.done());
      drain_wait(bars.done(), 0, global_ns() + 1000000000ull);
    }
  } else if (warp < C::EPI0) {
    // ----------------------------------------------------------- unpack
    const int ut = threadIdx.x - 64;  // rows ut + 32 * NU * rr, rr < UROWS
    bool ok = true;
    for (int b = 0; b < nsb && ok; ++b) {
      const int rs = b % C::RS;
      if (!warp_wait(bars.raw_full(rs), (b / C::RS) & 1, g)) break;
      const uint8_t* raw = smem + C::RAW_OFF + rs * C::RAW_BYTES;
      for (int s = 0; s < 4; ++s) {
        const int gs = 4 * b + s, as = gs % C::AS;
        if (!warp_wait(bars.a_empty(as), ((gs / C::AS) & 1) ^ 1, g)) {
          ok = false;
          break;
        }
        uint8_t* a = smem + C::A_OFF + as * C::A_BYTES;
        if (MIN && s == 0) {
          // m[r][j] of the 8 sub-blocks as bf16 (exact small integers), the
          // same 16 bytes for parts 0, 1, 2, zeros for the fourth chunk
#pragma unroll
          for (int rr = 0; rr < C::UROWS; ++rr) {
            const int r = ut + 32 * C::NU * rr;
            const uint4 hdr = *reinterpret_cast<const uint4*>(raw + r * C::RAW_ROW);
            uint32_t mw[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              uint32_t sc2, m2;
              q4k_pair_codes(hdr.y, hdr.z, hdr.w, p, sc2, m2);
              mw[p] = (__float_as_uint((float)(m2 & 0xFFu)) >> 16) | (__float_as_uint((float)(m2 >> 8)) & 0xFFFF0000u);
            }
            uint8_t* am = smem + C::AMIN_OFF + rs * C::AMIN_BYTES + r * 16;
            const uint4 v = make_uint4(mw[0], mw[1], mw[2], mw[3]);
            *reinterpret_cast<uint4*>(am) = v;
            *reinterpret_cast<uint4*>(am + 2048) = v;
            *reinterpret_cast<uint4*>(am + 4096) = v;
            *reinterpret_cast<uint4*>(am + 6144) = make_uint4(0, 0, 0, 0);
          }
        }
        // all rows' raw words first, then the conversions and stores: the
        // compiler cannot move a later row's loads above an earlier row's
        // stores (both are shared memory), so this overlaps their latency
        if constexpr (QT == kQ4) {
          Q4Raw rw[C::UROWS];
#pragma unroll
          for (int rr = 0; rr < C::UROWS; ++rr) rw[rr] = load_q4k_pair(raw + (ut + 32 * C::NU * rr) * C::RAW_ROW, s);
#pragma unroll
          for (int rr = 0; rr < C::UROWS; ++rr) unpack_q4k_pair<!DOTS>(rw[rr], s, a + (ut + 32 * C::NU * rr) * 16);
        } else {
          const int blk_off = ((b + b_off) * kQ6KBytes) & 15;
          Q6Raw rw[C::UROWS];
#pragma unroll
          for (int rr = 0; rr < C::UROWS; ++rr)
            load_q6k_stage(raw + (ut + 32 * C::NU * rr) * C::RAW_ROW, blk_off, s, rw[rr]);
#pragma unroll
          for (int rr = 0; rr < C::UROWS; ++rr) unpack_q6k_stage(rw[rr], s, a + (ut + 32 * C::NU * rr) * 16);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.a_full(as));
      }
      if (!ok) break;
      release_stage(bars.raw_empty(rs));
    }
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;               // TMEM lane quarter this warp may read
    const int hc = (warp - C::EPI0) >> 2;  // column half
    const int r = 32 * q + lane;          // tile row
    const int row_g = row0 + r;
    const bool row_ok = row_g < od;
    const int row_c = row_ok ? row_g : od - 1;
    constexpr int HALF = BN / 2;
    constexpr int CH = HALF / 32;
    const size_t row_bytes = (size_t)nsb_all * (QT == kQ4 ? kQ4KBytes : kQ6KBytes);
    const uint8_t* wrow = W + (size_t)row_c * row_bytes;
    // Q4_K: one f32 per token of the warp's columns (one FMA per output and
    // group, measured faster than packed pairs); Q6_K: packed pairs of tokens
    // (2i, 2i + 1), so the group's scale multiply and the FMA take one
    // instruction per two outputs each
    constexpr bool PK = QT != kQ4;
    float acc[PK ? 1 : HALF];
    f2 acc2[PK ? HALF / 2 : 1];
#pragma unroll
    for (int i = 0; i < (PK ? 1 : HALF); ++i) acc[i] = 0.0f;
#pragma unroll
    for (int i = 0; i < (PK ? HALF / 2 : 1); ++i) acc2[i] = 0ull;
    float sigma = 1.0f;  // acc holds (partial sum) / sigma
    int u = 0;
    bool ok = true;
    // the next super-block's scale words are fetched one super-block ahead,
    // so their global-load latency is off the epilogue's critical path
    uint4 hdr_next = make_uint4(0, 0, 0, 0);  // Q4_K: d, dmin and the 12 packed scale bytes
    uint32_t sw_next[9] = {};                 // Q6_K: the 16 int8 scales as 8 half-words, then d
    auto fetch_scales = [&](int bb) {
      if (DOTS || bb >= nsb) return;
      if (QT == kQ4) {
        hdr_next = __ldg(reinterpret_cast<const uint4*>(wrow + (size_t)(bb + b_off) * kQ4KBytes));
      } else {
        const uint16_t* hs = reinterpret_cast<const uint16_t*>(wrow + (size_t)(bb + b_off) * kQ6KBytes + 192);
#pragma unroll
        for (int i = 0; i < 9; ++i) sw_next[i] = __ldg(hs + i);
      }
    };
    fetch_scales(0);
    for (int b = 0; b < nsb && ok; ++b) {
      float gcoef[QT == kQ4 ? 1 : 16];  // Q4_K: -dmin / sigma; Q6_K: the groups' scales
      if (!DOTS) {
        const uint4 hdr = hdr_next;
        uint32_t sw[9];
#pragma unroll
        for (int i = 0; i < 9; ++i) sw[i] = sw_next[i];
        fetch_scales(b + 1);
        // the rescaling factors only feed the fp32 sums, so a reciprocal
        // within an ulp or two (instead of an IEEE division) is enough
        const float d = half_bits_to_float(QT == kQ4 ? hdr.x : sw[8]);
        if (d != 0.0f) {
          const float ratio = sigma * __fdividef(1.0f, d);
          sigma = d;
          if (b > 0) {
            if constexpr (PK) {
              const f2 r2 = pk2(ratio, ratio);
#pragma unroll
              for (int i = 0; i < HALF / 2; ++i) acc2[i] = mul2(acc2[i], r2);
            } else {
#pragma unroll
              for (int i = 0; i < HALF; ++i) acc[i] *= ratio;
            }
          }
        }
        if (QT == kQ4) {
          gcoef[0] = -half_bits_to_float(hdr.x >> 16) * __fdividef(1.0f, sigma);  // -dmin / sigma
        } else {
#pragma unroll
          for (int gg = 0; gg < 16; ++gg) {
            const int sc = (int)(int8_t)((sw[gg >> 1] >> (8 * (gg & 1))) & 0xFF);
            gcoef[gg] = d != 0.0f ? (float)sc : 0.0f;
          }
        }
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int gs = 4 * b + s, bs = gs % C::BS;
        if (!warp_wait(bars.b_full(bs), (gs / C::BS) & 1, g)) {
          ok = false;
          break;
        }
        const float* scp = reinterpret_cast<const float*>(smem + C::SC_OFF + bs * C::SC_BYTES);
#pragma unroll
        for (int gi = 0; gi < C::GPS; ++gi, ++u) {
          const int buf = u % C::NBUF;
          if (!warp_wait(bars.acc_full(buf), (u / C::NBUF) & 1, g)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // one 32-column chunk at a time: load, wait, use (32 live
          // registers of TMEM data instead of BN/2, so nothing spills)
          const int sub = QT == kQ4 ? gi : (gi >> 1);  // 32-value sub-block within the stage
          const float* sg = scp + sub * BN + hc * HALF;  // dx of this group's tokens
          const float coef = DOTS || QT == kQ4 ? 1.0f : gcoef[4 * s + gi];
          const f2 coef2 = pk2(coef, coef);
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            uint32_t P[32];
            __syncwarp();
            tc_ld_32x32_sync(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * BN + hc * HALF + 32 * c), P);
            if (DOTS) {
              const int ng = QT == kQ4 ? (K >> 5) : (K >> 4);
              const int grp = QT == kQ4 ? 8 * (b + b_off) + 2 * s + gi : 16 * (b + b_off) + 4 * s + gi;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                const int t = tok0 + hc * HALF + 32 * c + i;
                if (row_ok && t < nt)
                  dots[((size_t)t * od + row_g) * ng + grp] = __float2int_rn(__uint_as_float(P[i]));
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 v = *reinterpret_cast<const float4*>(sg + 32 * c + i);
                if constexpr (PK) {  // Q6_K: dx times the group's scale, then the FMA
                  const f2 dx01 = mul2(pk2(v.x, v.y), coef2), dx23 = mul2(pk2(v.z, v.w), coef2);
                  f2& a01 = acc2[(32 * c + i) / 2];
                  f2& a23 = acc2[(32 * c + i) / 2 + 1];
                  a01 = fma2(dx01, pk2(__uint_as_float(P[i]), __uint_as_float(P[i + 1])), a01);
                  a23 = fma2(dx23, pk2(__uint_as_float(P[i + 2]), __uint_as_float(P[i + 3])), a23);
                } else {  // Q4_K: the group's scale is folded into the weight operand
                  static_assert(QT == kQ4, "the scalar form has no group scale");
                  const float dx[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    acc[32 * c + i + e] = fmaf(dx[e], __uint_as_float(P[i + e]), acc[32 * c + i + e]);
                }
              }
            }
          }
          // hand the accumulator back only now, after its values were used
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars.acc_empty(buf));
        }
        if (!ok) break;
        release_stage(bars.b_empty(bs));  // the stage's dx rows were read
      }
      if (MIN && ok) {
        // the super-block's min term: acc += (-dmin / sigma) * D_min
        if (!warp_wait(bars.min_full(), b & 1, g)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float mc = gcoef[0];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          uint32_t Q[32];
          __syncwarp();
          tc_ld_32x32_sync(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(C::NBUF * BN + hc * HALF + 32 * c), Q);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[32 * c + i] = fmaf(mc, __uint_as_float(Q[i]), acc[32 * c + i]);
        }
        // hand the accumulator back only after its values were used
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.min_empty());
      }
    }
    if (!DOTS && ok && row_ok) {
#pragma unroll
      for (int i = 0; i < HALF; i += 2) {
        const float2 a = PK ? upk2(acc2[i / 2]) : make_float2(acc[i], acc[i + 1]);
        const int t = tok0 + hc * HALF + i;  // slice z's partials
        if (t < nt) out[((size_t)blockIdx.z * nt + t) * od + row_g] = sigma * a.x;
        if (t + 1 < nt) out[((size_t)blockIdx.z * nt + t + 1) * od + row_g] = sigma * a.y;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                 : "memory");
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
  CUtensorMap mw, mx;
  if (!make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, W, row_bytes, (uint64_t)od, row_bytes,
                   (uint32_t)C::RAW_ROW, (uint32_t)C::BM, CU_TENSOR_MAP_SWIZZLE_NONE))
    return QMM_ELAUNCH;
  if (!make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xh, (uint64_t)K, (uint64_t)nt, (uint64_t)K * 2, 64,
                   (uint32_t)BN, CU_TENSOR_MAP_SWIZZLE_128B))
    return QMM_ELAUNCH;
  // the block-dot hook writes every group once and needs no slicing
  const int S = DOTS ? 1 : gemm_splits(od, K, nt);
  if (S > 1 && !part) return QMM_EWORKSPACE;
  const dim3 grid((unsigned)((od + C::BM - 1) / C::BM), (unsigned)((nt + BN - 1) / BN), (unsigned)S);
  const int limit_ms = stall_ms > 0 ? stall_ms : 4000;
  gemm_tc_kernel<QT, BN, DOTS><<<grid, C::THREADS, C::SMEM, stream>>>(
      mw, mx, scl, static_cast<const uint8_t*>(W), S > 1 ? part : out, dots,
      (int)od, (int)K, (int)nt, (int)gemm_ntp(nt), status, limit_ms, stall_ms > 0 ? 1 : 0);
  if (cudaGetLastError() != cudaSuccess) return QMM_ELAUNCH;
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
  // the block-dot hook always takes the 128-token tile, so only the product
  // path instantiates the 64-token one
  if constexpr (DOTS) {
    return launch_cfg<QT, 128, true>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
  } else {
    if (nt > 64)
      return launch_cfg<QT, 128, false>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
    return launch_cfg<QT, 64, false>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
  }
}

}  // namespace

int launch_gemm_tc(int qtype, const void* W, const __half* xh, const float* scl, float* out, int32_t* dots,
                   float* part, int64_t od, int64_t K, int64_t nt, int* status, int stall_ms, cudaStream_t stream) {
  if (qtype == QMM_Q4_K)
    return dots ? launch_qt<kQ4, true>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream)
                : launch_qt<kQ4, false>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
  if (qtype == QMM_Q6_K) {
    if (K % 2048) return QMM_EINVAL_SHAPE;  // 16-byte row pitch for the TMA weight map
    return dots ? launch_qt<kQ6, true>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream)
                : launch_qt<kQ6, false>(W, xh, scl, out, dots, part, od, K, nt, status, stall_ms, stream);
  }
  return QMM_EINVAL_QTYPE;
}

}  // namespace qmm
