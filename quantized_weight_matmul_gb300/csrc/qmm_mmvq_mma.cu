// qmm_mmvq_mma.cu -- small-batch MMVQ (a few to 16 tokens) on the warp-level
// f16 tensor-core MMA.
//
// What it computes is the MMVQ of qmm_gemv.cu ("04 - Reading minfer's kernels
// II", sec. 3.4; "llama.cpp MMQ", sec. 12.2; "The quantized GEMM", "The GPU
// path"):
//   Q4_K: out[t][r] = sum_j ( d*sc_j*dx_tj*D_trj - dmin*m_j*s_tj ),
//         D_trj = sum over the 32 values of sub-block j of nibble * q
//   Q6_K: out[t][r] = sum_g d*sc_g*dx_t(g/2)*D_trg,
//         D_trg = sum over the 16 values of group g of (q6 - 32) * q
//
// GB300 design.  The dp4a MMVQ spends one instruction on 4 products of one
// token, so from a few tokens on it is bound by instruction issue, not by
// HBM.  Here the integer dots run on mma.sync.m16n8k16 (f16 operands, f32
// accumulation; about 4x the MACs of dp4a per SM on this part, 2048 products
// per instruction):
//  * A (weights, 16 rows x 16 k) holds the codes as f16 SUBNORMALS: the 16-bit
//    pattern of an integer c < 1024 is the f16 value c * 2^-24, so a nibble
//    becomes an operand with one mask and no conversion.  B holds the q8_1
//    codes as f16 integers.  Every product is exact and the f32 sums of one
//    scale group stay far below 2^24 * 2^-24, so D * 2^24 is the exact
//    integer dot.  Q4_K's high nibbles are masked in place (16 * nibble, so
//    D * 2^20); Q6_K's A holds q in [0, 63] and the MMA's C input supplies the
//    -32 as -32 * 2^-24 * (sum of the group's codes).
//  * The k order inside a 32-value block is permuted so that each thread's A
//    elements are bytes of one or two 32-bit words of the raw block (rows g
//    and g+8 of the tile, g = lane/4); the activation codes are written to
//    shared memory once per CTA in the same permuted order, so one 16-byte
//    load per thread gives the B operand of a block and an 8-token tile.
// Work split: a persistent grid of one CTA per SM, each owning a balanced
// range of 16-row tiles.  A producer warp streams every tile in stages of 16
// rows x 2048 k (one TMA box per stage, in a bank-conflict-free row pitch);
// eight consumer warps take one eighth of a stage's k each (Q4_K: one
// super-block; Q6_K: one half of each of two adjacent super-blocks, so every
// warp meets 4-byte- and 2-byte-aligned blocks; sixteen warps for Q4_K with
// raw activations, half a super-block each) and add their partial sums at
// the end of a tile through shared memory in a fixed order.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kQ4 = 0, kQ6 = 1;
constexpr int kSegSB = 8;      // super-blocks per stage (2048 k)
constexpr int kTileRows = 16;  // one m16 tile
constexpr int kMaxStages = 8;
constexpr int kPreStages = 2;  // weight stages a CTA may request before the activations are ready
constexpr int kRedRow = 130;   // floats per (warp, token tile) of the tile-sum buffer (128 + 2: no bank conflicts)
constexpr int kSmemLimit = 227 * 1024;

// Consumer warps.  A stage holds 32 (super-block, 64-value pair) units of
// work; eight warps (four units each) take fewer instructions per stage than
// sixteen and measured faster, except for Q4_K with raw int8 activations,
// whose per-use conversion favours the wider split.
__host__ __device__ constexpr int mma_warps(int qt, int x16) { return qt == kQ4 && !x16 ? 16 : 8; }
__host__ __device__ constexpr int mma_threads(int qt, int x16) { return 32 * (mma_warps(qt, x16) + 1); }
// bytes per row of a warp's coefficient table: one 16-byte entry per block
// of the warp's units, plus 16 (no bank conflicts for the rows g = 0..7)
__host__ __device__ constexpr int mma_coef_row(int nw) { return 64 * 16 / nw + 16; }

template <int QT>
struct MC {
  static constexpr int BLK = QT == kQ4 ? kQ4KBytes : kQ6KBytes;
  static constexpr int SEG = kSegSB * BLK;  // 1152 | 1680
  // Row pitch of a stage = the inner extent of its TMA box.  Q4_K: threads
  // read 8 bytes at row*PITCH + 8c, so PITCH = 32 (mod 128) puts rows
  // g = 0..3 of a half-warp in distinct banks: the box reads 32 bytes past
  // the 8 super-blocks (the next ones, or zero fill past the row's end) and
  // they are ignored.  Q6_K: 4-byte reads at row*PITCH + 4c; 1680 = 16
  // (mod 128) already does.
  static constexpr int PITCH = QT == kQ4 ? SEG + 32 : SEG;
  static constexpr int STAGE = kTileRows * PITCH;
};

// Rows whose pitch is not a multiple of 16 bytes (Q6_K with K % 2048 != 0)
// cannot be described by a TMA tensor map: the producer stages them one by
// one as 16-byte-aligned windows, in rows 32 bytes wider (1712 = 48 mod 128,
// still conflict-free for the 4-byte reads of rows g = 0..3).
__host__ __device__ constexpr bool mma_row_copy(int qt, int64_t K) { return qt != kQ4 && K % 2048 != 0; }
__host__ __device__ constexpr int mma_pitch(int qt, int64_t K) {
  return qt == kQ4 ? MC<kQ4>::PITCH : MC<kQ6>::PITCH + (mma_row_copy(qt, K) ? 32 : 0);
}

// Shared-memory plan of one launch (host and device agree on it).  The raw
// (d, s) pairs of the activations are staged in the coefficient and
// tile-sum areas, which are free until the main loop starts.
struct Plan {
  int stages;
  int x16;       // activations as permuted f16 operands (1) or raw bytes (0)
  int xpitch;    // bytes per token of the activation area
  int x_off, tab_off, coef_off, red_off, bar_off, total;
};

__host__ __device__ inline Plan make_plan(int qt, int ntl, int nt, int K, int stages, int x16) {
  Plan p;
  const int stage_bytes = kTileRows * mma_pitch(qt, K);
  p.stages = stages;
  p.x16 = x16;
  // x16: 64 bytes per (token, block), pitch = 64 (mod 128), the raw codes
  // staged in the upper half; raw: K + 32 | K + 16 (see the loads)
  p.xpitch = x16 ? 2 * K + 64 : (qt == kQ4 ? K + 32 : K + 16);
  p.x_off = stages * stage_bytes;
  p.tab_off = p.x_off + ((nt * p.xpitch + 127) & ~127);
  const int tab_bytes = (K / 32) * 4 * ntl * (qt == kQ4 ? 16 : 32);
  p.coef_off = p.tab_off + tab_bytes;
  const int nw = mma_warps(qt, x16);
  p.red_off = p.coef_off + nw * kTileRows * mma_coef_row(nw);
  // the raw (d, s) pairs are staged from coef_off on: the area ends past
  // the tile-sum buffer and past them
  const int pair_end = p.coef_off + nt * (K / 32) * 8, red_end = p.red_off + 2 * nw * ntl * kRedRow * 4;
  p.bar_off = ((pair_end > red_end ? pair_end : red_end) + 15) & ~15;
  p.total = p.bar_off + (2 * stages + 5) * 8 + 16;
  return p;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// Two signed q8 codes (bytes sel of word u) as an f16x2 of their integer
// values: (q + 128) under the f16 exponent of 1024 is 1152 + q, minus 1152.
__device__ __forceinline__ uint32_t code_pair_f16(uint32_t u, uint32_t sel) {
  return hfma2_bits(prmt(u ^ 0x80808080u, 0x64646464u, sel), 0x3C003C00u, 0xE480E480u);
}

// The B registers of one block for one token from 8 raw codes in the
// thread's permuted order (see the kernel's A layout):
//   Q4_K: w0 = codes 8c..8c+3, w1 = 8c+4..8c+7 -> (0,2) (1,3) of w0, then of w1
//   Q6_K: w0 = codes 4c..4c+3, w1 = 16+4c..16+4c+3, same pairing
__device__ __forceinline__ uint4 b_regs(uint32_t w0, uint32_t w1) {
  return make_uint4(code_pair_f16(w0, 0x4240u), code_pair_f16(w0, 0x4341u), code_pair_f16(w1, 0x4240u),
                    code_pair_f16(w1, 0x4341u));
}

// 32-bit word at byte offset off (even) of a 4-byte-aligned row.
__device__ __forceinline__ uint32_t word_even(const uint8_t* row, int off) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(row + (off & ~3));
  return (off & 2) ? prmt(p[0], p[1], 0x5432u) : p[0];
}

// The consumer warps: the activations (copied in by the producer) into their
// operand layout once, then per stage the warp's share (an eighth or a
// sixteenth) of the k range of one 16-row tile, and one stage after a tile
// ends the fixed-order sum of the warps' partials.
template <int QT, int NTL, bool X16, bool DOTS>
__device__ __forceinline__ void consume(uint8_t* smem, const Plan& P, float* __restrict__ out,
                                        int32_t* __restrict__ dots, int od, int K, int nt, int stages, int t_begin,
                                        int nitems, uint32_t full0, uint32_t empty0, uint32_t red0, uint32_t xbar,
                                        const Guard& gd) {
  using C = MC<QT>;
  constexpr int kNW = mma_warps(QT, X16), CT = 32 * kNW;  // consumer warps, threads
  constexpr int kUPW = 32 / kNW;                           // units of a stage per warp
  constexpr int kCoefRow = mma_coef_row(kNW);
  const int nsb = K >> 8, nbk = K >> 5, nseg = (nsb + kSegSB - 1) / kSegSB;
  const int np = 4 * NTL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // stage row pitch, and the matrix row pitch for the per-row window offsets
  // of rows staged one by one (0 offset for TMA boxes)
  const bool row_copy = mma_row_copy(QT, K);
  const int pitch = mma_pitch(QT, K), stage_sz = kTileRows * pitch;
  const size_t row_bytes = (size_t)nsb * C::BLK;
  const uint32_t rfree0 = red0 + 16;  // red0: two "partials written" barriers, then two "sums read"
  uint8_t* xw = smem + P.x_off;
  bool ok = __all_sync(0xffffffffu, wait_bar(xbar, 0, gd));
  // Operand layout of the activations, per (token, block), in rounds of
  // U per thread whose reads all precede their writes: the f16 B registers
  // (x16; a token's raw codes sit in the upper half of its own row, and a
  // block's operands only overwrite raw codes of lower blocks of the same
  // token, read in this or an earlier round) and the scale table [block]
  // [token pair]: Q4_K (dx_a, dx_b, s_a, s_b); Q6_K (dx_a, dx_b, c0_a, c0_b),
  // (c1_a, c1_b, 0, 0) with c_g = -32 * 2^-24 * (sum of the codes of 16-value
  // group g).  Tokens nt..8*NTL-1 (padding of the last tile) get zero scales.
  {
    constexpr int U = 4;
    float* tab = reinterpret_cast<float*>(smem + P.tab_off);
    const float2* dsr = reinterpret_cast<const float2*>(smem + P.coef_off);  // staged (d, s) pairs
    const int nblk = 8 * NTL * nbk, rounds = (nblk + U * CT - 1) / (U * CT);
    for (int r = 0; r < rounds; ++r) {  // the same count on every thread: a barrier per round
      const int base = r * U * CT + threadIdx.x;
      uint4 c0[U], c1[U];
      float2 dsv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * CT, t = i / nbk, j = i - t * nbk;
        c0[u] = c1[u] = make_uint4(0, 0, 0, 0);
        dsv[u] = make_float2(0.f, 0.f);
        if (ok && i < nblk && t < nt) {
          const uint4* src = reinterpret_cast<const uint4*>(xw + t * P.xpitch + (X16 ? K + 64 : 0) + 32 * j);
          if (X16 || QT == kQ6) {
            c0[u] = src[0];
            c1[u] = src[1];
          }
          dsv[u] = dsr[t * nbk + j];
        }
      }
      if (X16) asm volatile("bar.sync 3, %0;" ::"r"(CT) : "memory");
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * CT, t = i / nbk, j = i - t * nbk;
        if (!ok || i >= nblk) continue;
        if (X16 && t < nt) {
          uint4* d16 = reinterpret_cast<uint4*>(xw + t * P.xpitch + 64 * j);
          if (QT == kQ4) {  // thread c of the MMA takes codes 8c..8c+7
            d16[0] = b_regs(c0[u].x, c0[u].y);
            d16[1] = b_regs(c0[u].z, c0[u].w);
            d16[2] = b_regs(c1[u].x, c1[u].y);
            d16[3] = b_regs(c1[u].z, c1[u].w);
          } else {  // thread c takes codes 4c..4c+3 and 16+4c..16+4c+3
            d16[0] = b_regs(c0[u].x, c1[u].x);
            d16[1] = b_regs(c0[u].y, c1[u].y);
            d16[2] = b_regs(c0[u].z, c1[u].z);
            d16[3] = b_regs(c0[u].w, c1[u].w);
          }
        }
        const int e = t & 1;
        if (QT == kQ4) {
          float* te = tab + ((size_t)j * np + (t >> 1)) * 4;
          te[e] = dsv[u].x;
          te[2 + e] = dsv[u].y;
        } else {
          const uint4 a = c0[u], b = c1[u];
          int s0 = __dp4a((int)a.x, 0x01010101, 0);
          s0 = __dp4a((int)a.y, 0x01010101, s0);
          s0 = __dp4a((int)a.z, 0x01010101, s0);
          s0 = __dp4a((int)a.w, 0x01010101, s0);
          int s1 = __dp4a((int)b.x, 0x01010101, 0);
          s1 = __dp4a((int)b.y, 0x01010101, s1);
          s1 = __dp4a((int)b.z, 0x01010101, s1);
          s1 = __dp4a((int)b.w, 0x01010101, s1);
          float* te = tab + ((size_t)j * np + (t >> 1)) * 8;
          te[e] = dsv[u].x;
          te[2 + e] = -32.0f * 0x1p-24f * (float)s0;  // |32 s| < 2^17: exact
          te[4 + e] = -32.0f * 0x1p-24f * (float)s1;
          te[6 + e] = 0.f;
        }
      }
    }
  }
  asm volatile("bar.sync 3, %0;" ::"r"(CT) : "memory");

  const uint8_t* xs = xw;
  const int g = lane >> 2, c = lane & 3;
  // per row and local block: (c, c, m, m) -- Q4_K c = d*sc*2^24|2^20, m =
  // -dmin*m; Q6_K (c0, c0, c1, c1), the two groups' d*sc*2^24
  uint8_t* coef = smem + P.coef_off + warp * kTileRows * kCoefRow;
  float* red_base = reinterpret_cast<float*>(smem + P.red_off);
  f2 acc[NTL][2];  // rows g, g+8 x tokens (2c, 2c+1) of each 8-token tile
#pragma unroll
  for (int n = 0; n < NTL; ++n) acc[n][0] = acc[n][1] = 0ull;

  // the B operand (8 permuted codes as f16) of block j for token tb
  auto load_b = [&](int tb, int j) -> uint4 {
    if (tb >= nt) return make_uint4(0, 0, 0, 0);
    if (X16) return *reinterpret_cast<const uint4*>(xs + tb * P.xpitch + 64 * j + 16 * c);
    if (QT == kQ4) {
      const uint2 v = *reinterpret_cast<const uint2*>(xs + tb * P.xpitch + 32 * j + 8 * c);
      return b_regs(v.x, v.y);
    }
    const uint8_t* xp = xs + tb * P.xpitch + 32 * j + 4 * c;
    return b_regs(*reinterpret_cast<const uint32_t*>(xp), *reinterpret_cast<const uint32_t*>(xp + 16));
  };

  // Fixed-order sum of the warps' partials of finished tile `to` (rows from
  // tr0), once all warps have written them; done one stage later than the
  // write, so that no warp waits for the slowest one at a tile boundary.
  // A warp owns OPW of the 128 outputs of a token tile; thread T adds warps
  // 4q..4q+3 (q = lane / OPW) for output o, then the partial sums of the q's
  // meet by shuffles in a fixed order: ((w0..3 + w4..7) + (w8..11 + w12..15)).
  constexpr int OPW = 128 / kNW;
  auto reduce_tile = [&](int to, int tr0) -> bool {
    const int par = to & 1;
    if (!__all_sync(0xffffffffu, wait_bar(red0 + 8 * par, (to >> 1) & 1, gd))) return false;
    const float* red = red_base + par * (kNW * NTL * kRedRow);
    const int q = lane / OPW, o = OPW * warp + lane % OPW;
#pragma unroll
    for (int n = 0; n < NTL; ++n) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) sum += red[((4 * q + w) * NTL + n) * kRedRow + o];
#pragma unroll
      for (int m = OPW; m < 32; m <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, m);
      const int ln = o >> 2, e = o & 3;
      const int row = tr0 + (ln >> 2) + 8 * (e >> 1), t = 8 * n + 2 * (ln & 3) + (e & 1);
      if (q == 0 && row < od && t < nt) out[(size_t)t * od + row] = sum;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(rfree0 + 8 * par);
    return true;
  };

  int st = 0, ph = 0, seg = 0, tile = t_begin, tord = 0, pend = -1, pend_r0 = 0;
  for (int it = 0; it < nitems && ok; ++it) {
    ok = __all_sync(0xffffffffu, wait_bar(full0 + 8 * st, ph, gd));
    if (!ok) break;
    const uint8_t* stage = smem + st * stage_sz;
    const int r0 = tile * kTileRows;
    // offset of the stage's first block in row r's window (row copies only)
    auto row_shift = [&](int r) -> int {
      return row_copy ? (int)(((size_t)(r0 + r) * row_bytes + (size_t)seg * C::SEG) & 15) : 0;
    };
    if constexpr (QT == kQ4) {
      // warp -> super-block sbl of the stage, block pairs p0 .. p0 + kUPW - 1
      constexpr int WPS = 4 / kUPW;  // warps per super-block
      const int sbl = warp / WPS, p0 = (warp % WPS) * kUPW, sbi = seg * kSegSB + sbl;
      if (sbi < nsb) {
        {  // coefficients, 16 rows x kUPW pairs: lane -> row lane/2, pairs p0 + 2i + (lane&1)
          const int row = lane >> 1;
          const uint4 hdr = *reinterpret_cast<const uint4*>(stage + row * C::PITCH + sbl * kQ4KBytes);
          const float d = half_bits_to_float(hdr.x), dmin = half_bits_to_float(hdr.x >> 16);
#pragma unroll
          for (int i = 0; i < kUPW / 2; ++i) {
            const int pp = 2 * i + (lane & 1);
            uint32_t sc2, m2;
            q4k_pair_codes(hdr.y, hdr.z, hdr.w, p0 + pp, sc2, m2);
            // D comes out as 2^-24 (low nibbles) or 2^-20 (high nibbles) x the dot
            const float clo = d * 0x1p24f * (float)(sc2 & 0xFFu), mlo = -dmin * (float)(m2 & 0xFFu);
            const float chi = d * 0x1p20f * (float)(sc2 >> 8), mhi = -dmin * (float)(m2 >> 8);
            float4* cr = reinterpret_cast<float4*>(coef + row * kCoefRow + 32 * pp);
            cr[0] = make_float4(clo, clo, mlo, mlo);
            cr[1] = make_float4(chi, chi, mhi, mhi);
          }
        }
        __syncwarp();
        const uint8_t* bg = stage + g * C::PITCH + sbl * kQ4KBytes + 16 + 8 * c;
        const uint8_t* bh = bg + 8 * C::PITCH;
#pragma unroll
        for (int pp = 0; pp < kUPW; ++pp) {
          const int p = p0 + pp;
          const uint2 wg = *reinterpret_cast<const uint2*>(bg + 32 * p);
          const uint2 wh = *reinterpret_cast<const uint2*>(bh + 32 * p);
          const uint32_t g0s = wg.x >> 8, g1s = wg.y >> 8, h0s = wh.x >> 8, h1s = wh.y >> 8;
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const uint32_t M = hi ? 0x00F000F0u : 0x000F000Fu;
            const int jl = 2 * pp + hi, j = 8 * sbi + 2 * p + hi;
            const ulonglong2 cg = *reinterpret_cast<const ulonglong2*>(coef + g * kCoefRow + 16 * jl);
            const ulonglong2 ch = *reinterpret_cast<const ulonglong2*>(coef + (g + 8) * kCoefRow + 16 * jl);
#pragma unroll
            for (int n = 0; n < NTL; ++n) {
              const uint4 b = load_b(8 * n + g, j);
              float D[4];
              mma16816(D, wg.x & M, wh.x & M, g0s & M, h0s & M, b.x, b.y, 0.f, 0.f, 0.f, 0.f);
              mma16816(D, wg.y & M, wh.y & M, g1s & M, h1s & M, b.z, b.w, D[0], D[1], D[2], D[3]);
              if constexpr (DOTS) {
                const float sc = hi ? 0x1p20f : 0x1p24f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int row = r0 + g + 8 * (e >> 1), t = 8 * n + 2 * c + (e & 1);
                  if (row < od && t < nt) dots[((size_t)t * od + row) * nbk + j] = __float2int_rn(D[e] * sc);
                }
              } else {
                // (dx_a, dx_b), (s_a, s_b) of tokens 8n + 2c, 8n + 2c + 1
                const ulonglong2 sx =
                    *reinterpret_cast<const ulonglong2*>(smem + P.tab_off + ((size_t)j * np + 4 * n + c) * 16);
                acc[n][0] = fma2(cg.y, sx.y, fma2(mul2(cg.x, sx.x), pk2(D[0], D[1]), acc[n][0]));
                acc[n][1] = fma2(ch.y, sx.y, fma2(mul2(ch.x, sx.x), pk2(D[2], D[3]), acc[n][1]));
              }
            }
          }
        }
      }
    } else {
      // Q6_K: warp -> super-blocks k2 and k2+1, half h, quad pairs qp0 ..
      // qp0 + QPW - 1 of that half (quads 2qp and 2qp+1): blocks of both
      // alignments.  Quad pairs 0 and 1 read the same ql and qh words (low
      // and high nibbles, other qh bits), loaded once for both.
      constexpr int QPW = kUPW / 2, WPH = 2 / QPW;  // quad pairs per warp, warps per half
      const int k2 = 2 * (warp / (2 * WPH)), h = (warp / WPH) & 1, qp0 = (warp % WPH) * QPW;
      // (super-blocks past the row's end, in a partial last stage, are skipped:
      // rows staged one by one carry the next row's bytes there, not zeros)
      {  // coefficients, 16 rows x 2 super-blocks x QPW quad pairs x 2 blocks
         // x 2 groups: lane -> row lane/2, super-block k2 + (lane&1)
        const int row = lane >> 1, u = lane & 1;
        const uint8_t* rowp = stage + row * pitch;
        const int boff = row_shift(row) + (k2 + u) * kQ6KBytes;
        const float d = half_bits_to_float(*reinterpret_cast<const uint16_t*>(rowp + boff + 208)) * 0x1p24f;
#pragma unroll
        for (int qi = 0; qi < QPW; ++qi) {
          const uint32_t sw = word_even(rowp, boff + 192 + 8 * h + 4 * (qp0 + qi));  // groups 8h+4qp..+3
          float v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) v[i] = d * (float)(int8_t)((sw >> (8 * i)) & 0xFFu);
          float4* cr = reinterpret_cast<float4*>(coef + row * kCoefRow + 16 * (4 * qi + 2 * u));
          cr[0] = make_float4(v[0], v[0], v[1], v[1]);
          cr[1] = make_float4(v[2], v[2], v[3], v[3]);
        }
      }
      __syncwarp();
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int sbl = k2 + u, sbi = seg * kSegSB + sbl;
        if (sbi >= nsb) break;
        const uint8_t* rg = stage + g * pitch;
        const uint8_t* rh = rg + 8 * pitch;
        const int boff = sbl * kQ6KBytes, sg = row_shift(g), sh = row_shift(g + 8);
        // words of rows g and g+8 for steps s = 0, 1: ql at the half's two
        // 32-byte offsets (quad q takes offset q & 1, nibble q >> 1); qh
        uint32_t QL[2][2][2], QH[2][2];
#pragma unroll
        for (int s = 0; s < 2; ++s) {
          const int o = boff + 64 * h + 16 * s + 4 * c, oh = boff + 128 + 32 * h + 16 * s + 4 * c;
          QL[0][s][0] = word_even(rg, sg + o);
          QL[0][s][1] = word_even(rg, sg + o + 32);
          QH[0][s] = word_even(rg, sg + oh);
          QL[1][s][0] = word_even(rh, sh + o);
          QL[1][s][1] = word_even(rh, sh + o + 32);
          QH[1][s] = word_even(rh, sh + oh);
        }
#pragma unroll
        for (int qx = 0; qx < 2 * QPW; ++qx) {
          const int qi = qx >> 1, qq = qx & 1, qp = qp0 + qi;
          const int q = 2 * qp + qq, jl = 4 * qi + 2 * u + qq, j = 8 * sbi + 4 * h + q;  // j: block within the row
          const ulonglong2 cg = *reinterpret_cast<const ulonglong2*>(coef + g * kCoefRow + 16 * jl);
          const ulonglong2 ch = *reinterpret_cast<const ulonglong2*>(coef + (g + 8) * kCoefRow + 16 * jl);
          // 6-bit codes of quad q: low 4 bits from ql (high nibbles for quads
          // 2, 3), top 2 bits from bits 2q..2q+1 of qh
          uint32_t A[2][4];  // [step][a0..a3]
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            uint32_t code[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
              code[rr] = ((QL[rr][s][qq] >> (4 * qp)) & 0x0F0F0F0Fu) | (((QH[rr][s] >> (2 * q)) << 4) & 0x30303030u);
            A[s][0] = prmt(code[0], 0u, 0x4240u);
            A[s][1] = prmt(code[1], 0u, 0x4240u);
            A[s][2] = prmt(code[0], 0u, 0x4341u);
            A[s][3] = prmt(code[1], 0u, 0x4341u);
          }
#pragma unroll
          for (int n = 0; n < NTL; ++n) {
            const uint4 b = load_b(8 * n + g, j);
            const float4* tp = reinterpret_cast<const float4*>(smem + P.tab_off + ((size_t)j * np + 4 * n + c) * 32);
            const float4 t0 = tp[0], t1 = tp[1];
            float D0[4], D1[4];
            mma16816(D0, A[0][0], A[0][1], A[0][2], A[0][3], b.x, b.y, t0.z, t0.w, t0.z, t0.w);
            mma16816(D1, A[1][0], A[1][1], A[1][2], A[1][3], b.z, b.w, t1.x, t1.y, t1.x, t1.y);
            if constexpr (DOTS) {
              const int ng = K >> 4;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int row = r0 + g + 8 * (e >> 1), t = 8 * n + 2 * c + (e & 1);
                if (row < od && t < nt) {
                  int32_t* dp = dots + ((size_t)t * od + row) * ng + 2 * j;
                  dp[0] = __float2int_rn(D0[e] * 0x1p24f);
                  dp[1] = __float2int_rn(D1[e] * 0x1p24f);
                }
              }
            } else {
              const f2 dx = pk2(t0.x, t0.y);
              acc[n][0] = fma2(dx, fma2(cg.y, pk2(D1[0], D1[1]), mul2(cg.x, pk2(D0[0], D0[1]))), acc[n][0]);
              acc[n][1] = fma2(dx, fma2(ch.y, pk2(D1[2], D1[3]), mul2(ch.x, pk2(D0[2], D0[3]))), acc[n][1]);
            }
          }
        }
      }
    }
    release_stage(empty0 + 8 * st);

    int fresh = -1;
    if (!DOTS && seg == nseg - 1) {
      // the tile is done: its partials go to buffer tord & 1, once the sums
      // of tile tord - 2 have been read out of it
      const int par = tord & 1;
      if (tord >= 2 && !__all_sync(0xffffffffu, wait_bar(rfree0 + 8 * par, ((tord >> 1) - 1) & 1, gd))) {
        ok = false;
        break;
      }
      float* red = red_base + par * (kNW * NTL * kRedRow);
#pragma unroll
      for (int n = 0; n < NTL; ++n) {
        float* rw = red + (warp * NTL + n) * kRedRow + 4 * lane;
        *reinterpret_cast<float2*>(rw) = upk2(acc[n][0]);
        *reinterpret_cast<float2*>(rw + 2) = upk2(acc[n][1]);
        acc[n][0] = acc[n][1] = 0ull;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(red0 + 8 * par);
      fresh = tord++;
    }
    if (pend >= 0) {
      if (!reduce_tile(pend, pend_r0)) {
        ok = false;
        break;
      }
      pend = -1;
    }
    if (fresh >= 0) {
      pend = fresh;
      pend_r0 = r0;
    }
    if (++st == stages) {
      st = 0;
      ph ^= 1;
    }
    if (++seg == nseg) {
      seg = 0;
      ++tile;
    }
  }
  if (ok && pend >= 0) reduce_tile(pend, pend_r0);
}

template <int QT, int NTL, bool X16, bool DOTS>
__global__ void __launch_bounds__(mma_threads(QT, X16), 1)
    mmvq_mma_kernel(const __grid_constant__ CUtensorMap tmW, const uint8_t* __restrict__ W,
                    const int8_t* __restrict__ xq, const float* __restrict__ xds,
                    float* __restrict__ out, int32_t* __restrict__ dots, int od, int K, int nt, int stages,
                    int* status, int static_w, int limit_ms, int skip_first) {
  using C = MC<QT>;
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t s0 = smem_addr(smem_dyn);
  const uint32_t pad = (1024u - (s0 & 1023u)) & 1023u;
  uint8_t* smem = smem_dyn + pad;
  const uint32_t sb = s0 + pad;
  const Plan P = make_plan(QT, NTL, nt, K, stages, X16 ? 1 : 0);

  const int nsb = K >> 8, nbk = K >> 5, nseg = (nsb + kSegSB - 1) / kSegSB;
  const int G = (od + kTileRows - 1) / kTileRows;
  const int t_begin = (int)((int64_t)G * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)G * (blockIdx.x + 1) / gridDim.x);
  const int nitems = (t_end - t_begin) * nseg;
  // barriers: stage full x stages, stage empty x stages, tile sums (4), activations
  const uint32_t full0 = sb + P.bar_off, empty0 = full0 + 8 * stages, red0 = empty0 + 8 * stages;
  const uint32_t xbar = red0 + 32;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P.bar_off + (2 * stages + 5) * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kNW = mma_warps(QT, X16);
  const Guard gd{abort_flag, status, global_ns() + (uint64_t)limit_ms * 1000000ull};

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kNW);
    }
    for (int i = 0; i < 4; ++i) mbar_init(red0 + 8 * i, kNW);  // partials written x2, sums read x2
    mbar_init(xbar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  griddep_launch_dependents();

  if (warp == kNW) {
    // ------------------------------------------------------------- producer
    // Lane 0 issues the copies.  Rows staged one by one (Q6_K rows whose
    // pitch is not a multiple of 16 bytes) take one bulk copy per row: there
    // the whole warp runs the weight stream and lane r stages row r.
    const bool row_copy = mma_row_copy(QT, K);
    const unsigned am = row_copy ? 0xffffffffu : 1u;  // the lanes issuing weights
    if (lane == 0 || row_copy) {
      const int pitch = mma_pitch(QT, K), stage_sz = kTileRows * pitch;
      const size_t row_bytes = (size_t)nsb * C::BLK, total = (size_t)od * row_bytes;
      if (!row_copy) prefetch_tmap(&tmW);
      int issued = 0, st = 0, ph = 0, seg = 0, tile = t_begin;
      // one box: 16 rows x PITCH bytes from super-block 8*seg (rows past od
      // and bytes past the row's end arrive zero-filled)
      auto issue = [&]() -> bool {
        if (!__all_sync(am, wait_bar(empty0 + 8 * st, ph ^ 1, gd))) return false;
        if (!(skip_first && issued == 0)) {  // the stall test hook skips the first stage
          if (!row_copy) {
            mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)C::STAGE);
            tma_load_2d(sb + st * C::STAGE, &tmW, seg * (C::SEG / 8), tile * kTileRows, full0 + 8 * st);
          } else {
            // the stage's super-blocks of row `lane`, one window
            const int nbs = min(kSegSB, nsb - seg * kSegSB);
            size_t a0 = 0, a1 = 0;
            if (lane < kTileRows && tile * kTileRows + lane < od) {
              const size_t start = (size_t)(tile * kTileRows + lane) * row_bytes + (size_t)seg * C::SEG;
              const RowWindow w = stage_row_window(start, start + (size_t)nbs * C::BLK, total,
                                                   smem + st * stage_sz + lane * pitch, W);
              a0 = w.a0;
              a1 = w.a1 > w.a0 ? w.a1 : w.a0;
            }
            uint32_t bytes = (uint32_t)(a1 - a0);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
            // the bytes a lane stored itself (past the matrix's last 16-byte
            // boundary) are ordered before lane 0's arrive by the warp sync
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * st, bytes);
            __syncwarp();
            if (a1 > a0) bulk_load(sb + st * stage_sz + lane * pitch, W + a0, (uint32_t)(a1 - a0), full0 + 8 * st);
          }
        }
        ++issued;
        if (++st == stages) {
          st = 0;
          ph ^= 1;
        }
        if (++seg == nseg) {
          seg = 0;
          ++tile;
        }
        return true;
      };
      bool pok = true;
      // weights the caller declared static may start before the preceding
      // kernel completes -- a couple of stages only, so that the activations
      // copied next do not queue behind a full ring
      const int pre = static_w ? min(kPreStages, nitems) : 0;
      for (int i = 0; i < pre && pok; ++i) pok = issue();
      // every lane that copies weights waits for the preceding grid from here
      griddep_wait();
      if (lane == 0) {
        // the activations: each token's codes (x16: into the upper half of its
        // row), then all (d, s) pairs into the staging area
        mbar_arrive_expect_tx(xbar, (uint32_t)(nt * K + nt * nbk * 8));
        for (int t = 0; t < nt; ++t)
          bulk_load(sb + P.x_off + t * P.xpitch + (X16 ? K + 64 : 0), xq + (size_t)t * K, (uint32_t)K, xbar);
        bulk_load(sb + P.coef_off, xds, (uint32_t)(nt * nbk * 8), xbar);
      }
      while (pok && issued < nitems) pok = issue();
      if (lane == 0) {
        // drain: every copy in flight lands before the CTA exits
        const uint64_t dl = global_ns() + 1000000000ull;
        for (int i = issued - stages; i < issued; ++i) {
          if (i < 0 || (skip_first && i == 0)) continue;
          for (uint32_t k = 0; !mbar_try_wait(full0 + 8 * (i % stages), (i / stages) & 1); ++k)
            if ((k & 63u) == 63u && global_ns() > dl) break;
        }
        for (uint32_t k = 0; !mbar_try_wait(xbar, 0); ++k)
          if ((k & 63u) == 63u && global_ns() > dl) break;
      }
    }
  } else if (nitems > 0) {
    consume<QT, NTL, X16, DOTS>(smem, P, out, dots, od, K, nt, stages, t_begin, nitems, full0, empty0, red0, xbar,
                                gd);
  }
  __syncthreads();
}

// Largest ring that fits next to the activations; x16 when it still leaves
// at least 4 stages, else raw activation bytes with at least 2.
bool choose_plan(int qt, int ntl, int64_t nt, int64_t K, Plan* out) {
  if (nt < 1 || nt > 8 * ntl || K < 256 || K > (1 << 20)) return false;
  for (int x16 = 1; x16 >= 0; --x16) {
    for (int st = kMaxStages; st >= (x16 ? 4 : 2); --st) {
      const Plan p = make_plan(qt, ntl, (int)nt, (int)K, st, x16);
      if (p.total + 1024 <= kSmemLimit) {
        *out = p;
        return true;
      }
    }
  }
  return false;
}

template <int QT, int NTL, bool X16, bool DOTS>
int launch_mma_cfg(const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots, int64_t od,
                   int64_t K, int64_t nt, int* status, Dep dep, const Plan& p, cudaStream_t stream) {
  const bool pdl = dep != Dep::kNone, static_w = dep == Dep::kPdlStaticW;
  auto kern = mmvq_mma_kernel<QT, NTL, X16, DOTS>;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QMM_EDEVICE;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  static PerDevice<bool> attr_done;
  if (int rc = smem_attr_once(kern, kSmemLimit, attr_done, dev)) return rc;
  // W viewed as [od][row_bytes/8] 8-byte elements; one box = 16 rows x PITCH bytes
  using C = MC<QT>;
  auto fn = tensor_map_encoder();
  if (!fn) return QMM_ELAUNCH;
  const uint64_t row_bytes = (uint64_t)(K / 256) * C::BLK;
  CUtensorMap m = {};
  const cuuint64_t dims[2] = {row_bytes / 8, (cuuint64_t)od};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(C::PITCH / 8), (cuuint32_t)kTileRows};
  const cuuint32_t estr[2] = {1, 1};
  // rows whose pitch is not a multiple of 16 bytes are staged by the kernel
  // itself, one window per row
  if (!mma_row_copy(QT, K) &&
      fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(W), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return QMM_ELAUNCH;
  const int64_t tiles = (od + kTileRows - 1) / kTileRows;
  const int stall = stall_ms();
  int grid = nsm > 0 ? nsm : 152;
  if (grid > tiles) grid = (int)tiles;
  return launch_ex(kern, dim3(grid), dim3(mma_threads(QT, X16)), (size_t)p.total + 1024, stream, pdl, m,
                   static_cast<const uint8_t*>(W), xq, xds, out, dots,
                   (int)od, (int)K, (int)nt, p.stages, status, static_w ? 1 : 0, stall > 0 ? stall : 4000,
                   stall > 0 ? 1 : 0);
}

template <int QT, int NTL, bool DOTS>
int launch_mma_ntl(const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots, int64_t od,
                   int64_t K, int64_t nt, int* status, Dep dep, cudaStream_t stream) {
  Plan p;
  if (!choose_plan(QT, NTL, nt, K, &p)) return QMM_ESMEM;
  if (p.x16) return launch_mma_cfg<QT, NTL, true, DOTS>(W, xq, xds, out, dots, od, K, nt, status, dep, p, stream);
  return launch_mma_cfg<QT, NTL, false, DOTS>(W, xq, xds, out, dots, od, K, nt, status, dep, p, stream);
}

template <int QT, bool DOTS>
int launch_mma_qt(const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots, int64_t od,
                  int64_t K, int64_t nt, int* status, Dep dep, cudaStream_t stream) {
  if (nt <= 8) return launch_mma_ntl<QT, 1, DOTS>(W, xq, xds, out, dots, od, K, nt, status, dep, stream);
  return launch_mma_ntl<QT, 2, DOTS>(W, xq, xds, out, dots, od, K, nt, status, dep, stream);
}

}  // namespace

bool mmvq_mma_fits(int qtype, int64_t nt, int64_t K) {
  if (qtype != QMM_Q4_K && qtype != QMM_Q6_K) return false;
  if (nt < 1 || nt > kMmaMaxNt) return false;
  Plan p;
  return choose_plan(qtype == QMM_Q4_K ? kQ4 : kQ6, nt <= 8 ? 1 : 2, nt, K, &p);
}

int launch_mmvq_mma(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots,
                    int64_t od, int64_t K, int64_t nt, int* status, Dep dep, cudaStream_t stream) {
  if (!mmvq_mma_fits(qtype, nt, K)) return QMM_ESMEM;
  if (qtype == QMM_Q4_K)
    return dots ? launch_mma_qt<kQ4, true>(W, xq, xds, out, dots, od, K, nt, status, dep, stream)
                : launch_mma_qt<kQ4, false>(W, xq, xds, out, dots, od, K, nt, status, dep, stream);
  return dots ? launch_mma_qt<kQ6, true>(W, xq, xds, out, dots, od, K, nt, status, dep, stream)
              : launch_mma_qt<kQ6, false>(W, xq, xds, out, dots, od, K, nt, status, dep, stream);
}

}  // namespace qmm
