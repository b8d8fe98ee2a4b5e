// qmm_gemv.cu -- MMVQ: the small-batch (nt <= 8) Q4_K / Q6_K x q8_1 matmul.
//
// What it computes ("04 - Reading minfer's kernels II", sec. 3.4; "llama.cpp
// MMQ", sec. 12.2; "The quantized GEMM", "The GPU path"): for every weight
// row r and token t
//   Q4_K: out[t][r] = sum_j ( d*sc_j*dx_tj*D_trj - dmin*m_j*s_tj ),
//         D_trj = sum_{i<32} nibble[r][32j+i] * q[t][32j+i]   (exact int32, dp4a)
//   Q6_K: out[t][r] = sum_g d*sc_g*dx_t(g/2)*D_trg,
//         D_trg = sum_{i<16} (q6[r][16g+i] - 32) * q[t][16g+i]
//         (the 6-bit codes are dotted as unsigned bytes; the -32 comes off as
//         32 x the group's code sum)
// The weight matrix is streamed from HBM exactly once and every weight block
// meets all nt tokens while it is on chip: nt never multiplies the weight
// traffic.
//
// GB300 design: a persistent grid, one CTA per SM, each CTA owning a
// contiguous, balanced range of CR-row groups.  One producer thread keeps a
// ring of shared-memory stages full with 2-D TMA tiles of the raw weight
// bytes (CR rows x 8 super-blocks = 2048 k), so tens of KB per SM are in
// flight whatever the consumers do.  Each consumer warp takes R rows of a
// stage; lane l handles super-block l/4 of the stage and part p = l%4 of it,
// i.e. 64 consecutive weights (Q4_K: sub-blocks 2p and 2p+1; Q6_K: groups
// 4p..4p+3), so its activation slice is the same for all R rows.
//
// Two ways in for the activations:
//   * staged: q8_1 codes and scales produced by the quantizer are copied
//     once per CTA into shared memory (bulk copy);
//   * fused: the consumer warps quantize the f32 activations themselves into
//     shared memory (two lanes per 32-value block; the same codes as the
//     quantizer, see q8_code_words) and write the q8_1 outputs too -- one kernel
//     per matmul instead of two, for the decode shapes where nt*K is small.
// Kernels are launched as programmatic dependents of the preceding kernel
// and let their own dependents start early, so consecutive matmuls overlap
// their launch and ramp.  Every global access that may depend on the
// preceding kernel waits for it (griddepcontrol.wait) -- except, when the
// caller declares the weights static, the weight stream itself, which then
// starts before the preceding kernel has finished.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

namespace {

constexpr int kQ4 = 0, kQ6 = 1;
constexpr int kSegSB = 8;  // super-blocks per stage (2048 k)
// bytes of one row per stage: 1152 (Q4_K), 1680 (Q6_K; a multiple of 16)
__host__ __device__ constexpr int seg_bytes(int qt) { return kSegSB * (qt == kQ4 ? kQ4KBytes : kQ6KBytes); }
// Shared-memory pitch of a stage row: seg_bytes for a TMA box; 32 more
// bytes when the rows are staged one by one as 16-byte-aligned windows (a
// matrix row pitch that is not a multiple of 16: Q6_K with K % 2048 != 0)
__host__ __device__ constexpr bool row_copy_needed(int qt, int64_t K) { return qt != kQ4 && K % 2048 != 0; }
__host__ __device__ constexpr int stage_row(int qt, int64_t K) {
  return seg_bytes(qt) + (row_copy_needed(qt, K) ? 32 : 0);
}
constexpr int kSmemBudget = 200 * 1024;        // staged path (large nt*K)
// Fused path: two CTAs (of consecutive kernels) share an SM, so each gets at
// most half of the 228 KB less the 1 KB the hardware reserves per CTA; the
// activations come first and the weight ring takes what is left, 3..5 stages.
constexpr int kFusedCtaSmem = (228 * 1024 - 2 * 1024) / 2;
constexpr int kFusedMaxStages = 5;
constexpr int kFusedMinStages = 3;

template <int QT, int NW, int R>
struct GemvCfg {
  static constexpr int CR = NW * R;  // rows per stage (R rows per consumer warp)
  static constexpr int SEG_BYTES = seg_bytes(QT);
  static constexpr int BLK = QT == kQ4 ? kQ4KBytes : kQ6KBytes;
  static constexpr int STAGE_BYTES = CR * SEG_BYTES;
  static constexpr int THREADS = 32 * (NW + 1);
};

int64_t act_bytes_of(int64_t nt, int64_t K) { return nt * K + nt * (K / 32) * 8; }

// The fused path pads each token's code plane to whole 2048-code stages.
int64_t fused_plane(int64_t K) { return (K + 2047) / 2048 * 2048; }
int64_t fused_act_bytes(int64_t nt, int64_t K) { return nt * fused_plane(K) + nt * (K / 32) * 8; }

// Ring stages of the fused kernel for nt x K (16-row, 2048-k stages), 0 if
// fewer than kFusedMinStages fit next to the activations.
int fused_stages(int qt, int64_t nt, int64_t K) {
  const int64_t fixed = ((fused_act_bytes(nt, K) + 15) & ~15) + 32 + 1024;
  int64_t st = (kFusedCtaSmem - fixed) / (16 * stage_row(qt, K) + 16);
  if (st > kFusedMaxStages) st = kFusedMaxStages;
  return st >= kFusedMinStages ? (int)st : 0;
}

int stages_for(int qt, int64_t nt, int64_t K, int CR, int64_t budget) {
  int s = (int)((budget - act_bytes_of(nt, K) - 1024 - 256) / ((int64_t)CR * stage_row(qt, K)));
  return s > 8 ? 8 : s;
}

// Byte offset, in the fused path's shared activation plane of one token, of
// code k: the 64 codes a lane reads per stage are split into four 16-byte
// chunks stored chunk-major across the 32 lanes, so a warp's chunk loads
// touch 32 consecutive 16-byte words (no bank conflicts).
__device__ __forceinline__ int fused_code_offset(int k) {
  const int seg = k >> 11, r = k & 2047;
  return (((seg * 4 + ((r & 63) >> 4)) * 32 + (r >> 6)) << 4) + (r & 15);
}

// Lane-constant part of the Q4_K (scale, min) decode of sub-blocks 2p and
// 2p+1 ("llama.cpp MMQ", sec. 6): pairs 0-1 keep both 6-bit codes in the low
// six bits of scale bytes j and j+4; pairs 2-3 keep their low 4 bits in the
// nibbles of bytes j+4 and their top 2 bits in the top of bytes j-4 / j.
// With the header words w1..w3 holding scales[0..11] and sh = 16(p%2),
//   p < 2:  sc2 = (w1 >> sh) & 0x3F3F,   m2 = (w2 >> sh) & 0x3F3F
//   p >= 2: sc2 = ((w3 >> sh) & 0x0F0F) | ((w1 >> (sh+2)) & 0x3030)
//           m2  = ((w3 >> (sh+4)) & 0x0F0F) | ((w2 >> (sh+2)) & 0x3030)
// which one branch-free form covers with per-lane shifts and masks.
struct Q4PairDecode {
  uint32_t sh, sh2, shm, mA, mB;
  bool upper;
  __device__ explicit Q4PairDecode(int p)
      : sh(16u * (uint32_t)(p & 1)), sh2(16u * (uint32_t)(p & 1) + 2u), shm(16u * (uint32_t)(p & 1) + (p >= 2 ? 4u : 0u)),
        mA(p >= 2 ? 0x0F0Fu : 0x3F3Fu), mB(p >= 2 ? 0x3030u : 0u), upper(p >= 2) {}
  // the two scale codes (bytes 0, 1) and the two min codes of the pair
  __device__ __forceinline__ void codes(uint32_t w1, uint32_t w2, uint32_t w3, uint32_t& sc2, uint32_t& m2) const {
    const uint32_t a = upper ? w3 : w1, am = upper ? w3 : w2;
    sc2 = ((a >> sh) & mA) | ((w1 >> sh2) & mB);
    m2 = ((am >> shm) & mA) | ((w2 >> sh2) & mB);
  }
};

// 2^23 + byte b of w as an f32 bit pattern (b = 0 or 1): one PRMT, no
// integer-to-float conversion; fma(s, f, -s * 2^23) is then s * byte exactly
// whenever s * byte fits the f32 significand.
__device__ __forceinline__ float magic_byte(uint32_t w, uint32_t b) {
  return __uint_as_float(prmt(w, 0x4B000000u, 0x7650u + b));
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void named_arrive(int id, int threads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int QT, int NT, int NW, int R, bool DOTS, bool FUSED>
__global__ void __launch_bounds__(32 * (NW + 1), FUSED ? 2 : 1)
    mmvq_stream_kernel(const __grid_constant__ CUtensorMap tmW, const uint8_t* __restrict__ W,
                           const float* __restrict__ x, int8_t* __restrict__ xq, float* __restrict__ xds,
                           float* __restrict__ out, int32_t* __restrict__ dots, int od, int K, int stages,
                           int* status, int static_w, int limit_ms, int skip_first) {
  using C = GemvCfg<QT, NW, R>;
  extern __shared__ uint8_t smem_dyn[];
  const uint32_t s0 = smem_addr(smem_dyn);
  const uint32_t pad = (1024u - (s0 & 1023u)) & 1023u;
  uint8_t* smem = smem_dyn + pad;
  const uint32_t sb = s0 + pad;

  const int nsb = K >> 8, nseg = (nsb + kSegSB - 1) / kSegSB;
  const int Kp = FUSED ? ((K + 2047) & ~2047) : K;  // per-token stride of the code plane
  const int act_q = NT * Kp;                         // int8 codes
  const int act_bytes = act_q + NT * (K >> 5) * 8;
  // rows staged by TMA boxes, or one by one (row_copy) when the matrix row
  // pitch is not a multiple of 16 bytes
  const bool row_copy = row_copy_needed(QT, K);
  const int srow = stage_row(QT, K), stage_bytes = C::CR * srow;
  const size_t row_bytes = (size_t)nsb * C::BLK;
  const int act_off = stages * stage_bytes;
  const int bar_off = (act_off + act_bytes + 15) & ~15;
  const uint32_t full0 = sb + bar_off, empty0 = full0 + 8 * stages, act_bar = empty0 + 8 * stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + bar_off + 16 * stages + 8);
  int8_t* sx = reinterpret_cast<int8_t*>(smem + act_off);
  float* sds = reinterpret_cast<float*>(smem + act_off + act_q);

  // CR-row groups of this CTA: a balanced split of all groups of the matrix
  const int G = (od + C::CR - 1) / C::CR;
  const int g_begin = (int)((int64_t)G * blockIdx.x / gridDim.x);
  const int g_end = (int)((int64_t)G * (blockIdx.x + 1) / gridDim.x);
  const int nchunks = (g_end - g_begin) * nseg;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Guard g{abort_flag, status, global_ns() + (uint64_t)limit_ms * 1000000ull};

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, NW);
    }
    mbar_init(act_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // the next kernel may launch now: it waits for this grid before touching
  // anything this grid writes
  griddep_launch_dependents();

  if (warp == NW) {
    // ----------------------------------------------------------- producer
    // Lane 0 waits for free stages and issues the copies.  Rows staged one by
    // one (a row pitch that is not a multiple of 16 bytes) take one bulk copy
    // per row: there the whole warp runs the loop and lane r stages row r of
    // the stage, so that sixteen windows are computed and issued at once.
    const unsigned am = row_copy ? 0xffffffffu : 1u;  // the lanes in the loop
    if (nchunks > 0 && (lane == 0 || row_copy)) {
      if (!row_copy) prefetch_tmap(&tmW);
      if (!static_w) griddep_wait();
      int issued = 0, st = 0, ph = 0, seg = 0, grp = g_begin;
      bool act_issued = FUSED;
      for (int c = 0; c < nchunks; ++c) {
        if (c == stages && !act_issued) {
          // the first stages of weights are in flight; now the activations,
          // which the preceding kernel may still be writing
          if (lane == 0) {
            griddep_wait();
            mbar_arrive_expect_tx(act_bar, (uint32_t)act_bytes);
            bulk_load(sb + act_off, xq, (uint32_t)act_q, act_bar);
            bulk_load(sb + act_off + act_q, xds, (uint32_t)(act_bytes - act_q), act_bar);
          }
          act_issued = true;
        }
        if (!__all_sync(am, wait_bar(empty0 + 8 * st, ph ^ 1, g))) break;
        if (!(skip_first && c == 0)) {  // the stall test hook skips the first stage
          if (!row_copy) {
            mbar_arrive_expect_tx(full0 + 8 * st, (uint32_t)C::STAGE_BYTES);
            tma_load_2d(sb + st * C::STAGE_BYTES, &tmW, seg * (C::SEG_BYTES / 8), grp * C::CR, full0 + 8 * st);
          } else {
            // the stage's super-blocks of row `lane`, one window
            const int nbs = min(kSegSB, nsb - seg * kSegSB);
            const size_t total = (size_t)od * row_bytes;
            size_t a0 = 0, a1 = 0;
            if (lane < C::CR && grp * C::CR + lane < od) {
              const size_t start = (size_t)(grp * C::CR + lane) * row_bytes + (size_t)seg * C::SEG_BYTES;
              const RowWindow w = stage_row_window(start, start + (size_t)nbs * C::BLK, total,
                                                   smem + st * stage_bytes + lane * srow, W);
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
            if (a1 > a0) bulk_load(sb + st * stage_bytes + lane * srow, W + a0, (uint32_t)(a1 - a0), full0 + 8 * st);
          }
        }
        ++issued;
        if (++st == stages) {
          st = 0;
          ph ^= 1;
        }
        if (++seg == nseg) {
          seg = 0;
          ++grp;
        }
      }
      if (lane == 0) {
        if (!act_issued) {
          griddep_wait();
          mbar_arrive_expect_tx(act_bar, (uint32_t)act_bytes);
          bulk_load(sb + act_off, xq, (uint32_t)act_q, act_bar);
          bulk_load(sb + act_off + act_q, xds, (uint32_t)(act_bytes - act_q), act_bar);
        }
        // drain: every copy in flight lands before the CTA exits
        const uint64_t dl = global_ns() + 1000000000ull;
        for (int i = issued - stages; i < issued; ++i) {
          if (i < 0 || (skip_first && i == 0)) continue;
          for (uint32_t it = 0; !mbar_try_wait(full0 + 8 * (i % stages), (i / stages) & 1); ++it)
            if ((it & 63u) == 63u && global_ns() > dl) break;
        }
        if (!FUSED)
          for (uint32_t it = 0; !mbar_try_wait(act_bar, 0); ++it)
            if ((it & 63u) == 63u && global_ns() > dl) break;
      }
    }
  } else if (nchunks > 0) {
    // ----------------------------------------------------------- consumers
    const int sbo = lane >> 2, p = lane & 3;
    const Q4PairDecode q4d(p);
    // this lane's first block in a stage: row warp*R of the stage, super-block sbo
    const int lane_w = QT == kQ4 ? (warp * R) * C::SEG_BYTES + sbo * kQ4KBytes : 0;
    bool ok = true;
    // the preceding grid is complete before any consumer reads x or writes:
    // one warp waits for it, the others sleep on a named barrier meanwhile
    if (warp == 0) {
      griddep_wait();
      named_arrive(2, 32 * NW);
    } else {
      named_barrier(2, 32 * NW);
    }
    if (FUSED) {
      // q8_1 of x [NT][K] into shared memory: eight lanes per 32-value block,
      // four values per lane; block maximum and code sum by shuffles within
      // the eight lanes; d = amax/127 and q = round-half-even(x/d) by IEEE
      // division, s = d*(float)sum(q).  CTA (b mod grid) also writes block b
      // of the xq / xds outputs.
      const int nblk = NT * (K >> 5), nbk = K >> 5;
      const int tid = warp * 32 + lane, half = lane & 1;
      // two lanes per 32-value block, sixteen values (four 16-byte loads) each:
      // the decode shapes (nt = 1, K <= 4096) take a single pass
      for (int it = 0; it * 16 * NW < nblk; ++it) {
        const int b = it * 16 * NW + (tid >> 1);
        const bool in = b < nblk;
        const float4* src = reinterpret_cast<const float4*>(x + (size_t)b * 32 + 16 * half);
        float v[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 t4 = in ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
          v[4 * i] = t4.x;
          v[4 * i + 1] = t4.y;
          v[4 * i + 2] = t4.z;
          v[4 * i + 3] = t4.w;
        }
        float m[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m[i] = fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
#pragma unroll
        for (int w2 = 4; w2 > 0; w2 >>= 1)
#pragma unroll
          for (int i = 0; i < w2; ++i) m[i] = fmaxf(m[i], m[i + w2]);
        const float amax = fmaxf(m[0], __shfl_xor_sync(0xffffffffu, m[0], 1));
        const float d = __fdiv_rn(amax, 127.0f);
        uint32_t cw[16];
        q8_code_words<16>(v, d, cw);
        // pack the codes and sum them (a signed-byte dp4a against ones)
        int sum = 0;
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pk[i] = pack_low_bytes(cw[4 * i], cw[4 * i + 1], cw[4 * i + 2], cw[4 * i + 3]);
          sum = __dp4a((int)pk[i], 0x01010101, sum);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        const float s = __fmul_rn(d, (float)sum);
        if (in) {
          // codes k..k+15 are one contiguous 16-byte chunk of the plane
          const int t = b / nbk, kb = b - t * nbk;
          *reinterpret_cast<uint4*>(sx + t * Kp + fused_code_offset(kb * 32 + 16 * half)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
          if (half == 0) *reinterpret_cast<float2*>(sds + 2 * b) = make_float2(d, s);
          if (blockIdx.x == 0) {  // one CTA writes the q8_1 outputs
            *reinterpret_cast<uint4*>(xq + (size_t)b * 32 + 16 * half) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            if (half == 0) reinterpret_cast<float2*>(xds)[b] = make_float2(d, s);
          }
        }
      }
      named_barrier(1, 32 * NW);
    } else {
      ok = __all_sync(0xffffffffu, wait_bar(act_bar, 0, g));
    }
    float acc[R][NT];
    int st = 0, ph = 0, seg = 0, grp = g_begin;
    for (int c = 0; c < nchunks && ok; ++c) {
      if (seg == 0) {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[i][t] = 0.0f;
      }
      ok = __all_sync(0xffffffffu, wait_bar(full0 + 8 * st, ph, g));
      if (!ok) break;
      const int sbi = seg * kSegSB + sbo;  // super-block of this lane
      const bool live = sbi < nsb;
      const int kbase = sbi * 256 + 64 * p;
      const int jlo = sbi * 8 + 2 * p;
      const int row0 = grp * C::CR + warp * R;
      if constexpr (QT == kQ4) {
      // the R weight rows of this lane: nibbles split into the low (sub-block
      // 2p) and high (sub-block 2p+1) planes, and the four scale factors
      const uint8_t* stage = smem + st * stage_bytes + lane_w;
      uint32_t lo[R][8], hi[R][8];
      float a_lo[R], a_hi[R], c_lo[R], c_hi[R];
      // a whole stage -- all R rows in the matrix, the segment's 8 super-
      // blocks in the row -- takes unpredicated loads (every stage but the
      // last of a ragged matrix)
      const bool whole = row0 + R <= od && (seg + 1) * kSegSB <= nsb;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        uint4 hdr, q0, q1;
        const uint8_t* blk = stage + i * C::SEG_BYTES;
        if (whole) {
          hdr = *reinterpret_cast<const uint4*>(blk);
          q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * p);
          q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * p);
        } else {
          hdr = q0 = q1 = make_uint4(0, 0, 0, 0);
          if (live && row0 + i < od) {
            hdr = *reinterpret_cast<const uint4*>(blk);
            q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * p);
            q1 = *reinterpret_cast<const uint4*>(blk + 32 + 32 * p);
          }
        }
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          lo[i][k] = w[k] & 0x0F0F0F0Fu;
          hi[i][k] = w[k] & 0xF0F0F0F0u;  // 16 x the high nibbles: one AND instead of a shift and an AND
        }
        uint32_t sc2, m2;
        q4d.codes(hdr.y, hdr.z, hdr.w, sc2, m2);
        const float2 dd = __half22float2(*reinterpret_cast<const __half2*>(&hdr.x));  // (d, dmin)
        // d * sc and dmin * m are exact in f32; the high-nibble dot comes out
        // 16x, so its factor carries 1/16 (an exact power of 2)
        const float dq = dd.x * 0.0625f;
        a_lo[i] = fmaf(dd.x, magic_byte(sc2, 0), -0x1p23f * dd.x);
        a_hi[i] = fmaf(dq, magic_byte(sc2, 1), -0x1p23f * dq);
        c_lo[i] = fmaf(dd.y, magic_byte(m2, 0), -0x1p23f * dd.y);
        c_hi[i] = fmaf(dd.y, magic_byte(m2, 1), -0x1p23f * dd.y);
      }
      // the stage's words are in registers: hand it back before the dots
      release_stage(empty0 + 8 * st);
      if (live) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          // activation slice of token t: 64 codes and the two (d, s) pairs
          uint4 x0, x1, x2, x3;
          if (FUSED) {
            const uint4* px = reinterpret_cast<const uint4*>(sx + t * Kp) + seg * 128 + lane;
            x0 = px[0];
            x1 = px[32];
            x2 = px[64];
            x3 = px[96];
          } else {
            const uint4* px = reinterpret_cast<const uint4*>(sx + t * K + kbase);
            x0 = px[0];
            x1 = px[1];
            x2 = px[2];
            x3 = px[3];
          }
          const float4 xs = *reinterpret_cast<const float4*>(sds + (t * (K >> 5) + jlo) * 2);
          const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          const uint32_t yw[8] = {x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
#pragma unroll
          for (int i = 0; i < R; ++i) {
            int dlo = 0, dhi = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              dlo = __dp4a((int)lo[i][k], (int)xw[k], dlo);
              dhi = dp4a_us(hi[i][k], yw[k], dhi);
            }
            if constexpr (DOTS) {
              if (row0 + i < od) {
                int32_t* dst = dots + ((size_t)t * od + row0 + i) * (K >> 5) + jlo;
                dst[0] = dlo;
                dst[1] = dhi >> 4;  // a multiple of 16: exact
              }
            } else {
              float a = acc[i][t];
              a = fmaf(a_lo[i] * xs.x, (float)dlo, a);
              a = fmaf(a_hi[i] * xs.z, (float)dhi, a);
              a = fmaf(-c_lo[i], xs.y, a);
              a = fmaf(-c_hi[i], xs.w, a);
              acc[i][t] = a;
            }
          }
        }
      }
      } else {
      const uint8_t* stage = smem + st * stage_bytes;
      // Q6_K: the lane's 64 values are quads 2(p%2), 2(p%2)+1 of half n = p/2:
      // low 4 bits from ql[64n + l] / ql[64n + 32 + l] (low nibbles for even p,
      // high for odd p), top 2 bits from qh[32n + l] (bits 0-1 / 2-3 for even p,
      // 4-5 / 6-7 for odd p); value q - 32, scale scales[4p + j] per 16 values.
      // The blocks are 2 bytes aligned: words are read realigned.
      const int n = p >> 1;
      const uint32_t shl = (p & 1) ? 4u : 0u, shh = (p & 1) ? 0u : 4u;
      uint32_t qa[R][8], qb[R][8];
      float scl[R][4];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const bool use = live && row0 + i < od;
        uint32_t L0[8] = {}, L1[8] = {}, H[8] = {}, sw[1] = {0};
        uint32_t dbits = 0;
        if (use) {
          const uint8_t* rowp = stage + (warp * R + i) * srow;  // 16-byte aligned
          // even: the row's blocks start at its window's offset (0 for TMA boxes)
          const int boff = (row_copy ? (int)(((size_t)(row0 + i) * row_bytes + (size_t)seg * C::SEG_BYTES) & 15) : 0) +
                           sbo * kQ6KBytes;
          // (the lanes' blocks alternate between 4- and 2-byte alignment:
          // branch-free realignment.  The extra word each run reads stays
          // inside the stage row: the furthest, after the scale word of block
          // 7, ends on byte 1680 of a 1680-byte TMA row, or at most 14 bytes
          // later inside the 32 spare bytes of a row staged as a window)
          load_words_even_bf<8>(rowp, boff + 64 * n, L0);
          load_words_even_bf<8>(rowp, boff + 64 * n + 32, L1);
          load_words_even_bf<8>(rowp, boff + 128 + 32 * n, H);
          load_words_even_bf<1>(rowp, boff + 192 + 4 * p, sw);
          dbits = *reinterpret_cast<const uint16_t*>(rowp + boff + 208);
        }
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const uint32_t h = H[w] << shh;
          qa[i][w] = ((L0[w] >> shl) & 0x0F0F0F0Fu) | (h & 0x30303030u);
          qb[i][w] = ((L1[w] >> shl) & 0x0F0F0F0Fu) | ((h >> 2) & 0x30303030u);
        }
        const float d = half_bits_to_float(dbits);
#pragma unroll
        for (int j = 0; j < 4; ++j) scl[i][j] = d * (float)(int8_t)((sw[0] >> (8 * j)) & 0xFFu);
      }
      // the stage's words are in registers: hand it back before the dots
      release_stage(empty0 + 8 * st);
      if (live) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          uint4 x0, x1, x2, x3;
          if (FUSED) {
            const uint4* px = reinterpret_cast<const uint4*>(sx + t * Kp) + seg * 128 + lane;
            x0 = px[0];
            x1 = px[32];
            x2 = px[64];
            x3 = px[96];
          } else {
            const uint4* px = reinterpret_cast<const uint4*>(sx + t * K + kbase);
            x0 = px[0];
            x1 = px[1];
            x2 = px[2];
            x3 = px[3];
          }
          const float4 xs = *reinterpret_cast<const float4*>(sds + (t * (K >> 5) + jlo) * 2);
          const uint32_t xw[16] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w,
                                   x2.x, x2.y, x2.z, x2.w, x3.x, x3.y, x3.z, x3.w};
          // 32 x the code sum of each 16-value group: the -32 of q - 32
          int s32[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            int sj = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) sj = __dp4a(0x01010101, (int)xw[4 * j + k], sj);
            s32[j] = 32 * sj;
          }
#pragma unroll
          for (int i = 0; i < R; ++i) {
            int dj[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              int v = -s32[j];
#pragma unroll
              for (int k = 0; k < 4; ++k) v = dp4a_us(j < 2 ? qa[i][4 * j + k] : qb[i][4 * (j - 2) + k], xw[4 * j + k], v);
              dj[j] = v;  // sum over the group of (q - 32) * x
            }
            if constexpr (DOTS) {
              if (row0 + i < od) {
                int32_t* dst = dots + ((size_t)t * od + row0 + i) * (K >> 4) + sbi * 16 + 4 * p;
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[j] = dj[j];
              }
            } else {
              float a = acc[i][t];
              a = fmaf(scl[i][0] * xs.x, (float)dj[0], a);
              a = fmaf(scl[i][1] * xs.x, (float)dj[1], a);
              a = fmaf(scl[i][2] * xs.z, (float)dj[2], a);
              a = fmaf(scl[i][3] * xs.z, (float)dj[3], a);
              acc[i][t] = a;
            }
          }
        }
      }
      }
      if (!DOTS && seg == nseg - 1) {
        // reduce the R x NT partial sums over the warp; lane i*NT+t stores (row i, token t)
        float mine = 0.0f;
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            float v = acc[i][t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == i * NT + t) mine = v;
          }
        if (lane < R * NT) {
          const int i = lane / NT, t = lane % NT;
          if (row0 + i < od) out[(size_t)t * od + row0 + i] = mine;
        }
      }
      if (++st == stages) {
        st = 0;
        ph ^= 1;
      }
      if (++seg == nseg) {
        seg = 0;
        ++grp;
      }
    }
  }
  __syncthreads();
}

struct GemvArgs {
  const void* W;
  const float* x;  // fused path
  int8_t* xq;      // staged path: input; fused path: output
  float* xds;      // likewise
  float* out;
  int32_t* dots;
  int64_t od, K;
  int* status;
  bool pdl, static_w;
  cudaStream_t stream;
};

template <int QT, int NT, int NW, int R, bool DOTS, bool FUSED>
int launch_stream(const GemvArgs& a, int stages) {
  using C = GemvCfg<QT, NW, R>;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QMM_EDEVICE;
  cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
  const int64_t act_bytes = FUSED ? fused_act_bytes(NT, a.K) : act_bytes_of(NT, a.K);
  const int smem = stages * C::CR * stage_row(QT, a.K) + (int)((act_bytes + 15) & ~15) + 16 * stages + 32 + 1024;
  auto kern = mmvq_stream_kernel<QT, NT, NW, R, DOTS, FUSED>;
  static PerDevice<bool> attr_done;
  if (int rc = smem_attr_once(kern, kSmemBudget + 8192, attr_done, dev)) return rc;
  if (smem > kSmemBudget + 8192) return QMM_ESMEM;
  auto fn = tensor_map_encoder();
  if (!fn) return QMM_ELAUNCH;
  // W viewed as [od][row_bytes/8] 8-byte elements; one box = CR rows x 8 super-blocks
  const uint64_t row_bytes = (uint64_t)(a.K / 256) * C::BLK;
  CUtensorMap m = {};
  const cuuint64_t dims[2] = {row_bytes / 8, (cuuint64_t)a.od};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {C::SEG_BYTES / 8, (cuuint32_t)C::CR};
  const cuuint32_t estr[2] = {1, 1};
  // rows whose pitch is not a multiple of 16 bytes are staged by the kernel
  // itself, one window per row
  if (!row_copy_needed(QT, a.K) &&
      fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void*>(a.W), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return QMM_ELAUNCH;
  const int groups = (int)((a.od + C::CR - 1) / C::CR);
  int grid = nsm > 0 ? nsm : 152;
  // One CTA per SM leaves room for a CTA of the next kernel, which then
  // starts its weight stream early.  Q6_K on many row groups (the LM head)
  // runs two instead: its consumers spend more instructions per weight, and
  // twice the warps hide more of their latency (32000 x 4096: 26.1 -> 21.9
  // us).  Q4_K measured slower that way (11008 x 4096: 6.2 -> 7.2 us).
  if (FUSED && QT == kQ6 && groups >= 4 * grid) grid *= 2;
  if (grid > groups) grid = groups;
  const int iod = (int)a.od, iK = (int)a.K, sw = a.static_w ? 1 : 0;
  const int stall = stall_ms();
  return launch_ex(kern, dim3(grid), dim3(C::THREADS), (size_t)smem, a.stream, a.pdl, m,
                   static_cast<const uint8_t*>(a.W), a.x, a.xq, a.xds,
                   a.out, a.dots, iod, iK, stages, a.status, sw, stall > 0 ? stall : 4000, stall > 0 ? 1 : 0);
}

// Staged path: consumer warps and rows per warp by nt -- 16 warps of one row
// for nt <= 2, 16 warps of two rows for nt <= 4, 8 warps of four rows above
// (the rows of a warp share its activation registers); fewer rows when the
// activations leave too little shared memory for a 3-stage ring.  DOTS (a
// test hook) uses 16 x 1.
template <int QT, int NT, bool DOTS>
int launch_staged(const GemvArgs& a) {
  constexpr int NW = (DOTS || NT <= 4) ? 16 : 8;
  constexpr int RP = DOTS ? 1 : (NT <= 2 ? 1 : (NT <= 4 ? 2 : 4));
  int st = stages_for(QT, NT, a.K, NW * RP, kSmemBudget);
  if (st >= 3) return launch_stream<QT, NT, NW, RP, DOTS, false>(a, st);
  if constexpr (RP >= 2) {
    st = stages_for(QT, NT, a.K, NW * (RP / 2), kSmemBudget);
    if (st >= 3) return launch_stream<QT, NT, NW, RP / 2, DOTS, false>(a, st);
  }
  st = stages_for(QT, NT, a.K, 8, kSmemBudget);
  if (st >= 2) return launch_stream<QT, NT, 8, 1, DOTS, false>(a, st);
  return QMM_ESMEM;
}

// Fused path: 8 consumer warps of two rows (a 16-row, 18 KB stage) and a
// ring of 3..5 stages next to the activations, so that a CTA of the next
// kernel fits on the SM next to this one.
template <int QT, int NT>
int launch_fused(const GemvArgs& a) {
  const int st = fused_stages(QT, NT, a.K);
  if (st == 0) return QMM_ESMEM;
  return launch_stream<QT, NT, 8, 2, false, true>(a, st);
}

template <int QT, bool DOTS>
int launch_staged_nt(const GemvArgs& a, int64_t nt) {
  switch (nt) {
    case 1: return launch_staged<QT, 1, DOTS>(a);
    case 2: return launch_staged<QT, 2, DOTS>(a);
    case 3: return launch_staged<QT, 3, DOTS>(a);
    case 4: return launch_staged<QT, 4, DOTS>(a);
    case 5: return launch_staged<QT, 5, DOTS>(a);
    case 6: return launch_staged<QT, 6, DOTS>(a);
    case 7: return launch_staged<QT, 7, DOTS>(a);
    case 8: return launch_staged<QT, 8, DOTS>(a);
    default: return QMM_EINVAL_SHAPE;
  }
}

// (from 5 tokens qmm_matmul takes the warp-MMA kernel instead)
template <int QT>
int launch_fused_nt(const GemvArgs& a, int64_t nt) {
  switch (nt) {
    case 1: return launch_fused<QT, 1>(a);
    case 2: return launch_fused<QT, 2>(a);
    case 3: return launch_fused<QT, 3>(a);
    case 4: return launch_fused<QT, 4>(a);
    default: return QMM_EINVAL_SHAPE;
  }
}

int qt_of(int qtype) { return qtype == QMM_Q4_K ? kQ4 : kQ6; }

// Both types at any K % 256 (Q6_K rows with a pitch that is not a multiple of
// 16 bytes are staged row by row).
bool gemv_type_ok(int qtype, int64_t K) {
  (void)K;
  return qtype == QMM_Q4_K || qtype == QMM_Q6_K;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

bool gemv_fits(int qtype, int64_t nt, int64_t K) {
  return gemv_type_ok(qtype, K) && nt >= 1 && nt <= 8 && stages_for(qt_of(qtype), nt, K, 8, kSmemBudget) >= 2;
}

bool gemv_fused_fits(int qtype, int64_t nt, int64_t K) {
  return gemv_type_ok(qtype, K) && nt >= 1 && nt <= 4 && fused_stages(qt_of(qtype), nt, K) > 0;
}

int launch_gemv(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots,
                int64_t od, int64_t K, int64_t nt, int* status, Dep dep, cudaStream_t stream) {
  if (qtype != QMM_Q4_K && qtype != QMM_Q6_K) return QMM_EINVAL_QTYPE;
  if (!gemv_type_ok(qtype, K)) return QMM_EINVAL_SHAPE;
  // from a few tokens on the dots run on the warp-level tensor-core MMA
  if (!dots && (nt > 8 || nt >= mma_min_nt(qtype)) && mmvq_mma_fits(qtype, nt, K))
    return launch_mmvq_mma(qtype, W, xq, xds, out, nullptr, od, K, nt, status, dep, stream);
  if (!gemv_fits(qtype, nt, K)) return QMM_ESMEM;
  const GemvArgs a{W,      nullptr, const_cast<int8_t*>(xq), const_cast<float*>(xds), out, dots, od, K, status,
                   dep != Dep::kNone, dep == Dep::kPdlStaticW, stream};
  if (qtype == QMM_Q4_K)
    return dots ? launch_staged_nt<kQ4, true>(a, nt) : launch_staged_nt<kQ4, false>(a, nt);
  return dots ? launch_staged_nt<kQ6, true>(a, nt) : launch_staged_nt<kQ6, false>(a, nt);
}

int launch_gemv_fused(int qtype, const void* W, const float* x, int8_t* xq, float* xds, float* out, int64_t od,
                      int64_t K, int64_t nt, int* status, bool static_w, cudaStream_t stream) {
  if (qtype != QMM_Q4_K && qtype != QMM_Q6_K) return QMM_EINVAL_QTYPE;
  if (!gemv_fused_fits(qtype, nt, K)) return QMM_ESMEM;
  const GemvArgs a{W, x, xq, xds, out, nullptr, od, K, status, true, static_w, stream};
  return qtype == QMM_Q4_K ? launch_fused_nt<kQ4>(a, nt) : launch_fused_nt<kQ6>(a, nt);
}

}  // namespace qmm
