// qmm_gemv.cu -- MMVQ: the small-batch (nt <= 8) Q4_K x q8_1 matmul.
//
// Design ("04 - Reading minfer's kernels II", sec. 3.4; "llama.cpp MMQ",
// sec. 12.2): the weight matrix is streamed from HBM exactly once, with
// 16-byte coalesced loads, and every weight block is dotted against all nt
// tokens, whose accumulators live in registers -- the token count never
// multiplies the weight traffic.  The dots are exact int32 (dp4a over
// nibbles and int8 codes); the scales fold in once per 32-value sub-block:
//     acc += d*sc_j*dx_j*D_j - dmin*m_j*s_j
// ("The quantized GEMM", "The GPU path").
//
// Mapping: one warp per weight row.  Lane l handles 16-byte chunk (l & 7) of
// the 128 nibble bytes of super-block 4*i + (l >> 3) in iteration i, so one
// warp instruction reads four consecutive super-blocks' nibbles (512 B) plus
// their 16-byte headers (one broadcast load per 8 lanes).  Chunk c holds
// bytes 16c..16c+15 of the nibble array: pair p = c/2, half h = c%2, i.e.
// elements 64p+16h.. (low nibbles, sub-block 2p) and 64p+32+16h.. (high
// nibbles, sub-block 2p+1).
#include <cuda_runtime.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int NT, bool DOTS>
__global__ void __launch_bounds__(256) gemv_q4k_kernel(const uint8_t* __restrict__ W,
                                                       const int8_t* __restrict__ xq,
                                                       const float* __restrict__ xds,
                                                       float* __restrict__ out, int32_t* __restrict__ dots,
                                                       int od, int K) {
  constexpr int U = 4;  // iterations whose weight loads are issued together
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= od) return;
  const int lane = threadIdx.x & 31;
  const int sbl = lane >> 3, c = lane & 7, p = c >> 1, h = c & 1;
  const int nsb = K >> 8;
  const int nb32 = K >> 5;
  const uint8_t* wrow = W + (size_t)row * nsb * kQ4KBytes;

  float acc[NT];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.0f;

  const int iters = (nsb + 3) >> 2;
  for (int i0 = 0; i0 < iters; i0 += U) {
    uint4 hdr[U], qs[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int sb = (i0 + u) * 4 + sbl;
      if (i0 + u < iters && sb < nsb) {
        const uint8_t* blk = wrow + (size_t)sb * kQ4KBytes;
        hdr[u] = ldg_nc_v4(blk);
        qs[u] = ldg_nc_v4(blk + 16 + 16 * c);
      } else {
        hdr[u] = make_uint4(0, 0, 0, 0);
        qs[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int sb = (i0 + u) * 4 + sbl;
      const bool live = (i0 + u < iters) && sb < nsb;
      int sc_lo, m_lo, sc_hi, m_hi;
      q4k_scale_min_words(hdr[u].y, hdr[u].z, hdr[u].w, 2 * p, sc_lo, m_lo);
      q4k_scale_min_words(hdr[u].y, hdr[u].z, hdr[u].w, 2 * p + 1, sc_hi, m_hi);
      const float d = half_bits_to_float(hdr[u].x);
      const float dmin = half_bits_to_float(hdr[u].x >> 16);
      const float a_lo = d * (float)sc_lo, a_hi = d * (float)sc_hi;
      // the min term of a sub-block is added once, by the lane holding its first half
      const float mm = h == 0 ? dmin : 0.0f;
      const float c_lo = mm * (float)m_lo, c_hi = mm * (float)m_hi;
      const uint32_t w[4] = {qs[u].x, qs[u].y, qs[u].z, qs[u].w};
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        lo[k] = w[k] & 0x0F0F0F0Fu;
        hi[k] = (w[k] >> 4) & 0x0F0F0F0Fu;
      }
      const int k_lo = sb * 256 + 64 * p + 16 * h;
      const int j_lo = sb * 8 + 2 * p;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        int dlo = 0, dhi = 0;
        if (live) {
          const int8_t* xt = xq + (size_t)t * K;
          const int4 xl = __ldg(reinterpret_cast<const int4*>(xt + k_lo));
          const int4 xh = __ldg(reinterpret_cast<const int4*>(xt + k_lo + 32));
          dlo = __dp4a((int)lo[0], xl.x, dlo);
          dlo = __dp4a((int)lo[1], xl.y, dlo);
          dlo = __dp4a((int)lo[2], xl.z, dlo);
          dlo = __dp4a((int)lo[3], xl.w, dlo);
          dhi = __dp4a((int)hi[0], xh.x, dhi);
          dhi = __dp4a((int)hi[1], xh.y, dhi);
          dhi = __dp4a((int)hi[2], xh.z, dhi);
          dhi = __dp4a((int)hi[3], xh.w, dhi);
        }
        if constexpr (DOTS) {
          // the two halves of each sub-block sit in lanes c and c^1
          const int flo = dlo + __shfl_xor_sync(0xffffffffu, dlo, 1);
          const int fhi = dhi + __shfl_xor_sync(0xffffffffu, dhi, 1);
          if (live && h == 0) {
            int32_t* dst = dots + ((size_t)t * od + row) * nb32 + j_lo;
            dst[0] = flo;
            dst[1] = fhi;
          }
        } else if (live) {
          const float4 sx = __ldg(reinterpret_cast<const float4*>(xds + ((size_t)t * nb32 + j_lo) * 2));
          acc[t] = fmaf(a_lo * sx.x, (float)dlo, acc[t]);
          acc[t] = fmaf(a_hi * sx.z, (float)dhi, acc[t]);
          acc[t] = fmaf(-c_lo, sx.y, acc[t]);
          acc[t] = fmaf(-c_hi, sx.w, acc[t]);
        }
      }
    }
  }
  if constexpr (!DOTS) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      float v = acc[t];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      acc[t] = v;
    }
    if (lane < NT) {
      float v = acc[0];
#pragma unroll
      for (int t = 1; t < NT; ++t)
        if (lane == t) v = acc[t];
      out[(size_t)lane * od + row] = v;
    }
  }
}

template <bool DOTS>
static int launch_q4k(const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots,
                      int64_t od, int64_t K, int64_t nt, cudaStream_t stream) {
  const dim3 grid((unsigned)((od + 7) / 8)), block(256);
  const uint8_t* w = static_cast<const uint8_t*>(W);
  switch (nt) {
#define QMM_GEMV_CASE(N) \
  case N: gemv_q4k_kernel<N, DOTS><<<grid, block, 0, stream>>>(w, xq, xds, out, dots, (int)od, (int)K); break;
    QMM_GEMV_CASE(1)
    QMM_GEMV_CASE(2)
    QMM_GEMV_CASE(3)
    QMM_GEMV_CASE(4)
    QMM_GEMV_CASE(5)
    QMM_GEMV_CASE(6)
    QMM_GEMV_CASE(7)
    QMM_GEMV_CASE(8)
#undef QMM_GEMV_CASE
    default: return QMM_EINVAL_SHAPE;
  }
  return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ELAUNCH;
}

int launch_gemv(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots,
                int64_t od, int64_t K, int64_t nt, int* status, cudaStream_t stream) {
  (void)status;
  if (qtype != QMM_Q4_K) return QMM_EINVAL_QTYPE;
  return dots ? launch_q4k<true>(W, xq, xds, out, dots, od, K, nt, stream)
              : launch_q4k<false>(W, xq, xds, out, dots, od, K, nt, stream);
}

}  // namespace qmm
