// qmm_quantize.cu -- q8_1 activation quantizer and the tensor-core GEMM's
// activation-operand prepass.
//
// q8_1 ("The quantized GEMM", mojo-dllm, section "The GPU path"): per
// 32-value block the maximum |x| and the integer sum of the codes are
// warp-shuffle reductions; d = amax/127 by IEEE f32 division; the code is
// round-half-even of the IEEE quotient x/d; s = d * sum(q).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qmm_device.cuh"
#include "qmm_internal.h"

namespace qmm {

// bf16 bits of v rounded to nearest even (v finite).
__device__ __forceinline__ uint32_t bf16_rn_bits(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

// Scale planes of one (token t, block j) for the tensor-core GEMM: d into
// the dx plane, and s = s0 + s1 + s2 exactly as three bf16 (each part takes
// the next 8 significant bits of the remainder: the remainders are exact in
// f32 and the third part holds the last at most 8 bits) into the min-term
// planes, chunk 3 zero.
__device__ __forceinline__ void write_gemm_scales(float* scl, int64_t nb, int64_t ntp, int64_t t, int64_t j,
                                                  float d, float s) {
  scl[j * ntp + t] = d;
  uint16_t* sm = reinterpret_cast<uint16_t*>(scl + nb * ntp);
  const uint32_t p0 = bf16_rn_bits(s);
  const float r0 = s - __uint_as_float(p0 << 16);
  const uint32_t p1 = bf16_rn_bits(r0);
  const uint32_t p2 = bf16_rn_bits(r0 - __uint_as_float(p1 << 16));
  const int64_t base = ((j >> 3) * 4 * ntp + t) * 8 + (j & 7);  // chunk 0 of super-block j/8
  sm[base] = (uint16_t)p0;
  sm[base + ntp * 8] = (uint16_t)p1;
  sm[base + 2 * ntp * 8] = (uint16_t)p2;
  sm[base + 3 * ntp * 8] = 0;
}

// Eight lanes per 32-value block, four values per lane (one 16-byte load);
// a warp takes four blocks per step, grid-stride over all nt*K/32 blocks.
// The block maximum and the code sum are 3-step shuffle reductions within the
// eight lanes; d = amax/127 by IEEE division, the codes by q8_code_words (the
// same integers IEEE division and round-half-even give), s = d * sum(q).
// When xh / scl are non-null the same pass also writes the tensor-core GEMM
// operands (the workspace layout of qmm_internal.h): the codes as exact f16
// (xh [nt][K]), d token-contiguous (scl [K/32][ntp]) and s as three bf16
// parts for the min-term MMA.
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const float* __restrict__ x, int64_t nblocks,
                                                            int64_t nb_per_row, int8_t* __restrict__ xq,
                                                            float2* __restrict__ xds,
                                                            __half* __restrict__ xh,
                                                            float* __restrict__ scl, int64_t ntp) {
  const int lane = threadIdx.x & 31, q8 = lane & 7;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  // wait until the preceding grid is done (it may write x or read xq / xds),
  // then let the next kernel -- the matmul -- start streaming its weights:
  // everything enqueued before this grid is complete at that point
  griddep_wait();
  griddep_launch_dependents();
  for (int64_t b0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 4; b0 < nblocks;
       b0 += warps * 4) {
    const int64_t b = b0 + (lane >> 3);
    const bool in = b < nblocks;
    const float4 v4 = in ? __ldg(reinterpret_cast<const float4*>(x + b * 32) + q8) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float d = __fdiv_rn(amax, 127.0f);
    uint32_t cw[4];
    q8_code_words<4>(v, d, cw);
    const uint32_t pk = pack_low_bytes(cw[0], cw[1], cw[2], cw[3]);
    int sum = __dp4a((int)pk, 0x01010101, 0);  // the four signed codes
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    const float s = __fmul_rn(d, (float)sum);
    if (in) {
      *reinterpret_cast<uint32_t*>(xq + b * 32 + 4 * q8) = pk;
      if (xh) {
        const int q[4] = {(int)(int8_t)(cw[0] & 0xFFu), (int)(int8_t)(cw[1] & 0xFFu), (int)(int8_t)(cw[2] & 0xFFu),
                          (int)(int8_t)(cw[3] & 0xFFu)};
        const __half2 h01 = __halves2half2(__int2half_rn(q[0]), __int2half_rn(q[1]));
        const __half2 h23 = __halves2half2(__int2half_rn(q[2]), __int2half_rn(q[3]));
        *reinterpret_cast<uint2*>(xh + b * 32 + 4 * q8) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
      }
      if (q8 == 0) {
        xds[b] = make_float2(d, s);
        if (scl) write_gemm_scales(scl, nb_per_row, ntp, b / nb_per_row, b % nb_per_row, d, s);
      }
    }
  }
}

// Prepass for qmm_gemm when the caller already holds xq / xds: 16 codes per
// thread to f16, and the scale planes (as the quantizer writes them).
__global__ void __launch_bounds__(256) gemm_operand_prep_kernel(const int8_t* __restrict__ xq,
                                                                const float2* __restrict__ xds, int64_t nt,
                                                                int64_t K, int64_t ntp,
                                                                __half* __restrict__ xh,
                                                                float* __restrict__ scl) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n16 = nt * K / 16;
  for (int64_t i = tid; i < n16; i += stride) {
    const int4 v = __ldg(reinterpret_cast<const int4*>(xq) + i);
    const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 lo = __halves2half2(__int2half_rn((int8_t)(w[k] & 0xFF)),
                                        __int2half_rn((int8_t)((w[k] >> 8) & 0xFF)));
      const __half2 hi = __halves2half2(__int2half_rn((int8_t)((w[k] >> 16) & 0xFF)),
                                        __int2half_rn((int8_t)((w[k] >> 24) & 0xFF)));
      h[2 * k] = *reinterpret_cast<const uint32_t*>(&lo);
      h[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&hi);
    }
    int4* dst = reinterpret_cast<int4*>(xh) + 2 * i;
    dst[0] = make_int4((int)h[0], (int)h[1], (int)h[2], (int)h[3]);
    dst[1] = make_int4((int)h[4], (int)h[5], (int)h[6], (int)h[7]);
  }
  const int64_t nb = K / 32;
  const int64_t nscl = nt * nb;
  for (int64_t i = tid; i < nscl; i += stride) {
    const int64_t t = i / nb, j = i % nb;
    const float2 ds = __ldg(xds + i);
    write_gemm_scales(scl, nb, ntp, t, j, ds.x, ds.y);
  }
}

static int grid_for(int64_t work_items, int per_block) {
  int64_t g = (work_items + per_block - 1) / per_block;
  const int64_t cap = 152LL * 16;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

int launch_quantize(const float* x, int64_t nt, int64_t K, int8_t* xq, float* xds, __half* xh,
                    float* scl, int64_t ntp, cudaStream_t stream) {
  const int64_t nblocks = nt * (K / 32);
  if (nblocks == 0) return QMM_OK;
  return launch_ex(quantize_q8_1_kernel, dim3(grid_for(nblocks, 32)), dim3(256), 0, stream, true, x, nblocks,
                    (int64_t)(K / 32), xq, reinterpret_cast<float2*>(xds), xh, scl, ntp);
}

int launch_gemm_prep(const int8_t* xq, const float* xds, int64_t nt, int64_t K, int64_t ntp, __half* xh,
                     float* scl, cudaStream_t stream) {
  const int64_t work = nt * K / 16;
  gemm_operand_prep_kernel<<<grid_for(work, 256), 256, 0, stream>>>(
      xq, reinterpret_cast<const float2*>(xds), nt, K, ntp, xh, scl);
  return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ELAUNCH;
}

}  // namespace qmm
