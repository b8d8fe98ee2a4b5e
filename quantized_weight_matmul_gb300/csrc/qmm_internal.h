// qmm_internal.h -- launchers shared between the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qmm.h"

namespace qmm {

// Layout of the tensor-core GEMM workspace: f16 codes [nt][K], then the
// token-contiguous scale rows [K/32][ntp] float2.  ntp pads nt to a whole
// number of the widest token tile so every bulk copy stays in bounds.
constexpr int64_t kMaxTokenTile = 256;
inline int64_t gemm_ntp(int64_t nt) { return (nt + kMaxTokenTile - 1) / kMaxTokenTile * kMaxTokenTile; }
inline size_t gemm_xh_bytes(int64_t nt, int64_t K) {
  return (size_t)((nt * K * 2 + 255) / 256 * 256);
}
inline size_t gemm_scl_bytes(int64_t nt, int64_t K) { return (size_t)(K / 32) * gemm_ntp(nt) * 8; }

int launch_quantize(const float* x, int64_t nt, int64_t K, int8_t* xq, float* xds, __half* xh,
                    float* scl, int64_t ntp, cudaStream_t stream);
int launch_gemm_prep(const int8_t* xq, const float* xds, int64_t nt, int64_t K, int64_t ntp, __half* xh,
                     float* scl, cudaStream_t stream);

// MMVQ (nt <= 8).  dots != nullptr selects the raw block-dot output.
int launch_gemv(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots,
                int64_t od, int64_t K, int64_t nt, int* status, cudaStream_t stream);

// Tensor-core GEMM over the prepared workspace.  dots != nullptr selects the
// raw block-dot output (no scale folded into the weight operand).
int launch_gemm_tc(int qtype, const void* W, const __half* xh, const float* scl, float* out, int32_t* dots,
                   int64_t od, int64_t K, int64_t nt, int* status, int stall_ms, cudaStream_t stream);

}  // namespace qmm
