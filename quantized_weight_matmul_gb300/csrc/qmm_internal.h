// qmm_internal.h -- launchers shared between the library's translation units.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "qmm.h"

namespace qmm {

constexpr int kMaxDevices = 64;

// Per-device memo of a set-up step that is idempotent (a kernel's shared-memory
// attribute, a device symbol's address).  Several host threads may make their
// first call on a device at the same time: each may then run the step, but the
// slot is atomic, so a thread that sees it set also sees everything written
// before it was set.
template <typename T>
struct PerDevice {
  std::atomic<T> slot[kMaxDevices];
  T get(int dev) const { return slot[dev].load(std::memory_order_acquire); }
  void set(int dev, T v) { slot[dev].store(v, std::memory_order_release); }
};

// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, bytes) once per
// device (dev < kMaxDevices); QMM_ESMEM if the runtime refuses it.
template <typename Kern>
int smem_attr_once(Kern kern, int bytes, PerDevice<bool>& done, int dev) {
  if (dev < 0 || dev >= kMaxDevices) return QMM_EDEVICE;
  if (done.get(dev)) return QMM_OK;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return QMM_ESMEM;
  done.set(dev, true);
  return QMM_OK;
}

// Layout of the tensor-core GEMM workspace: f16 codes [nt][K]; the scale
// planes -- the token-contiguous dx rows [K/32][ntp] f32, then for the Q4_K
// min term the three bf16 parts of s per super-block [K/256][4][ntp][8]
// (chunk p < 3: part p of s for the super-block's 8 blocks; chunk 3: zero);
// then the split-K partial sums.  ntp pads nt to a whole number of the widest
// token tile so every bulk copy stays in bounds.
constexpr int64_t kMaxTokenTile = 256;
inline int64_t gemm_ntp(int64_t nt) { return (nt + kMaxTokenTile - 1) / kMaxTokenTile * kMaxTokenTile; }
inline size_t gemm_xh_bytes(int64_t nt, int64_t K) {
  return (size_t)((nt * K * 2 + 255) / 256 * 256);
}
inline size_t gemm_dx_bytes(int64_t nt, int64_t K) { return (size_t)(K / 32) * gemm_ntp(nt) * 4; }
inline size_t gemm_smin_bytes(int64_t nt, int64_t K) { return (size_t)(K / 256) * 4 * gemm_ntp(nt) * 16; }
inline size_t gemm_scl_bytes(int64_t nt, int64_t K) { return gemm_dx_bytes(nt, K) + gemm_smin_bytes(nt, K); }

// Split-K factor of the tensor-core GEMM, a function of the shape alone: a
// grid of fewer 128-row x token tiles than the 152 SMs of a GB300 takes its K
// range in up to 8 contiguous slices of whole super-blocks, one slice per
// CTA, so that about one full wave of CTAs runs.  The slices' fp32 partial
// sums go to the workspace and are added in a fixed order afterwards.
inline int gemm_splits(int64_t od, int64_t K, int64_t nt) {
  const int64_t bn = nt > 64 ? 128 : 64;
  const int64_t tiles = ((od + 127) / 128) * ((nt + bn - 1) / bn);
  const int64_t nsb = K / 256;
  int64_t s = 152 / (tiles > 0 ? tiles : 1);
  if (s > 8) s = 8;
  if (s > nsb) s = nsb;
  if (s < 1) s = 1;
  const int64_t per = (nsb + s - 1) / s;
  return (int)((nsb + per - 1) / per);  // every slice is non-empty
}
inline size_t gemm_part_bytes(int64_t od, int64_t K, int64_t nt) {
  const int s = gemm_splits(od, K, nt);
  return s > 1 ? (size_t)s * (size_t)nt * (size_t)od * sizeof(float) : 0;
}

// Launch `kern` on `stream`; with `pdl` as a programmatic dependent of the
// preceding kernel: it may start while that kernel drains and must call
// griddepcontrol.wait before touching memory the preceding kernel writes.
template <typename... KArgs, typename... Args>
int launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...) == cudaSuccess ? QMM_OK : QMM_ELAUNCH;
}

// Test hook (qmm_debug_inject_stall): milliseconds after which the bounded
// waits of the next launches give up, with the first producer arrival of each
// CTA skipped so that they do; 0 when off.
int stall_ms();

// The driver's cuTensorMapEncodeTiled, looked up once (nullptr if absent).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

int launch_quantize(const float* x, int64_t nt, int64_t K, int8_t* xq, float* xds, __half* xh,
                    float* scl, int64_t ntp, cudaStream_t stream);
int launch_gemm_prep(const int8_t* xq, const float* xds, int64_t nt, int64_t K, int64_t ntp, __half* xh,
                     float* scl, cudaStream_t stream);

// Whether the MMVQ kernel can stage nt x K activations next to its weight ring
// (Q4_K, or Q6_K with K a multiple of 2048).
bool gemv_fits(int qtype, int64_t nt, int64_t K);
// Whether the fused quantize + MMVQ kernel covers nt x K (decode shapes, nt <= 4).
bool gemv_fused_fits(int qtype, int64_t nt, int64_t K);

// How an MMVQ kernel is launched relative to the kernel before it on the
// stream.
enum class Dep {
  kNone,        // an ordinary launch
  kPdl,         // a programmatic dependent: every global access, the weight
                // stream included, waits for the preceding grid
  kPdlStaticW,  // a programmatic dependent whose weight stream may start
                // before the preceding grid completes (right after our
                // quantizer, which releases its dependents only once
                // everything before it is complete)
};

// MMVQ (nt <= 8).  dots != nullptr selects the raw block-dot output.
int launch_gemv(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots,
                int64_t od, int64_t K, int64_t nt, int* status, Dep dep, cudaStream_t stream);

// Warp-MMA MMVQ (qmm_mmvq_mma.cu) for 1 <= nt <= kMmaMaxNt: whether the
// activations and a weight ring of at least two stages fit one SM's shared
// memory (Q6_K also needs K % 2048 == 0), and the launcher.  dots != nullptr
// selects the raw block-dot output.
constexpr int kMmaMaxNt = 16;
// Smallest nt the warp-MMA kernel takes (below it the dp4a MMVQ is faster:
// its cost per token is small while the MMA's 8-token tile is mostly padding).
inline int mma_min_nt(int qtype) { return qtype == QMM_Q4_K ? 5 : 2; }
bool mmvq_mma_fits(int qtype, int64_t nt, int64_t K);
int launch_mmvq_mma(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots,
                    int64_t od, int64_t K, int64_t nt, int* status, Dep dep, cudaStream_t stream);

// Fused quantize + MMVQ: x f32 in, q8_1 (xq, xds) and out written.  With
// `static_w` the weight stream starts before the preceding kernel completes.
int launch_gemv_fused(int qtype, const void* W, const float* x, int8_t* xq, float* xds, float* out, int64_t od,
                      int64_t K, int64_t nt, int* status, bool static_w, cudaStream_t stream);

// Tensor-core GEMM over the prepared workspace.  dots != nullptr selects the
// raw block-dot output (no scale folded into the weight operand).  `part`
// holds gemm_part_bytes of split-K partial sums (unused when the shape does
// not split).
int launch_gemm_tc(int qtype, const void* W, const __half* xh, const float* scl, float* out, int32_t* dots,
                   float* part, int64_t od, int64_t K, int64_t nt, int* status, int stall_ms, cudaStream_t stream);

}  // namespace qmm
