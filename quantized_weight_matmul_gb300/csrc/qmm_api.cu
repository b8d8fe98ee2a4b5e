// qmm_api.cu -- the C ABI (include/qmm.h): host-side argument checks, the
// nt-based choice between the MMVQ and the tensor-core path, and the device
// status word bounded kernel waits report into.  Errors are returned, never
// papered over by another path ("04 - Reading minfer's kernels II", sec. 3.3).
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cstdint>

#include "qmm_internal.h"

namespace qmm {

// First error recorded by a kernel on this device since the last
// qmm_sync_status; 0 when none.
__device__ int g_status_word;

namespace {

PerDevice<int*> g_status_ptr;
std::atomic<int> g_stall_ms{0};

bool valid_qtype(int q) { return q == QMM_Q4_K || q == QMM_Q6_K; }
int block_bytes(int q) { return q == QMM_Q4_K ? 144 : (q == QMM_Q6_K ? 210 : 0); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int64_t od, int64_t K, int64_t nt) {
  if (od < 1 || nt < 1 || K < 256 || K % 256) return QMM_EINVAL_SHAPE;
  if (od > INT_MAX || K > INT_MAX || nt > INT_MAX) return QMM_EINVAL_SHAPE;
  if (od * nt > INT_MAX || nt * K > INT_MAX || od * (K / 32) > INT_MAX) return QMM_EINVAL_SHAPE;
  return QMM_OK;
}

// Device address of this device's status word (looked up once per device,
// with that device current).
int status_ptr(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMM_EDEVICE;
  int* ptr = g_status_ptr.get(dev);
  if (!ptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess || !p) return QMM_EDEVICE;
    ptr = static_cast<int*>(p);
    g_status_ptr.set(dev, ptr);
  }
  *out = ptr;
  return QMM_OK;
}

int check_device() {
  static PerDevice<int> cached;  // 0 unknown, 1 ok, -1 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMM_EDEVICE;
  int v = cached.get(dev);
  if (v == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    v = (major == 10 && minor == 3) ? 1 : -1;
    cached.set(dev, v);
  }
  return v == 1 ? QMM_OK : QMM_EDEVICE;
}

// f16 codes, token-contiguous scale rows, then the split-K partial sums
size_t gemm_ws(int64_t od, int64_t K, int64_t nt) {
  return gemm_xh_bytes(nt, K) + gemm_scl_bytes(nt, K) + gemm_part_bytes(od, K, nt);
}

// The qmm_matmul route for a valid problem (one place, so the query below and
// the dispatch cannot disagree).
int matmul_route(int qtype, int64_t nt, int64_t K) {
  if (nt >= mma_min_nt(qtype) && mmvq_mma_fits(qtype, nt, K)) return QMM_PATH_MMVQ;
  if (gemv_fused_fits(qtype, nt, K)) return QMM_PATH_FUSED_MMVQ;
  if (nt <= 8 && gemv_fits(qtype, nt, K)) return QMM_PATH_MMVQ;
  return QMM_PATH_MMQ;
}

// Every refusal of the tensor-core route, checked before any device work is
// enqueued (the route takes any shape check_shape accepts: rows of any pitch
// are staged); on success *status is the device status word.
int gemm_check(int64_t od, int64_t K, int64_t nt, const void* ws, size_t ws_bytes, int** status) {
  if (ws_bytes < gemm_ws(od, K, nt)) return QMM_EWORKSPACE;
  if (!ws) return QMM_ENULL;
  if (!aligned16(ws)) return QMM_EALIGN;
  return status_ptr(status);
}

int gemm_core(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int32_t* dots,
              int64_t od, int64_t K, int64_t nt, void* ws, size_t ws_bytes, bool prep, cudaStream_t st) {
  int* status = nullptr;
  int rc = gemm_check(od, K, nt, ws, ws_bytes, &status);
  if (rc) return rc;
  __half* xh = static_cast<__half*>(ws);
  float* scl = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + gemm_xh_bytes(nt, K));
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + gemm_xh_bytes(nt, K) + gemm_scl_bytes(nt, K));
  if (prep) {
    rc = launch_gemm_prep(xq, xds, nt, K, gemm_ntp(nt), xh, scl, st);
    if (rc) return rc;
  }
  return launch_gemm_tc(qtype, W, xh, scl, out, dots, part, od, K, nt, status, stall_ms(), st);
}

}  // namespace

int stall_ms() { return g_stall_ms.load(); }

}  // namespace qmm

using namespace qmm;

extern "C" {

size_t qmm_weight_bytes(int qtype, int64_t od, int64_t K) {
  if (!valid_qtype(qtype) || od < 0 || K < 0 || K % 256) return 0;
  return (size_t)od * (size_t)(K / 256) * (size_t)block_bytes(qtype);
}

size_t qmm_xq_bytes(int64_t nt, int64_t K) { return nt < 0 || K < 0 ? 0 : (size_t)nt * (size_t)K; }

size_t qmm_q8_1_bytes(int64_t nt, int64_t K) { return qmm_xq_bytes(nt, K); }

size_t qmm_xds_bytes(int64_t nt, int64_t K) {
  return nt < 0 || K < 0 || K % 32 ? 0 : (size_t)nt * (size_t)(K / 32) * 2 * sizeof(float);
}

size_t qmm_gemm_workspace_bytes(int qtype, int64_t od, int64_t K, int64_t nt) {
  if (!valid_qtype(qtype) || check_shape(od, K, nt)) return 0;
  return gemm_ws(od, K, nt);
}

size_t qmm_matmul_workspace_bytes(int qtype, int64_t od, int64_t K, int64_t nt) {
  if (!valid_qtype(qtype) || check_shape(od, K, nt)) return 0;
  if (matmul_route(qtype, nt, K) != QMM_PATH_MMQ) return 0;
  return gemm_ws(od, K, nt);
}

int qmm_matmul_path(int qtype, int64_t od, int64_t K, int64_t nt) {
  if (!valid_qtype(qtype)) return QMM_EINVAL_QTYPE;
  int rc = check_shape(od, K, nt);
  if (rc) return rc;
  return matmul_route(qtype, nt, K);
}

int qmm_gemv_max_nt(void) { return kMmaMaxNt; }

int qmm_quantize_q8_1(const float* x, int64_t nt, int64_t K, int8_t* xq, float* xds, void* stream) {
  if (!x || !xq || !xds) return QMM_ENULL;
  if (nt < 1 || K < 32 || K % 32 || nt > INT_MAX || K > INT_MAX || nt * K > INT_MAX) return QMM_EINVAL_SHAPE;
  if (!aligned16(x) || !aligned16(xq) || !aligned16(xds)) return QMM_EALIGN;
  int rc = check_device();
  if (rc) return rc;
  return launch_quantize(x, nt, K, xq, xds, nullptr, nullptr, 0, static_cast<cudaStream_t>(stream));
}

int qmm_gemv(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int64_t od, int64_t K,
             int64_t nt, void* stream) {
  if (!valid_qtype(qtype)) return QMM_EINVAL_QTYPE;
  if (!W || !xq || !xds || !out) return QMM_ENULL;
  int rc = check_shape(od, K, nt);
  if (rc) return rc;
  if (nt > kMmaMaxNt) return QMM_EINVAL_SHAPE;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(xds) || !aligned16(out)) return QMM_EALIGN;
  rc = check_device();
  if (rc) return rc;
  int* status = nullptr;
  rc = status_ptr(&status);
  if (rc) return rc;
  // a programmatic dependent of the preceding kernel: every access that may
  // depend on it (the weights included) waits for it, the prologue does not
  return launch_gemv(qtype, W, xq, xds, out, nullptr, od, K, nt, status, Dep::kPdl,
                     static_cast<cudaStream_t>(stream));
}

int qmm_gemm(int qtype, const void* W, const int8_t* xq, const float* xds, float* out, int64_t od, int64_t K,
             int64_t nt, void* workspace, size_t ws_bytes, void* stream) {
  if (!valid_qtype(qtype)) return QMM_EINVAL_QTYPE;
  if (!W || !xq || !xds || !out) return QMM_ENULL;
  int rc = check_shape(od, K, nt);
  if (rc) return rc;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(xds) || !aligned16(out)) return QMM_EALIGN;
  rc = check_device();
  if (rc) return rc;
  return gemm_core(qtype, W, xq, xds, out, nullptr, od, K, nt, workspace, ws_bytes, true,
                   static_cast<cudaStream_t>(stream));
}

int qmm_matmul(int qtype, const void* W, const float* x, int8_t* xq, float* xds, float* out, int64_t od,
               int64_t K, int64_t nt, void* workspace, size_t ws_bytes, unsigned flags, void* stream) {
  if (!valid_qtype(qtype)) return QMM_EINVAL_QTYPE;
  if (!W || !x || !xq || !xds || !out) return QMM_ENULL;
  int rc = check_shape(od, K, nt);
  if (rc) return rc;
  if (!aligned16(W) || !aligned16(x) || !aligned16(xq) || !aligned16(xds) || !aligned16(out)) return QMM_EALIGN;
  if (flags & ~(unsigned)QMM_FLAG_STATIC_WEIGHTS) return QMM_EINVAL_SHAPE;
  rc = check_device();
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int path = matmul_route(qtype, nt, K);
  if (path == QMM_PATH_FUSED_MMVQ) {
    int* status = nullptr;
    rc = status_ptr(&status);
    if (rc) return rc;
    return launch_gemv_fused(qtype, W, x, xq, xds, out, od, K, nt, status,
                             (flags & QMM_FLAG_STATIC_WEIGHTS) != 0, st);
  }
  if (path == QMM_PATH_MMVQ) {
    int* status = nullptr;
    rc = status_ptr(&status);
    if (rc) return rc;
    rc = launch_quantize(x, nt, K, xq, xds, nullptr, nullptr, 0, st);
    if (rc) return rc;
    return launch_gemv(qtype, W, xq, xds, out, nullptr, od, K, nt, status, Dep::kPdlStaticW, st);
  }
  int* status = nullptr;
  rc = gemm_check(od, K, nt, workspace, ws_bytes, &status);
  if (rc) return rc;
  // the quantizer writes the tensor-core operands directly: no separate prepass
  __half* xh = static_cast<__half*>(workspace);
  float* scl = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + gemm_xh_bytes(nt, K));
  rc = launch_quantize(x, nt, K, xq, xds, xh, scl, gemm_ntp(nt), st);
  if (rc) return rc;
  return gemm_core(qtype, W, xq, xds, out, nullptr, od, K, nt, workspace, ws_bytes, false, st);
}

int qmm_debug_block_dots(int qtype, const void* W, const int8_t* xq, const float* xds, int64_t od, int64_t K,
                         int64_t nt, int32_t* dots, int path, void* workspace, size_t ws_bytes, void* stream) {
  if (!valid_qtype(qtype)) return QMM_EINVAL_QTYPE;
  if (!W || !xq || !dots) return QMM_ENULL;
  int rc = check_shape(od, K, nt);
  if (rc) return rc;
  if (!aligned16(W) || !aligned16(xq)) return QMM_EALIGN;
  rc = check_device();
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (path == 0) {
    if (nt > 8) return QMM_EINVAL_SHAPE;
    if (!xds) return QMM_ENULL;
    int* status = nullptr;
    rc = status_ptr(&status);
    if (rc) return rc;
    return launch_gemv(qtype, W, xq, xds, nullptr, dots, od, K, nt, status, Dep::kNone, st);
  }
  if (path == 2) {
    if (nt > kMmaMaxNt) return QMM_EINVAL_SHAPE;
    if (!xds) return QMM_ENULL;
    if (!aligned16(xds)) return QMM_EALIGN;
    int* status = nullptr;
    rc = status_ptr(&status);
    if (rc) return rc;
    return launch_mmvq_mma(qtype, W, xq, xds, nullptr, dots, od, K, nt, status, Dep::kNone, st);
  }
  if (path != 1) return QMM_EINVAL_SHAPE;
  if (!xds) return QMM_ENULL;
  if (!aligned16(xds)) return QMM_EALIGN;
  return gemm_core(qtype, W, xq, xds, nullptr, dots, od, K, nt, workspace, ws_bytes, true, st);
}

int qmm_sync_status(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return QMM_ELAUNCH;
  int* status = nullptr;
  int rc = status_ptr(&status);
  if (rc) return rc;
  int h = 0;
  if (cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return QMM_ELAUNCH;
  if (h != 0) {
    const int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return QMM_ELAUNCH;
  }
  return h;
}

int qmm_debug_inject_stall(int on, int ms) {
  if (on && (ms < 1 || ms > 10000)) return QMM_EINVAL_SHAPE;
  g_stall_ms.store(on ? ms : 0);
  return QMM_OK;
}

const char* qmm_strerror(int status) {
  switch (status) {
    case QMM_OK: return "ok";
    case QMM_EINVAL_QTYPE: return "unsupported weight type";
    case QMM_EINVAL_SHAPE: return "invalid shape (od, K, nt)";
    case QMM_EALIGN: return "pointer not 16-byte aligned";
    case QMM_ENULL: return "required pointer is NULL";
    case QMM_EWORKSPACE: return "workspace too small";
    case QMM_ESMEM: return "shared memory request exceeds the device limit";
    case QMM_ELAUNCH: return "CUDA launch or runtime error";
    case QMM_ETIMEOUT: return "a bounded device-side wait timed out";
    case QMM_EDEVICE: return "no usable sm_103 device is current";
    default: return "unknown status";
  }
}

}  // extern "C"

// ------------------------------------------- GEMM with a built-in workspace --
// For callers that may not allocate device memory at all: the scratch the
// tensor-core GEMM needs (f16 codes and token-contiguous scale rows) lives in
// one fixed array that is part of the loaded module.  Its device address is
// taken once per device and passed to the same prepass and GEMM kernels that
// qmm_gemm runs on a caller's workspace.
namespace qmm {
namespace {

static __device__ __align__(256) uint8_t g_builtin_ws[QMM_BUILTIN_WORKSPACE_BYTES];
PerDevice<void*> g_builtin_ws_ptr;

int builtin_ws_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMM_EDEVICE;
  void* ptr = g_builtin_ws_ptr.get(dev);
  if (!ptr) {
    if (cudaGetSymbolAddress(&ptr, g_builtin_ws) != cudaSuccess || !ptr) return QMM_EDEVICE;
    g_builtin_ws_ptr.set(dev, ptr);
  }
  *out = ptr;
  return QMM_OK;
}

}  // namespace
}  // namespace qmm

extern "C" int qmm_gemm_builtin_workspace(int qtype, const void* W, const int8_t* xq, const float* xds, float* out,
                                          int64_t od, int64_t K, int64_t nt, void* stream) {
  if (!valid_qtype(qtype)) return QMM_EINVAL_QTYPE;
  if (!W || !xq || !xds || !out) return QMM_ENULL;
  int rc = check_shape(od, K, nt);
  if (rc) return rc;
  if (!aligned16(W) || !aligned16(xq) || !aligned16(xds) || !aligned16(out)) return QMM_EALIGN;
  const size_t need = gemm_ws(od, K, nt);
  if (need > (size_t)QMM_BUILTIN_WORKSPACE_BYTES) return QMM_EWORKSPACE;
  rc = check_device();
  if (rc) return rc;
  void* ws = nullptr;
  rc = builtin_ws_ptr(&ws);
  if (rc) return rc;
  // every remaining refusal happens here, before the padding clears below
  // are enqueued: a refused call leaves the shared array untouched
  int* status = nullptr;
  rc = gemm_check(od, K, nt, ws, (size_t)QMM_BUILTIN_WORKSPACE_BYTES, &status);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The prepass writes the scale planes only for tokens < nt; the padding
  // tokens of the last tile would otherwise hold whatever an earlier call of
  // another shape left there.  They feed only output columns that are never
  // stored, but they are zeroed so every call computes on defined values.
  const int64_t ntp = gemm_ntp(nt);
  if (ntp > nt) {
    uint8_t* dxp = static_cast<uint8_t*>(ws) + gemm_xh_bytes(nt, K);
    uint8_t* smp = dxp + gemm_dx_bytes(nt, K);
    if (cudaMemset2DAsync(dxp + nt * 4, (size_t)ntp * 4, 0, (size_t)(ntp - nt) * 4, (size_t)(K / 32), st) !=
            cudaSuccess ||
        cudaMemset2DAsync(smp + nt * 16, (size_t)ntp * 16, 0, (size_t)(ntp - nt) * 16, (size_t)(K / 256) * 4, st) !=
            cudaSuccess)
      return QMM_ELAUNCH;
  }
  return gemm_core(qtype, W, xq, xds, out, nullptr, od, K, nt, ws, (size_t)QMM_BUILTIN_WORKSPACE_BYTES, true, st);
}
