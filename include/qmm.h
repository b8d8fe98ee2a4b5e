/*
 * qmm.h -- C ABI of the GB300 (sm_103a) quantized-weight matmul library.
 *
 *     out[t][r] = sum_k W[r][k] * x[t][k]        t < nt, r < od, k < K
 *
 * W is kept as raw GGUF K-quant super-blocks (never dequantized to a float
 * copy); the activations are quantized on the device to q8_1 blocks and the
 * products are exact integer dots rescaled in fp32.
 *
 * Sources (page titles and sections):
 *   [MMQ]  "llama.cpp MMQ -- quantized-weight int8 tensor-core matmul":
 *          sec. 4 (Q4_K and Q6_K block layouts), sec. 6 (the (scale, min)
 *          unpack, the rescale sum += dA*dB*C + mA*sB), sec. 12 (MMVQ keeps
 *          up to 8 tokens in registers; MMQ beyond).
 *   [MOJO] mojo-dllm "The quantized GEMM": "The GPU path" (warp-per-32 q8_1
 *          quantizer with f32 scale and scale*sum(q); the identity
 *          sum w x = d*sc*dx*sum(q*qx) - dmin*m*(dx*sum(qx)); one MMA per
 *          scale group), "Weights" (zero points off the inner loop).
 *   [CH04] "04 - Reading minfer's kernels II": sec. 2.2 (W row-major
 *          [out][in], activations token-major [nt][in], out [nt][od]),
 *          sec. 3.3 (errors, not silent fallbacks), sec. 3.4 (MMVQ).
 *
 * Conventions shared by every entry point
 *   - Pointers named "device" are CUDA device pointers owned by the caller;
 *     the library never frees, keeps or allocates device memory.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; no call synchronizes the
 *     host except qmm_sync_status.
 *   - Layouts: W is row-major [od][K/256] super-blocks (raw GGUF bytes,
 *     16-byte aligned base); x and xq are token-major [nt][K]; xds is
 *     [nt][K/32][2] f32 = (d, s); out is [nt][od] f32, od contiguous.
 *   - Preconditions checked on the host: qtype is QMM_Q4_K or QMM_Q6_K;
 *     K > 0 and K % 256 == 0; od >= 1; nt >= 1 (qmm_gemv: 1 <= nt <= 16);
 *     od, K, nt and od*nt, nt*K below 2^31; non-NULL pointers; W, x, xq,
 *     xds, out and the workspace 16-byte aligned.  Inputs must be finite.
 *   - Every call returns QMM_OK (0) or a negative QMM_E* code and launches
 *     nothing when it fails a check.  There is no fallback to another kernel,
 *     to the CPU or to a dense library GEMM.
 */
#ifndef QMM_H
#define QMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Flags of qmm_matmul. */
#define QMM_FLAG_STATIC_WEIGHTS 1u /* see qmm_matmul */

/* Weight block types.  12 is the GGML id of Q4_K ([MMQ] sec. 1); 14 is the
 * public GGML id of Q6_K. */
typedef enum { QMM_Q4_K = 12, QMM_Q6_K = 14 } qmm_qtype;

enum {
    QMM_OK = 0,
    QMM_EINVAL_QTYPE = -1, /* qtype is not QMM_Q4_K / QMM_Q6_K            */
    QMM_EINVAL_SHAPE = -2, /* od, K or nt out of range                    */
    QMM_EALIGN = -3,       /* a pointer is not 16-byte aligned            */
    QMM_ENULL = -4,        /* a required pointer is NULL                  */
    QMM_EWORKSPACE = -5,   /* workspace smaller than required             */
    QMM_ESMEM = -6,        /* the kernel's shared memory exceeds the cap  */
    QMM_ELAUNCH = -7,      /* a CUDA runtime call or launch failed        */
    QMM_ETIMEOUT = -8,     /* a bounded device-side wait gave up          */
    QMM_EDEVICE = -9,      /* no usable sm_103 device is current          */
};

/* ------------------------------------------------------------ sizes ---- */

/* Bytes of W [od][K] in `qtype`: od*K/256*144 (Q4_K) or od*K/256*210
 * (Q6_K) ([MMQ] sec. 4).  0 for an invalid qtype or shape.  Host only. */
size_t qmm_weight_bytes(int qtype, int64_t od, int64_t K);

/* Bytes of the q8_1 activations: xq = nt*K int8, xds = nt*(K/32)*2 f32.
 * qmm_q8_1_bytes is the size of the codes, nt*K (the same as qmm_xq_bytes);
 * the (d, s) pairs take qmm_xds_bytes.  0 for a negative size (xds: or a K
 * that is not a multiple of 32). */
size_t qmm_q8_1_bytes(int64_t nt, int64_t K);
size_t qmm_xq_bytes(int64_t nt, int64_t K);
size_t qmm_xds_bytes(int64_t nt, int64_t K);

/* Workspace qmm_gemm needs for this problem (f16 copy of the int8 codes,
 * token-contiguous scale planes and, for shapes with fewer output tiles than
 * SMs, split-K partial sums; see qmm_gemm).  A function of the shape alone.
 * 0 for invalid input. */
size_t qmm_gemm_workspace_bytes(int qtype, int64_t od, int64_t K, int64_t nt);

/* Workspace qmm_matmul needs: 0 on its MMVQ routes (at most 16 tokens; see
 * qmm_matmul and qmm_matmul_path), else qmm_gemm_workspace_bytes. */
size_t qmm_matmul_workspace_bytes(int qtype, int64_t od, int64_t K, int64_t nt);

/* Routes of qmm_matmul (see there), as returned by qmm_matmul_path. */
#define QMM_PATH_FUSED_MMVQ 1 /* one kernel: quantize inside the MMVQ kernel  */
#define QMM_PATH_MMVQ 2       /* two kernels: quantizer, then MMVQ            */
#define QMM_PATH_MMQ 3        /* two kernels: quantizer, then tensor-core GEMM */

/* The route qmm_matmul takes for this problem (a QMM_PATH_* value), or the
 * negative QMM_E* code qmm_matmul would return for the shape or type.  Host
 * only; it depends on nothing but its arguments. */
int qmm_matmul_path(int qtype, int64_t od, int64_t K, int64_t nt);

/* Largest nt qmm_gemv accepts (16: two 8-token tiles of the warp-MMA MMVQ). */
int qmm_gemv_max_nt(void);

/* ------------------------------------------------------- device work ---- */

/*
 * q8_1 quantization of x [nt][K] f32 ([MOJO] "The GPU path"; [CH04]
 * sec. 3.4).  Per 32-value block: amax by a shuffle max, d = amax/127 (IEEE
 * f32 division), q = round-half-even of the IEEE quotient x/d clamped to
 * [-127, 127], s = d * (float)sum(q) with sum(q) an integer shuffle sum.  The
 * codes are decided from x * fl(1/d) and fall back to the division only when
 * that lands within 1e-4 of a half-integer, so they equal the division's.  A
 * block of zeros gives d = s = 0 and q = 0.
 * Output: xq [nt][K] int8, xds [nt][K/32][2] f32 (d, s).  K % 32 == 0
 * suffices here.  Bit-exact with the IEEE definition.
 */
int qmm_quantize_q8_1(const float *x, int64_t nt, int64_t K, int8_t *xq, float *xds,
                      void *stream);

/*
 * MMVQ: small-batch matmul for 1 <= nt <= 16 ([CH04] sec. 3.4; [MMQ] sec. 12).
 * Streams every weight row once in TMA-staged tiles and lets every weight
 * block meet all nt tokens while it is on chip, so the weight traffic does not
 * grow with nt.  Q4_K: per 32-value sub-block j the integer dot
 * D = sum(nibble * q) is rescaled as d*sc_j*dx*D - dmin*m_j*s.  Q6_K: per
 * 16-value group g, D = sum((q6 - 32) * q) is rescaled as d*sc_g*dx*D.  Rows
 * whose pitch is not a multiple of 16 bytes (Q6_K with K % 2048 != 0) are
 * staged row by row as 16-byte-aligned windows.  Few tokens (nt <= 4 for Q4_K,
 * nt = 1 for Q6_K) take the dp4a kernel, more tokens the warp-level
 * tensor-core MMA kernel (mma.sync on exact small-integer f16 operands).
 * QMM_ESMEM when the nt x K activations do not fit the chosen kernel's shared
 * memory next to its weight ring (for nt > 8 only the MMA kernel applies:
 * about nt*K <= 96K codes).  out [nt][od] f32 is overwritten.
 */
int qmm_gemv(int qtype, const void *W, const int8_t *xq, const float *xds, float *out,
             int64_t od, int64_t K, int64_t nt, void *stream);

/*
 * MMQ: matmul for any nt >= 1 on the tcgen05 tensor cores ([MMQ] sec. 2-6;
 * [MOJO] "One mma per scale group").  Raw super-blocks are staged into
 * shared memory by TMA and unpacked in registers into exact small-integer
 * f16 weight operands that carry the integer group scale (Q4_K sc*nibble;
 * Q6_K sc*(q - 32), split exactly into two operands), written into tensor
 * memory; one MMA chain per 32-value block accumulates the exact integer sum
 * in TMEM (fp32, exact for these magnitudes), and the fp32 epilogue applies
 * d, dx and, for Q4_K, the min term dmin * sum(m*s).
 * `workspace` (device, 16-byte aligned, >= qmm_gemm_workspace_bytes) holds
 * an f16 copy of xq and the scale planes written by a prepass on `stream`;
 * its contents need not be preserved between calls.  out is overwritten.
 * Any K % 256 == 0: rows whose pitch is not a multiple of 16 bytes (Q6_K with
 * K % 2048 != 0), which a TMA tensor map cannot describe, are staged row by
 * row as 16-byte-aligned windows around each block.
 * When the 128-row x token tiles are fewer than the GPU's SMs, K is split
 * into up to 8 slices of whole super-blocks computed by separate CTAs; their
 * fp32 partial sums (in the workspace) are added in a fixed order, so
 * results stay bitwise reproducible.
 */
int qmm_gemm(int qtype, const void *W, const int8_t *xq, const float *xds, float *out,
             int64_t od, int64_t K, int64_t nt, void *workspace, size_t ws_bytes, void *stream);

/*
 * qmm_gemm for callers that cannot allocate device memory.  The source pages
 * have no counterpart to this entry point: it exists only for code that must
 * not call cudaMalloc (or any allocating routine) itself.
 *
 * Same operation, arguments and kernels as qmm_gemm, but the scratch qmm_gemm
 * takes as `workspace` is a fixed array of QMM_BUILTIN_WORKSPACE_BYTES (8 MiB)
 * compiled into the library and reserved on each device when the library's
 * module loads.  The function itself allocates nothing.
 *   - Size limit: qmm_gemm_workspace_bytes(qtype, od, K, nt) must not exceed
 *     QMM_BUILTIN_WORKSPACE_BYTES (e.g. nt = 512 at K = 4096 needs 4.75 MiB;
 *     nt = 512 at K = 14336 needs 16.6 MiB and is refused).  A larger problem
 *     returns QMM_EWORKSPACE and launches nothing; use qmm_gemm with a
 *     workspace of your own for it.
 *   - Nothing in the array has to start at zero: the prepass rewrites every
 *     entry a stored output depends on, and each call zeroes the remaining
 *     padding entries of the last token tile itself.
 *   - There is one array per device, shared by all calls on that device.
 *     Calls whose work can overlap on the device (different streams, or
 *     different host threads without ordering between them) race on it and
 *     may produce wrong results: keep them ordered, e.g. on one stream.
 *   - The first call on each device looks the array's address up (a CUDA
 *     runtime query, cached afterwards).  If that first call is what does
 *     this set-up, make it before any stream capture begins.
 * Errors: as qmm_gemm, plus QMM_EWORKSPACE for the size limit above and
 * QMM_EDEVICE if the address lookup fails.
 */
#define QMM_BUILTIN_WORKSPACE_BYTES (8u << 20)
int qmm_gemm_builtin_workspace(int qtype, const void *W, const int8_t *xq, const float *xds, float *out,
                               int64_t od, int64_t K, int64_t nt, void *stream);

/*
 * The whole method from f32 activations, all on `stream` ([CH04] sec. 3.3:
 * the small-batch / prefill split by nt):
 *   - from 5 tokens (Q4_K) or 2 (Q6_K) up to 16, where the activations fit
 *     the warp-MMA MMVQ's shared memory: qmm_quantize_q8_1 into xq / xds,
 *     then qmm_gemv on the MMA kernel;
 *   - other nt <= 8 whose activations (nt*round_up(K, 2048) codes plus the
 *     scales) leave room for three weight stages (16 rows x 2048 k: 18 KB for
 *     Q4_K, 26 KB for Q6_K) in half of an SM's shared memory (the decode
 *     shapes): one fused kernel quantizes x to q8_1 inside the dp4a MMVQ
 *     kernel (bit-identical codes) and writes xq / xds and out;
 *   - other nt <= 8: qmm_quantize_q8_1 into xq / xds, then qmm_gemv;
 *   - otherwise: qmm_quantize_q8_1 (which also writes the GEMM workspace),
 *     then the tensor-core GEMM of qmm_gemm.
 * The matmul kernels are launched as programmatic dependents of the kernel
 * before them and wait for it before reading anything it may write.  With
 * QMM_FLAG_STATIC_WEIGHTS the caller promises that W is not written by any
 * work still in flight on `stream`; the weight stream then starts before the
 * preceding kernel has completed (weights-once decode overlaps kernel
 * boundaries).  `flags` = 0 is always safe.  `workspace` may be NULL when
 * qmm_matmul_workspace_bytes returns 0.  Unknown flag bits: QMM_EINVAL_SHAPE.
 */
int qmm_matmul(int qtype, const void *W, const float *x, int8_t *xq, float *xds, float *out,
               int64_t od, int64_t K, int64_t nt, void *workspace, size_t ws_bytes, unsigned flags,
               void *stream);

/*
 * Test hook: the exact int32 block dots, computed by the same device dot code
 * as a matmul path but written out before any scaling.
 *   Q4_K: dots[t][r][j] = sum_{i<32} nibble[r][32j+i] * xq[t][32j+i], j < K/32
 *   Q6_K: dots[t][r][g] = sum_{i<16} (q6[r][16g+i] - 32) * xq[t][16g+i], g < K/16
 * path 0: the dp4a MMVQ dot code, nt <= 8.
 * path 1: the tensor-core (qmm_gemm) dot code with the same tile choice and
 *         weight operands as the product kernel, which carry the integer
 *         group scales, so the sums come out scaled, one per 32-value block:
 *           Q4_K: dots[t][r][j] = sc_j * D_j (sc_j the 6-bit scale of
 *                 sub-block j), j < K/32;
 *           Q6_K: dots[t][r][b] = sc_2b * D_2b + sc_2b+1 * D_2b+1 (the signed
 *                 int8 scales of the block's two 16-value groups), b < K/32;
 *         both 0 for a super-block whose d is 0.  Needs xds (for the
 *         prepass) and a workspace of qmm_gemm_workspace_bytes.
 * path 2: the warp-MMA MMVQ dot code, nt <= 16; needs
 *         xds; QMM_ESMEM where the activations do not fit its shared memory.
 * dots is a device buffer of nt*od*ng int32: ng = K/32, except K/16 for
 * Q6_K on paths 0 and 2.
 */
int qmm_debug_block_dots(int qtype, const void *W, const int8_t *xq, const float *xds,
                         int64_t od, int64_t K, int64_t nt, int32_t *dots, int path,
                         void *workspace, size_t ws_bytes, void *stream);

/*
 * Synchronizes `stream`, then returns and clears the first error a kernel of
 * this library recorded on the current device since the last call
 * (QMM_ETIMEOUT when a bounded wait inside a kernel gave up), or QMM_ELAUNCH
 * if the stream reports a CUDA error, else QMM_OK.
 */
int qmm_sync_status(void *stream);

/* Test hook: while `on` is nonzero, every kernel launch with bounded waits
 * (the tensor-core GEMM and both MMVQ kernels, fused or not) skips one
 * producer arrival per CTA on purpose, so that its waits run out and report
 * QMM_ETIMEOUT through qmm_sync_status (no trap, no hang: every wait gives up
 * after about `ms` milliseconds, in-flight copies are drained).  Off by
 * default. */
int qmm_debug_inject_stall(int on, int ms);

/* Static string for a status code. */
const char *qmm_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* QMM_H */
