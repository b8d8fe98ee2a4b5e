/*
 * qmm_oracle.c -- plain, slow CPU oracle for the quantized-weight matmul
 *
 *     out[t][r] = sum_k W[r][k] * x[t][k]
 *
 * with W stored as raw GGUF K-quant super-blocks (Q4_K, Q6_K) and x quantized
 * to q8_1 blocks (int8 values, one f32 scale per 32 values, plus scale*sum(q)).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference the CUDA path is
 * checked against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg load it; the product library never links or calls it, and it
 * shares no code, header or table with the CUDA sources.
 *
 * Everything here is scalar C, one element at a time, in the order the method
 * is defined; no blocking, no SIMD intrinsics, no fast-math.  Build with
 * -ffp-contract=off so no multiply-add is fused on any host.
 *
 * Sources (page titles; sections):
 *   [MMQ]  "llama.cpp MMQ -- quantized-weight int8 tensor-core matmul",
 *          sec. 4 (weight staging, Q6_K specialization) and sec. 6 (numerics,
 *          get_scale_min_k4 semantics, the rescale).
 *   [MOJO] "The quantized GEMM" (mojo-dllm kernels page), sections
 *          "Weights: 8 rows per register" (zero points), "The GPU path"
 *          (q8_1 activations, the sum identity, Q4_K nibble placement, Q6_K).
 *   [CH04] "04 - Reading minfer's kernels II", sec. 3.4 (quantize: max, scale,
 *          round; the two-term Q4_K correction) and sec. 2.2 (memory layout:
 *          W row-major [out][in], activations token-major [nt][in]).
 *
 * Readings where the pages are silent (stated once, used everywhere):
 *   - q8_1: d = amax/127 (f32 division), q = round-half-even(x/d) (true f32
 *     division), clamped to [-127,127]; amax == 0 gives d = q = s = 0;
 *     s = d * (float)sum(q) (one f32 rounding).  Both d and s are stored f32.
 *   - Q6_K bit placement of ql/qh follows the public GGUF convention (the
 *     pages only say "low nibbles, two high bits"); scales are signed int8.
 *   - Output sums are taken in f64 and rounded to f32 once.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_Q4_K 12 /* GGML type id for Q4_K, named in [MMQ] sec. 1 */
#define ORACLE_Q6_K 14 /* GGML type id for Q6_K (public numbering) */

#define ORACLE_OK 0
#define ORACLE_EQTYPE (-1)
#define ORACLE_ESHAPE (-2)
#define ORACLE_ENOMEM (-3)

/* ---------------------------------------------------------------- f16 --- */

/* IEEE binary16 -> double, exactly (subnormals kept). */
static double half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static uint16_t load_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ---------------------------------------------------------------- Q4_K --- */
/*
 * Q4_K super-block, 144 bytes, 256 weights ([MMQ] sec. 4; [MOJO] "The GPU
 * path": the 16-byte header d, dmin, packed scales comes first, then 128 bytes
 * of nibbles):
 *   [0,2)  d     f16
 *   [2,4)  dmin  f16
 *   [4,16) scales[12]: eight 6-bit (sc, m) pairs
 *   [16,144) qs[128]
 */
#define Q4K_BYTES 144
#define Q6K_BYTES 210

/* The 6-bit (scale, min) of sub-block j, as [MMQ] sec. 6 defines them. */
static void q4k_scale_min(const uint8_t *scales, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 0x0F) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

/*
 * Nibble of element e (0..255) of a Q4_K block.  Byte i of nibble pair p
 * (qs[32p + i]) holds element i of sub-block 2p in its low nibble and element
 * i of sub-block 2p+1 in its high nibble ([MOJO] "The GPU path"; [MMQ] sec. 4
 * stages the low and high nibbles of the same word as separate 32-value runs).
 * Sub-block j covers elements 32j .. 32j+31.
 */
static int q4k_nibble(const uint8_t *qs, int e)
{
    int p = e / 64;
    int i = e % 64;
    if (i < 32)
        return qs[32 * p + i] & 0x0F;
    return qs[32 * p + (i - 32)] >> 4;
}

/* Dequantized weight e of a Q4_K block: d*sc*q - dmin*m ([MMQ] sec. 6). */
static double q4k_weight(const uint8_t *blk, int e)
{
    double d = half_to_double(load_u16(blk));
    double dmin = half_to_double(load_u16(blk + 2));
    int sc, m;
    q4k_scale_min(blk + 4, e / 32, &sc, &m);
    return d * sc * q4k_nibble(blk + 16, e) - dmin * m;
}

/* ---------------------------------------------------------------- Q6_K --- */
/*
 * Q6_K super-block, 210 bytes, 256 weights:
 *   [0,128)   ql: low 4 bits
 *   [128,192) qh: high 2 bits
 *   [192,208) scales[16]: signed int8, one per 16 weights
 *   [208,210) d f16
 * Weight e is d * scales[e/16] * (q_e - 32), q_e in [0,63] ([MMQ] sec. 4:
 * centred by 32 at use, int8 scale per 16 values; [MOJO] "Weights": the 32
 * comes off like a zero point).
 */
static int q6k_q(const uint8_t *blk, int e)
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    int half = e / 128;          /* which 128-weight half */
    int quad = (e % 128) / 32;   /* which 32-weight quarter of that half */
    int l = e % 32;
    const uint8_t *L = ql + 64 * half;
    const uint8_t *H = qh + 32 * half;
    int lo;
    switch (quad) {
    case 0: lo = L[l] & 0x0F; break;
    case 1: lo = L[l + 32] & 0x0F; break;
    case 2: lo = L[l] >> 4; break;
    default: lo = L[l + 32] >> 4; break;
    }
    int hi = (H[l] >> (2 * quad)) & 3;
    return lo | (hi << 4);
}

static int q6k_scale(const uint8_t *blk, int g) { return (int)(int8_t)blk[192 + g]; }

static double q6k_weight(const uint8_t *blk, int e)
{
    double d = half_to_double(load_u16(blk + 208));
    return d * q6k_scale(blk, e / 16) * (q6k_q(blk, e) - 32);
}

static int block_bytes(int qtype)
{
    if (qtype == ORACLE_Q4_K) return Q4K_BYTES;
    if (qtype == ORACLE_Q6_K) return Q6K_BYTES;
    return 0;
}

/* ---------------------------------------------------------- public API --- */

/* Bytes of one weight matrix [od][K] in the given type; 0 if invalid. */
int64_t oracle_weight_bytes(int qtype, int64_t od, int64_t K)
{
    int bb = block_bytes(qtype);
    if (!bb || od < 0 || K < 0 || K % 256) return 0;
    return od * (K / 256) * bb;
}

/* Dequantize W [od][K] into f64, row-major. */
int oracle_dequantize(int qtype, const uint8_t *W, int64_t od, int64_t K, double *out)
{
    int bb = block_bytes(qtype);
    if (!bb) return ORACLE_EQTYPE;
    if (od < 0 || K <= 0 || K % 256) return ORACLE_ESHAPE;
    int64_t nsb = K / 256;
    for (int64_t r = 0; r < od; r++)
        for (int64_t b = 0; b < nsb; b++) {
            const uint8_t *blk = W + (r * nsb + b) * bb;
            for (int e = 0; e < 256; e++)
                out[r * K + b * 256 + e] =
                    qtype == ORACLE_Q4_K ? q4k_weight(blk, e) : q6k_weight(blk, e);
        }
    return ORACLE_OK;
}

/*
 * q8_1 quantization of x [nt][K] ([MOJO] "The GPU path": int8 per value, one
 * f32 scale per 32 and scale*sum(q) next to it; [CH04] sec. 3.4: max, scale,
 * round).  xq [nt][K] int8; xds [nt][K/32][2] = (d, s).
 */
int oracle_quantize_q8_1(const float *x, int64_t nt, int64_t K, int8_t *xq, float *xds)
{
    if (nt < 0 || K <= 0 || K % 32) return ORACLE_ESHAPE;
    int64_t nb = K / 32;
    for (int64_t t = 0; t < nt; t++)
        for (int64_t b = 0; b < nb; b++) {
            const float *xb = x + t * K + b * 32;
            int8_t *qb = xq + t * K + b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            int sum = 0;
            for (int i = 0; i < 32; i++) {
                int q = 0;
                if (d != 0.0f) {
                    float r = xb[i] / d;
                    q = (int)nearbyintf(r); /* default rounding: ties to even */
                    if (q > 127) q = 127;
                    if (q < -127) q = -127;
                }
                qb[i] = (int8_t)q;
                sum += q;
            }
            xds[2 * (t * nb + b) + 0] = d;
            xds[2 * (t * nb + b) + 1] = d * (float)sum;
        }
    return ORACLE_OK;
}

/*
 * Exact int32 block dots.
 *   Q4_K: D[t][r][j] = sum_{i<32} nibble(32j+i) * q[t][32j+i]   (j < K/32)
 *         (the nibble is not centred; the min comes off through s).
 *   Q6_K: D[t][r][g] = sum_{i<16} (q6(16g+i) - 32) * q[t][16g+i] (g < K/16).
 * dots is [nt][od][ngroups], ngroups = K/32 (Q4_K) or K/16 (Q6_K).
 */
int oracle_block_dots(int qtype, const uint8_t *W, const int8_t *xq, int64_t od, int64_t K,
                      int64_t nt, int32_t *dots)
{
    int bb = block_bytes(qtype);
    if (!bb) return ORACLE_EQTYPE;
    if (od < 0 || nt < 0 || K <= 0 || K % 256) return ORACLE_ESHAPE;
    int64_t nsb = K / 256;
    int gsz = qtype == ORACLE_Q4_K ? 32 : 16;
    int64_t ng = K / gsz;
    for (int64_t t = 0; t < nt; t++)
        for (int64_t r = 0; r < od; r++)
            for (int64_t g = 0; g < ng; g++) {
                int64_t k0 = g * gsz;
                const uint8_t *blk = W + (r * nsb + k0 / 256) * bb;
                int32_t acc = 0;
                for (int i = 0; i < gsz; i++) {
                    int e = (int)((k0 + i) % 256);
                    int w = qtype == ORACLE_Q4_K ? q4k_nibble(blk + 16, e) : q6k_q(blk, e) - 32;
                    acc += w * (int32_t)xq[t * K + k0 + i];
                }
                dots[(t * od + r) * ng + g] = acc;
            }
    return ORACLE_OK;
}

/* One output row r for all tokens, from quantized activations. */
static void matmul_row(int qtype, const uint8_t *W, const int8_t *xq, const float *xds,
                       int64_t od, int64_t K, int64_t nt, int64_t r, float *out)
{
    int bb = block_bytes(qtype);
    int64_t nsb = K / 256;
    int64_t nb32 = K / 32;
    for (int64_t t = 0; t < nt; t++) {
        double acc = 0.0;
        for (int64_t b = 0; b < nsb; b++) {
            const uint8_t *blk = W + (r * nsb + b) * bb;
            const int8_t *q = xq + t * K + b * 256;
            if (qtype == ORACLE_Q4_K) {
                /* sum w x = d*sc*dx * sum(q*qx) - dmin*m * (dx*sum(qx))  ([MOJO]) */
                double d = half_to_double(load_u16(blk));
                double dmin = half_to_double(load_u16(blk + 2));
                for (int j = 0; j < 8; j++) {
                    int sc, m;
                    q4k_scale_min(blk + 4, j, &sc, &m);
                    int32_t D = 0;
                    for (int i = 0; i < 32; i++)
                        D += q4k_nibble(blk + 16, 32 * j + i) * (int32_t)q[32 * j + i];
                    double dx = xds[2 * (t * nb32 + b * 8 + j) + 0];
                    double s = xds[2 * (t * nb32 + b * 8 + j) + 1];
                    acc += d * sc * dx * D - dmin * m * s;
                }
            } else {
                /* sum w x = d*sc_g*dx * sum((q-32)*qx) per 16-value group */
                double d = half_to_double(load_u16(blk + 208));
                for (int g = 0; g < 16; g++) {
                    int32_t D = 0;
                    for (int i = 0; i < 16; i++)
                        D += (q6k_q(blk, 16 * g + i) - 32) * (int32_t)q[16 * g + i];
                    double dx = xds[2 * (t * nb32 + b * 8 + g / 2) + 0];
                    acc += d * q6k_scale(blk, g) * dx * D;
                }
            }
        }
        out[t * od + r] = (float)acc;
    }
}

struct row_job {
    int qtype;
    const uint8_t *W;
    const int8_t *xq;
    const float *xds;
    int64_t od, K, nt, r0, r1;
    float *out;
};

static void *row_worker(void *arg)
{
    struct row_job *j = (struct row_job *)arg;
    for (int64_t r = j->r0; r < j->r1; r++)
        matmul_row(j->qtype, j->W, j->xq, j->xds, j->od, j->K, j->nt, r, j->out);
    return NULL;
}

/*
 * out [nt][od] f32 from W and the q8_1 activations (xq, xds).  Rows are split
 * over nthreads POSIX threads (row ranges only; the arithmetic of every output
 * is the single-threaded one).
 */
int oracle_matmul_q8_1(int qtype, const uint8_t *W, const int8_t *xq, const float *xds,
                       int64_t od, int64_t K, int64_t nt, float *out, int nthreads)
{
    if (!block_bytes(qtype)) return ORACLE_EQTYPE;
    if (od < 0 || nt < 0 || K <= 0 || K % 256) return ORACLE_ESHAPE;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > od) nthreads = od > 0 ? (int)od : 1;
    struct row_job *jobs = (struct row_job *)calloc((size_t)nthreads, sizeof(*jobs));
    pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(*tid));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return ORACLE_ENOMEM;
    }
    for (int i = 0; i < nthreads; i++) {
        jobs[i] = (struct row_job){qtype, W, xq, xds, od, K, nt,
                                   od * i / nthreads, od * (i + 1) / nthreads, out};
    }
    int started = 0;
    for (int i = 1; i < nthreads; i++) {
        if (pthread_create(&tid[i], NULL, row_worker, &jobs[i]) != 0) break;
        started = i;
    }
    row_worker(&jobs[0]);
    for (int i = 1; i <= started; i++) pthread_join(tid[i], NULL);
    for (int i = started + 1; i < nthreads; i++) row_worker(&jobs[i]); /* threads we could not start */
    free(jobs);
    free(tid);
    return ORACLE_OK;
}

/* The whole method from f32 activations: quantize, then the matmul. */
int oracle_matmul(int qtype, const uint8_t *W, const float *x, int64_t od, int64_t K, int64_t nt,
                  float *out, int nthreads)
{
    if (!block_bytes(qtype)) return ORACLE_EQTYPE;
    if (od < 0 || nt < 0 || K <= 0 || K % 256) return ORACLE_ESHAPE;
    int8_t *xq = (int8_t *)malloc((size_t)(nt * K) + 1);
    float *xds = (float *)malloc(sizeof(float) * (size_t)(nt * (K / 32) * 2) + 1);
    if (!xq || !xds) {
        free(xq);
        free(xds);
        return ORACLE_ENOMEM;
    }
    int rc = oracle_quantize_q8_1(x, nt, K, xq, xds);
    if (rc == ORACLE_OK) rc = oracle_matmul_q8_1(qtype, W, xq, xds, od, K, nt, out, nthreads);
    free(xq);
    free(xds);
    return rc;
}
