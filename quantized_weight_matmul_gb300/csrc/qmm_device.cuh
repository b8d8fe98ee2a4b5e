// qmm_device.cuh -- device-side helpers shared by the library's kernels:
// f16 field reads, the Q4_K 6-bit (scale, min) unpack, and thin inline-PTX
// wrappers for mbarrier, TMA / bulk copies and tcgen05 (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "qmm.h"

namespace qmm {

constexpr int kQ4KBytes = 144;  // d, dmin, scales[12], qs[128]
constexpr int kQ6KBytes = 210;  // ql[128], qh[64], scales[16], d

// Record the first error code a kernel reports (0 -> code); later codes are dropped.
__device__ __forceinline__ void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits16) {
  return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xFFFFu)));
}

// The (scale, min) pairs of sub-blocks 2p and 2p+1 from the header
// words holding scales[0..11] ("llama.cpp MMQ", sec. 6): sub-blocks 0-3 keep
// both 6-bit codes in bytes j and j+4; sub-blocks 4-7 keep the low 4 bits in
// the nibbles of byte j+4 and the top 2 bits in the top of bytes j-4 / j.
// Returns the two codes of each kind in the low two bytes.
__device__ __forceinline__ void q4k_pair_codes(uint32_t w1, uint32_t w2, uint32_t w3, int p, uint32_t& sc2,
                                               uint32_t& m2) {
  const uint32_t sh = 16u * (p & 1);
  const uint32_t t1 = (w1 >> sh) & 0xFFFFu, t2 = (w2 >> sh) & 0xFFFFu, t3 = (w3 >> sh) & 0xFFFFu;
  const uint32_t sc_low = t1 & 0x3F3Fu, m_low = t2 & 0x3F3Fu;
  const uint32_t sc_high = (t3 & 0x0F0Fu) | ((t1 >> 2) & 0x3030u);
  const uint32_t m_high = ((t3 >> 4) & 0x0F0Fu) | ((t2 >> 2) & 0x3030u);
  sc2 = p < 2 ? sc_low : sc_high;
  m2 = p < 2 ? m_low : m_high;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ------------------------------------------- programmatic dependent launch --
// Wait until the preceding grid in the stream has completed and its memory
// is visible (a no-op when the kernel was not launched as a dependent).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next grid in the stream start its prologue.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Packed pairs of f32 (one 64-bit register pair): one FMA-pipe instruction
// per two outputs.
typedef unsigned long long f2;
__device__ __forceinline__ f2 pk2(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 upk2(f2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c) {
  f2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2 mul2(f2 a, f2 b) {
  f2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Per-warpgroup register budgets (all four warps of the warpgroup execute
// it): a warpgroup may give registers back to the block's pool, or take them
// from it.  The block's pool is what it was launched with (threads x the
// kernel's register count), so the budgets of all warpgroups must add up to
// no more than that, or an increase would wait for registers forever.
template <uint32_t N>
__device__ __forceinline__ void regs_release() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_take() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------ timing ----
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------ mbarrier --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, "
      "p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared abort state of one CTA: a flag every wait polls, the device status
// word, and the deadline after which a wait gives up.
struct Guard {
  volatile int* abort_flag;  // shared memory
  int* status;               // global
  uint64_t deadline_ns;
};

// Bounded wait for phase `parity` of barrier `bar`.  Returns false (and raises
// the CTA's abort flag and QMM_ETIMEOUT) once the deadline passes, or false
// at once when another role already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Guard& g) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*g.abort_flag) return false;
    if ((it & 63u) == 0 && global_ns() > g.deadline_ns) {
      *g.abort_flag = 1;
      report(g.status, QMM_ETIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA ----
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// q8_1 codes of N values of one 32-value block whose scale is
// d = fl(amax/127): q = round-half-even(fl(x/d)), clamped to [-127, 127] --
// the IEEE quotient rounded to the nearest integer -- without a division per
// value.  With r = fl(1/d), y = fl(x*r) is within |x/d| * 2^-23 < 1.6e-5 of
// x/d (|x/d| <= 127.00001), and fl(x/d) within 2^-24 * |x/d| < 7.6e-6 of it,
// so when y is more than 1e-4 away from every half-integer, y and fl(x/d) lie
// inside the same rounding interval and rint(y) is the code.  rint(y) is taken
// by adding 1.5 * 2^23: the sum lies in [2^23, 2^24), where the f32 spacing
// is 1, so the addition rounds y to an integer, ties to even, and the low bits
// of the sum hold that integer in two's complement.  |y| < 127.5 here, so no
// clamp is needed.  A value that close to a half-integer (or every value, when
// 1/d overflows) takes the correctly rounded division instead; the warp votes
// first so that the divisions run only when some lane needs one.  All 32
// lanes of the warp must call this together.
//
// Output: c[i] is a word whose low byte is code i (two's complement).
template <int N>
__device__ __forceinline__ void q8_code_words(const float (&v)[N], float d, uint32_t (&c)[N]) {
  static_assert(N <= 32, "one bit per value");
  constexpr float kRound = 0x1.8p23f;  // 1.5 * 2^23
  uint32_t near = 0;
#pragma unroll
  for (int i = 0; i < N; ++i) c[i] = 0;
  if (d != 0.0f) {
    const float r = __frcp_rn(d);
    if (!(r < INFINITY)) near = N == 32 ? 0xFFFFFFFFu : (1u << N) - 1u;
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float y = __fmul_rn(v[i], r);
      const float t = __fadd_rn(y, kRound);
      const float n = __fsub_rn(t, kRound);
      if (fabsf(fabsf(y - n) - 0.5f) <= 1e-4f) near |= 1u << i;
      c[i] = __float_as_uint(t);
    }
  }
  if (__any_sync(0xffffffffu, near != 0)) {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (near & (1u << i)) c[i] = (uint32_t)max(-127, min(127, __float2int_rn(__fdiv_rn(v[i], d))));
  }
}

// The low bytes of four words, packed in order into one word.
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  uint32_t ab, cd, r;
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(ab) : "r"(a), "r"(b));
  asm("prmt.b32 %0, %1, %2, 0x0040;" : "=r"(cd) : "r"(c), "r"(d));
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(r) : "r"(ab), "r"(cd));
  return r;
}

// Dot product of the four unsigned bytes of a with the four signed bytes of b,
// plus c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// n consecutive 32-bit words starting at byte offset `off` (even) of `base`
// (4-byte aligned), realigned when off % 4 == 2.
template <int N>
__device__ __forceinline__ void load_words_even(const uint8_t* base, int off, uint32_t (&out)[N]) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(base + (off & ~3));
  if (off & 2) {
    uint32_t prev = p[0];
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const uint32_t nxt = p[i + 1];
      out[i] = prmt(prev, nxt, 0x5432u);
      prev = nxt;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = p[i];
  }
}

// The same words without a branch: N + 1 aligned words are read whatever the
// offset, and each output takes its bytes through a PRMT whose selector
// depends on the offset -- for lanes of one warp whose offsets differ in
// alignment (a branch would run both paths one after the other).  Reads one
// word past the N that an aligned offset needs; the caller's row must hold it.
template <int N>
__device__ __forceinline__ void load_words_even_bf(const uint8_t* base, int off, uint32_t (&out)[N]) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(base + (off & ~3));
  const uint32_t sel = (off & 2) ? 0x5432u : 0x3210u;
  uint32_t prev = p[0];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint32_t nxt = p[i + 1];
    out[i] = prmt(prev, nxt, sel);
    prev = nxt;
  }
}

// Rows whose pitch is not a multiple of 16 bytes (Q6_K with K % 2048 != 0)
// cannot be described by a TMA tensor map; they are staged row by row as
// the 16-byte-aligned window [start & ~15, (end + 15) & ~15) around the bytes
// [start, end) of a matrix of `total` bytes.  The window is cut at the
// matrix's last 16-byte boundary so that no copy reads past the matrix; the
// (even, at most 14) bytes past that boundary are copied here with ordinary
// 2-byte loads into their place in `dst`, the window's first byte.  Returns
// the byte range left to the bulk copy (empty when a1 <= a0).
struct RowWindow {
  size_t a0, a1;
};
__device__ __forceinline__ RowWindow stage_row_window(size_t start, size_t end, size_t total, uint8_t* dst,
                                                      const uint8_t* W) {
  RowWindow w{start & ~(size_t)15, (end + 15) & ~(size_t)15};
  const size_t cap = total & ~(size_t)15;
  if (w.a1 > cap) {
    for (size_t o = cap > w.a0 ? cap : w.a0; o < end; o += 2)
      *reinterpret_cast<uint16_t*>(dst + (o - w.a0)) = __ldg(reinterpret_cast<const uint16_t*>(W + o));
    w.a1 = cap;
  }
  return w;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Hand a shared-memory stage that this warp has READ back to a producer that
// refills it with TMA / bulk copies.  Those writes go through the async
// proxy, so the warp's generic-proxy reads are fenced against them first:
// without the fence a refill can land before the last reads are performed
// (seen as a few wrong values in the tail of a warp's reads when the
// producer runs right behind the consumers).  Whole warp; lane 0 arrives.
__device__ __forceinline__ void release_stage(uint32_t empty_bar) {
  fence_proxy_async();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar);
}

// ------------------------------------------------------------ tcgen05 ----
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (all >> 4), version 1, layout type in bits 61-63
// (0 = no swizzle, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(layout & 7u) << 61;
  return d;
}

// Instruction descriptor of kind::f16 with f32 accumulation, f16 A and B,
// both K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same MMA with A read from tensor memory: `tmem_a` is the TMEM address
// of the A tile (row i of A in lane i, K along the columns, two f16 / bf16
// per 32-bit column, the lower k in the low half).
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Store 32 (or 16) consecutive 32-bit columns of this warp's 32 TMEM lanes
// (lane = the thread's lane within the warp's lane quarter).  Completion is
// awaited with tc_wait_st before the columns are handed to another thread.
__device__ __forceinline__ void tc_st_32x32_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 32 consecutive f32 columns of this warp's 32 TMEM lanes, loaded and waited
// for in ONE asm statement.  tcgen05.ld writes its destination registers
// asynchronously and nothing orders a read of them before
// tcgen05.wait::ld: with the load and the wait in separate statements the
// compiler regards the registers as written at the load and may copy or
// spill one of them in between, which reads it before the data has arrived
// (wrong values in a few columns of one warp's load, more often under
// register pressure).  Here the outputs exist only after the wait.
__device__ __forceinline__ void tc_ld_32x32_sync(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]),
        "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]),
        "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

}  // namespace qmm
