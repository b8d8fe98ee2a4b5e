"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

* q8_1 codes and scales: bit-exact.
* int32 block dots (MMVQ and tensor-core dot code): bit-exact.
* fp32 outputs: within 1e-4 of each output row's L2 norm (gpu_helpers).
Shapes span several tiles with ragged tails, the edge cases (one row, one
super-block, one token) and the five workload families at full size (the
largest on a deterministic row sample).
"""
import numpy as np
import pytest

import brute
import quantized_weight_matmul_gb300 as qmm
from gpu_helpers import assert_close_rows, dev, ora, oracle_rows, row_sample, threads
from quantized_weight_matmul_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

Q4_K, Q6_K = qmm.Q4_K, qmm.Q6_K


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    qmm.load()


def _case(qtype, od, K, nt, outliers=False, seed=0):
    c = synth.Case(qtype, od, K, nt, outliers, seed)
    return c.generate()


# ------------------------------------------------------------- quantize ---

@pytest.mark.parametrize("nt,K,outliers", [(1, 512, False), (8, 4096, True), (513, 4096, True),
                                           (2048, 14336, False), (3, 96, False)])
def test_quantize_bit_exact(nt, K, outliers):
    x = synth.activations(nt, K, np.random.default_rng(nt + K), outliers)
    if nt >= 3:
        x[1, :64] = 0.0           # zero blocks
        x[2, 32:64] = -1.25       # constant block
        x[2, 0:32] = 0.0
        x[2, 5] = 381.0           # d = 3 exactly
        x[2, 6:10] = [1.5 * 3, 2.5 * 3, -0.5 * 3, 7.5 * 3]  # exact .5 quotients
    xq, xds = qmm.quantize_q8_1(dev(x, torch))
    oq, ods = ora().quantize_q8_1(x)
    assert np.array_equal(xq.cpu().numpy(), oq)
    assert np.array_equal(xds.cpu().numpy().view(np.uint32), ods.view(np.uint32))


def _near_tie_blocks(K=4096, seed=7):
    """One token of K values whose quotients x/d sit on, or a few ulps beside,
    half-integers -- where the rounding of the IEEE quotient is decided -- plus
    a block whose scale is subnormal (its reciprocal overflows) and a zero
    block."""
    rng = np.random.default_rng(seed)
    x = np.zeros(K, dtype=np.float32)
    nb = K // 32
    for b in range(nb - 2):
        amax = np.float32(rng.choice([127.0, 100.0, 3.7, 1e-3, 55.5]) * rng.uniform(0.5, 2.0))
        d = np.float32(amax / np.float32(127.0))
        blk = np.empty(32, dtype=np.float32)
        blk[0] = amax if b % 2 else -amax
        for i in range(1, 32):
            h = np.float32(rng.integers(-126, 126) + 0.5)
            v = np.float32(h * d)
            steps = int(rng.integers(-3, 4))  # 0: on the tie's product; else a few ulps aside
            for _ in range(abs(steps)):
                v = np.nextafter(v, np.float32(np.inf) if steps > 0 else np.float32(-np.inf), dtype=np.float32)
            blk[i] = v if abs(v) <= amax else np.float32(h * d)
        x[32 * b:32 * (b + 1)] = blk
    x[32 * (nb - 2):32 * (nb - 1)] = np.float32(1e-40) * np.arange(-16, 16, dtype=np.float32)  # subnormal scale
    return x[None, :]  # last block stays zero


def test_quantize_near_ties_bit_exact():
    """Values whose quotients lie on or within a few ulps of a rounding
    boundary: the quantizer and the fused decode kernel give the IEEE codes."""
    x = _near_tie_blocks()
    oq, ods = ora().quantize_q8_1(x)
    xq, xds = qmm.quantize_q8_1(dev(x, torch))
    assert np.array_equal(xq.cpu().numpy(), oq)
    assert np.array_equal(xds.cpu().numpy().view(np.uint32), ods.view(np.uint32))
    # the fused quantize + MMVQ route writes the same codes
    W, _ = synth.Case(Q4_K, 256, x.shape[1], 1).generate()
    assert qmm.qmm_matmul_path(Q4_K, 256, x.shape[1], 1) == qmm.QMM_PATH_FUSED_MMVQ
    _, fq, fds = qmm.matmul(Q4_K, dev(W, torch), dev(x, torch), 256, return_q8=True)
    assert np.array_equal(fq.cpu().numpy(), oq)
    assert np.array_equal(fds.cpu().numpy().view(np.uint32), ods.view(np.uint32))


# ------------------------------------------------------------ block dots ---

@pytest.mark.parametrize("od,K,nt", [(256, 512, 1), (256, 512, 8), (1000, 768, 3), (64, 14336, 2),
                                     (4096, 4096, 1), (1, 256, 5)])
def test_gemv_block_dots_bit_exact(od, K, nt):
    W, x = _case(Q4_K, od, K, nt, seed=od)
    xq, xds = ora().quantize_q8_1(x)
    d = qmm.block_dots(Q4_K, dev(W, torch), dev(xq, torch), dev(xds, torch), od, path=0)
    assert np.array_equal(d.cpu().numpy(), ora().block_dots(Q4_K, W, xq, od))


@pytest.mark.parametrize("od,K,nt", [(256, 2048, 1), (300, 4096, 8), (1, 2048, 3), (4096, 4096, 1),
                                     (130, 6144, 5)])
def test_gemv_q6k_block_dots_bit_exact(od, K, nt):
    """Q6_K through the MMVQ dot code: sum over each 16-value group of
    (q6 - 32) * q8, exact int32."""
    W, x = _case(Q6_K, od, K, nt, seed=od + 1)
    xq, xds = ora().quantize_q8_1(x)
    d = qmm.block_dots(Q6_K, dev(W, torch), dev(xq, torch), dev(xds, torch), od, path=0)
    assert np.array_equal(d.cpu().numpy(), ora().block_dots(Q6_K, W, xq, od))


def _tc_dots_expected(qtype, W, xq, od):
    """What the tensor-core kernel's accumulator holds per 32-value block, from
    the oracle's exact block dots and the scales decoded by the separate numpy
    restatement: Q4_K sc_j * D_j; Q6_K sc_2b * D_2b + sc_2b+1 * D_2b+1; zero
    for a super-block whose d is zero (the kernel folds no scale there)."""
    D = ora().block_dots(qtype, W, xq, od).astype(np.int64)
    nt, K = xq.shape
    nsb = K // 256
    if qtype == Q4_K:
        blocks = W.reshape(od, nsb, 144)
        sc, _ = brute.q4k_codes(blocks)
        dz = brute.f16_field(blocks, 0) == 0
        sc = np.where(dz[..., None], 0, sc).reshape(od, nsb * 8)
        return D * sc[None]
    blocks = W.reshape(od, nsb, 210)
    sc = brute.q6k_scales(blocks)
    dz = brute.f16_field(blocks, 208) == 0
    sc = np.where(dz[..., None], 0, sc).reshape(od, nsb * 16)
    return (D * sc[None]).reshape(nt, od, K // 32, 2).sum(-1)


@pytest.mark.parametrize("qtype,od,K,nt", [(Q4_K, 300, 512, 70), (Q4_K, 129, 1024, 200),
                                           (Q4_K, 128, 256, 1), (Q4_K, 257, 2048, 64),
                                           (Q6_K, 300, 2048, 70), (Q6_K, 130, 4096, 131),
                                           (Q6_K, 200, 2048, 33), (Q6_K, 129, 2048, 64)])
def test_gemm_block_dots_bit_exact(qtype, od, K, nt):
    """The tensor-core kernel's exact integer sums, as the product kernel
    forms them (scale folded into the weight operand; the 64-token tile up to
    64 tokens, the 128-token tile above), against the oracle's block dots."""
    W, x = _case(qtype, od, K, nt, seed=od + nt)
    xq, xds = ora().quantize_q8_1(x)
    d = qmm.block_dots(qtype, dev(W, torch), dev(xq, torch), dev(xds, torch), od, path=1)
    torch.cuda.synchronize()
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK
    assert np.array_equal(d.cpu().numpy().astype(np.int64), _tc_dots_expected(qtype, W, xq, od))


@pytest.mark.parametrize("qtype,nt", [(Q4_K, 40), (Q4_K, 100), (Q6_K, 40), (Q6_K, 100)])
def test_gemm_block_dots_extremes(qtype, nt):
    """Largest sums the folded operands can produce, where an inexact f32
    accumulation would show: Q4_K sc = 63 with all nibbles 15, Q6_K q = 0
    (q - 32 = -32) with scale -128 and q = 63 with scale 127, against codes of
    +-127 (|sum| up to 32*32*128*127 < 2^24), plus super-blocks with d = 0
    and mixed signs."""
    od, K = 200, 2048
    W, x = _case(qtype, od, K, nt, seed=5)
    nsb = K // 256
    if qtype == Q4_K:
        Wb = W.reshape(od, nsb, 144).copy()
        Wb[0::3, :, 4:16] = brute.pack_q4k_codes([63] * 8, [63] * 8)  # sc = m = 63
        Wb[0::3, :, 16:] = 0xFF                                         # nibbles 15
        Wb[1::7, 1, 0:2] = 0                                            # d = 0
    else:
        Wb = W.reshape(od, nsb, 210).copy()
        Wb[0::3, :, 0:192] = 0                                          # q = 0
        Wb[0::3, :, 192:208] = 0x80                                     # scale -128
        Wb[1::3, :, 0:192] = 0xFF                                       # q = 63
        Wb[1::3, :, 192:208] = 0x7F                                     # scale 127
        Wb[2::7, 1, 208:210] = 0                                        # d = 0
    W = Wb.reshape(od, -1)
    x = np.where(np.arange(K)[None, :] % 64 < 32, 1.0, -1.0).astype(np.float32) * np.ones((nt, 1), np.float32)
    x[1::2] *= -1.0
    x[2, 96:128] = 0.0
    xq, xds = ora().quantize_q8_1(x)
    assert np.abs(xq).max() == 127
    d = qmm.block_dots(qtype, dev(W, torch), dev(xq, torch), dev(xds, torch), od, path=1)
    torch.cuda.synchronize()
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK
    want = _tc_dots_expected(qtype, W, xq, od)
    assert np.abs(want).max() > (2 ** 23 if qtype == Q6_K else 2 ** 19)
    assert np.array_equal(d.cpu().numpy().astype(np.int64), want)


@pytest.mark.parametrize("qtype,od,K,nt", [(Q4_K, 256, 512, 1), (Q4_K, 300, 768, 3), (Q4_K, 1000, 4096, 8),
                                           (Q4_K, 17, 14336, 8), (Q4_K, 4096, 4096, 13), (Q4_K, 33, 2304, 16),
                                           (Q6_K, 256, 2048, 2), (Q6_K, 300, 4096, 8), (Q6_K, 33, 6144, 12), (Q6_K, 33, 4096, 16),
                                           (Q6_K, 1, 2048, 5), (Q6_K, 4096, 4096, 11)])
def test_mma_block_dots_bit_exact(qtype, od, K, nt):
    """The warp-MMA MMVQ dot code (subnormal-f16 weight codes times f16
    activation codes, f32 accumulation): every block dot exact.  Shapes cover
    a ragged last row tile, a K that ends inside a 2048-k stage, the raw-byte
    activation layout (K = 14336) and 9..16 tokens (two token tiles)."""
    W, x = _case(qtype, od, K, nt, seed=od + 3 * nt)
    xq, xds = ora().quantize_q8_1(x)
    d = qmm.block_dots(qtype, dev(W, torch), dev(xq, torch), dev(xds, torch), od, path=2)
    torch.cuda.synchronize()
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK
    assert np.array_equal(d.cpu().numpy(), ora().block_dots(qtype, W, xq, od))


# ---------------------------------------------------------------- GEMV ---

@pytest.mark.parametrize("od,K,nt", [(256, 512, 1), (256, 512, 8), (1000, 768, 5), (1, 256, 2),
                                     (4096, 4096, 1), (11008, 4096, 1), (14336, 4096, 2),
                                     (14336, 4096, 4), (14336, 4096, 8), (4096, 14336, 2),
                                     (4096, 14336, 4), (4096, 14336, 8), (4096, 4096, 16), (1000, 768, 11),
                                     (300, 4096, 13)])
def test_gemv_matches_oracle(od, K, nt):
    W, x = _case(Q4_K, od, K, nt, outliers=(nt == 1), seed=0)
    xq, xds = ora().quantize_q8_1(x)
    out = qmm.gemv(Q4_K, dev(W, torch), dev(xq, torch), dev(xds, torch), od)
    ref = ora().matmul_q8_1(Q4_K, W, xq, xds, od, nthreads=threads())
    assert_close_rows(out.cpu().numpy(), ref, f"gemv {od}x{K} nt={nt}")


@pytest.mark.parametrize("od,K,nt", [(256, 2048, 1), (1000, 4096, 5), (4096, 4096, 8), (129, 6144, 2),
                                     (32000, 4096, 1), (33, 2048, 7), (4096, 4096, 16), (32000, 4096, 8),
                                     (257, 2048, 12)])
def test_gemv_q6k_matches_oracle(od, K, nt):
    W, x = _case(Q6_K, od, K, nt, outliers=(nt == 1), seed=2)
    xq, xds = ora().quantize_q8_1(x)
    out = qmm.gemv(Q6_K, dev(W, torch), dev(xq, torch), dev(xds, torch), od).cpu().numpy()
    rows = row_sample(od)
    ref = oracle_rows(Q6_K, W, x, rows) if od > 4096 else ora().matmul_q8_1(Q6_K, W, xq, xds, od, nthreads=threads())
    assert_close_rows(out[:, rows] if od > 4096 else out, ref, f"q6k gemv {od}x{K} nt={nt}")


@pytest.mark.parametrize("od,K,nt,path", [(4096, 4096, 1, qmm.QMM_PATH_FUSED_MMVQ),
                                          (32000, 4096, 1, qmm.QMM_PATH_FUSED_MMVQ),
                                          (300, 2048, 3, qmm.QMM_PATH_MMVQ), (32000, 4096, 2, qmm.QMM_PATH_MMVQ),
                                          (1000, 2048, 4, qmm.QMM_PATH_MMVQ)])
def test_q6k_matmul_small_batch(od, K, nt, path):
    """Q6_K small-batch shapes through qmm_matmul: the fused quantize + dp4a
    MMVQ at nt = 1, quantize + the warp-MMA MMVQ from 2 tokens.  q8_1 outputs
    bit-exact, outputs within tolerance."""
    assert qmm.qmm_matmul_path(Q6_K, od, K, nt) == path
    W, x = _case(Q6_K, od, K, nt, outliers=True, seed=od)
    out, xq, xds = qmm.matmul(Q6_K, dev(W, torch), dev(x, torch), od, flags=qmm.QMM_FLAG_STATIC_WEIGHTS,
                              return_q8=True)
    oq, ods = ora().quantize_q8_1(x)
    assert np.array_equal(xq.cpu().numpy(), oq)
    assert np.array_equal(xds.cpu().numpy().view(np.uint32), ods.view(np.uint32))
    rows = row_sample(od)
    ref = oracle_rows(Q6_K, W, x, rows)
    assert_close_rows(out.cpu().numpy()[:, rows], ref, f"fused q6k {od}x{K} nt={nt}")
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK


# ---------------------------------------------------------------- GEMM ---

@pytest.mark.parametrize("qtype,od,K,nt", [(Q4_K, 384, 1024, 9), (Q4_K, 384, 1024, 64),
                                           (Q4_K, 384, 1024, 65), (Q4_K, 300, 1536, 130),
                                           (Q4_K, 200, 512, 300), (Q4_K, 1, 256, 1),
                                           (Q4_K, 1000, 768, 5), (Q6_K, 300, 2048, 33),
                                           (Q6_K, 257, 4096, 200), (Q6_K, 64, 2048, 1)])
def test_gemm_matches_oracle(qtype, od, K, nt):
    W, x = _case(qtype, od, K, nt, outliers=True, seed=nt)
    xq, xds = ora().quantize_q8_1(x)
    out = qmm.gemm(qtype, dev(W, torch), dev(xq, torch), dev(xds, torch), od)
    ref = ora().matmul_q8_1(qtype, W, xq, xds, od, nthreads=threads())
    assert_close_rows(out.cpu().numpy(), ref, f"gemm q{qtype} {od}x{K} nt={nt}")
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK


@pytest.mark.parametrize("qtype,nt", [(Q4_K, 1), (Q4_K, 8), (Q4_K, 70), (Q6_K, 1), (Q6_K, 8), (Q6_K, 70)])
def test_degenerate_blocks_match_oracle(qtype, nt):
    """Degenerate blocks on every route (fused MMVQ at nt = 1, warp-MMA MMVQ at
    nt = 8, tensor-core GEMM at nt = 70): super-blocks whose scale d is zero
    (also a row's first one, where the GEMM epilogue has no running scale yet),
    Q4_K super-blocks with dmin = 0, all-zero blocks, Q6_K group scales 0 and
    -128, and zero activation blocks and tokens."""
    od, K = 300, 4096
    W, x = _case(qtype, od, K, nt, outliers=True, seed=11)
    nsb, bb = K // 256, (144 if qtype == Q4_K else 210)
    Wb = W.reshape(od, nsb, bb).copy()
    r, b = np.meshgrid(np.arange(od), np.arange(nsb), indexing="ij")
    dpos = slice(0, 2) if qtype == Q4_K else slice(208, 210)
    Wb[(r + b) % 3 == 0, dpos] = 0                      # d = 0 (b = 0 for every third row)
    if qtype == Q4_K:
        Wb[(r + 2 * b) % 5 == 0, 2:4] = 0               # dmin = 0
    else:
        Wb[::2, :, 192] = 0                             # group scale 0
        Wb[::2, :, 193] = 0x80                          # group scale -128
    Wb[(7 * r + b) % 11 == 0, :] = 0                    # all-zero blocks
    W = Wb.reshape(od, nsb * bb)
    x = x.copy()
    x[:, 96:128] = 0.0                                  # a zero block in every token
    if nt > 1:
        x[nt // 2] = 0.0                                # a zero token
    out = qmm.matmul(qtype, dev(W, torch), dev(x, torch), od).cpu().numpy()
    ref = ora().matmul(qtype, W, x, od, nthreads=threads())
    assert_close_rows(out, ref, f"degenerate q{qtype} nt={nt}")
    if nt > 1:
        assert not out[nt // 2].any()
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK


def _full_size(case):
    W, x = case.generate()
    Wd, xd = dev(W, torch), dev(x, torch)
    out = qmm.matmul(case.qtype, Wd, xd, case.od).cpu().numpy()
    rows = row_sample(case.od, max_rows=1024 if case.macs > 2e10 else 4096)
    ref = oracle_rows(case.qtype, W, x, rows)
    return assert_close_rows(out[:, rows], ref, case.name)


@pytest.mark.parametrize("case", [c for w in ("tiny_q4k", "decode_gemv_q4k", "mmvq_q4k")
                                  for c in synth.WORKLOADS[w].cases], ids=lambda c: c.name)
def test_workload_small_batch(case):
    _full_size(case)


@pytest.mark.parametrize("case", synth.WORKLOADS["prefill_gemm_q4k"].cases, ids=lambda c: c.name)
def test_workload_prefill(case):
    _full_size(case)
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK


@pytest.mark.parametrize("case", synth.WORKLOADS["skinny_q6k"].cases, ids=lambda c: c.name)
def test_workload_skinny_q6k(case):
    _full_size(case)


@pytest.mark.parametrize("od,K,nt,flags", [(4096, 4096, 1, 0), (4096, 4096, 1, 1), (1000, 512, 3, 1),
                                           (300, 768, 4, 0), (11008, 4096, 2, 1), (64, 14336, 1, 1),
                                           (129, 2304, 2, 0), (2048, 4096, 8, 1), (1000, 2048, 6, 0),
                                           (300, 14336, 2, 1), (777, 1280, 7, 0), (4096, 4096, 5, 1)])
def test_fused_quantize_matmul(od, K, nt, flags):
    """qmm_matmul on the decode and small-batch shapes -- the fused quantize +
    dp4a MMVQ kernel up to 4 tokens, quantize + the warp-MMA MMVQ from 5:
    q8_1 outputs bit-exact, matmul output within tolerance, with and without
    the static-weights flag."""
    want = qmm.QMM_PATH_FUSED_MMVQ if nt <= 4 else qmm.QMM_PATH_MMVQ
    assert qmm.qmm_matmul_path(Q4_K, od, K, nt) == want
    W, x = _case(Q4_K, od, K, nt, outliers=True, seed=od + K)
    out, xq, xds = qmm.matmul(Q4_K, dev(W, torch), dev(x, torch), od, flags=flags, return_q8=True)
    oq, ods = ora().quantize_q8_1(x)
    assert np.array_equal(xq.cpu().numpy(), oq)
    assert np.array_equal(xds.cpu().numpy().view(np.uint32), ods.view(np.uint32))
    ref = ora().matmul_q8_1(Q4_K, W, oq, ods, od, nthreads=threads())
    assert_close_rows(out.cpu().numpy(), ref, f"fused {od}x{K} nt={nt}")
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK


def test_repeated_calls_are_bitwise_deterministic():
    """Back-to-back calls on every path, interleaved with a large GEMM, give
    bit-identical outputs (no stale or racing data between launches)."""
    cases = [synth.Case(Q4_K, 4096, 4096, 1, True), synth.Case(Q4_K, 2048, 4096, 8),
             synth.Case(Q6_K, 4096, 4096, 32), synth.Case(Q4_K, 1024, 4096, 96)]
    big = synth.Case(Q4_K, 4096, 14336, 1024, True)
    data = [(dev(W, torch), dev(x, torch)) for (W, x) in (c.generate() for c in cases)]
    Wb, xb = (dev(a, torch) for a in big.generate())
    first = [None] * len(cases)
    for it in range(6):
        if it % 2:
            qmm.matmul(big.qtype, Wb, xb, big.od, flags=qmm.QMM_FLAG_STATIC_WEIGHTS)
        for i, (c, (Wd, xd)) in enumerate(zip(cases, data)):
            o = qmm.matmul(c.qtype, Wd, xd, c.od, flags=it % 2).cpu().numpy()
            if first[i] is None:
                first[i] = o
            assert np.array_equal(o.view(np.uint32), first[i].view(np.uint32)), (c.name, it)
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK
    for c, o in zip(cases, first):
        W, x = c.generate()
        assert_close_rows(o, ora().matmul(c.qtype, W, x, c.od, nthreads=threads()), c.name)


@pytest.mark.parametrize("qtype,od,nt", [(Q6_K, 4096, 32), (Q6_K, 4096, 64), (Q6_K, 32000, 64), (Q4_K, 4096, 64),
                                         (Q4_K, 4096, 256), (Q4_K, 14336, 512)])
def test_gemm_repeats_bitwise(qtype, od, nt):
    """100 back-to-back tensor-core GEMMs of one problem are bit-identical: the
    TMEM accumulators are never overwritten before the epilogue has used them
    and no role reads a stage that is being refilled (races of that kind
    showed up as a few wrong sums in one warp's block of rows and tokens, most
    often on the 32000-row Q6_K LM head)."""
    c = synth.Case(qtype, od, 4096, nt)
    Wd, xd = (dev(a, torch) for a in c.generate())
    ws = qmm.workspace(qmm.qmm_matmul_workspace_bytes(qtype, c.od, c.K, nt), Wd.device)
    first = qmm.matmul(qtype, Wd, xd, c.od, ws=ws)
    bad = sum(int(not torch.equal(qmm.matmul(qtype, Wd, xd, c.od, ws=ws), first)) for _ in range(100))
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK
    assert bad == 0, f"{bad} of 100 repeats differ"


def test_matmul_paths_agree_at_the_boundary():
    """nt = 8 through MMVQ and through the tensor-core GEMM give the same result
    to rounding."""
    W, x = _case(Q4_K, 2048, 4096, 8, seed=3)
    Wd, xd = dev(W, torch), dev(x, torch)
    xq, xds = qmm.quantize_q8_1(xd)
    a = qmm.gemv(Q4_K, Wd, xq, xds, 2048).cpu().numpy()
    b = qmm.gemm(Q4_K, Wd, xq, xds, 2048).cpu().numpy()
    assert_close_rows(a, b.astype(np.float64), "gemv vs gemm")


# ------------------------------------------------------------- errors ---

def test_errors_and_bounded_wait():
    W, x = _case(Q4_K, 256, 512, 16, seed=1)
    Wd, xd = dev(W, torch), dev(x, torch)
    xq, xds = qmm.quantize_q8_1(xd)
    out = torch.empty((16, 256), device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    # a workspace that is too small, a bad type, a misaligned pointer
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    assert qmm.qmm_gemm(Q4_K, Wd.data_ptr(), xq.data_ptr(), xds.data_ptr(), out.data_ptr(), 256, 512, 16,
                        ws.data_ptr(), 64, st) == qmm.QMM_EWORKSPACE
    assert qmm.qmm_gemm(3, Wd.data_ptr(), xq.data_ptr(), xds.data_ptr(), out.data_ptr(), 256, 512, 16,
                        ws.data_ptr(), 64, st) == qmm.QMM_EINVAL_QTYPE
    assert qmm.qmm_gemv(Q4_K, Wd.data_ptr() + 8, xq.data_ptr(), xds.data_ptr(), out.data_ptr(), 256, 512, 8,
                        st) == qmm.QMM_EALIGN
    # a shape the MMVQ kernels refuse
    assert qmm.qmm_gemv(Q6_K, Wd.data_ptr(), xq.data_ptr(), xds.data_ptr(), out.data_ptr(), 256, 512, 17,
                        st) == qmm.QMM_EINVAL_SHAPE
    # bounded wait: a skipped producer arrival makes the waits give up and report
    assert qmm.qmm_sync_status(st) == qmm.QMM_OK
    assert qmm.qmm_debug_inject_stall(1, 200) == qmm.QMM_OK
    try:
        qmm.gemm(Q4_K, Wd, xq, xds, 256)
        assert qmm.qmm_sync_status(st) == qmm.QMM_ETIMEOUT
    finally:
        qmm.qmm_debug_inject_stall(0, 0)
    # the context is still usable and the status word was cleared
    ref = ora().matmul(Q4_K, W, x, 256)
    got = qmm.gemm(Q4_K, Wd, xq, xds, 256).cpu().numpy()
    assert qmm.qmm_sync_status(st) == qmm.QMM_OK
    assert_close_rows(got, ref, "after timeout")


@pytest.mark.parametrize("route,nt", [("fused", 1), ("fused", 3), ("staged", 2), ("mma", 8), ("mma", 13)])
def test_mmvq_bounded_wait(route, nt):
    """The MMVQ kernels' bounded waits: with the stall hook on, a skipped
    producer arrival makes their waits run out; qmm_sync_status reports
    QMM_ETIMEOUT, and the next call on the same context matches the oracle.
    Routes: the fused quantize + dp4a kernel (qmm_matmul, decode shapes), the
    staged dp4a kernel (qmm_gemv, few tokens), the warp-MMA kernel (qmm_gemv,
    5..16 tokens)."""
    od, K = 300, 4096
    W, x = _case(Q4_K, od, K, nt, outliers=True, seed=nt)
    Wd, xd = dev(W, torch), dev(x, torch)
    xq, xds = qmm.quantize_q8_1(xd)
    st = torch.cuda.current_stream().cuda_stream
    if route == "fused":
        assert qmm.qmm_matmul_path(Q4_K, od, K, nt) == qmm.QMM_PATH_FUSED_MMVQ
        run = lambda: qmm.matmul(Q4_K, Wd, xd, od)
        ref = ora().matmul(Q4_K, W, x, od, nthreads=threads())
    else:
        run = lambda: qmm.gemv(Q4_K, Wd, xq, xds, od)
        oq, ods = ora().quantize_q8_1(x)
        ref = ora().matmul_q8_1(Q4_K, W, oq, ods, od, nthreads=threads())
    assert qmm.qmm_sync_status(st) == qmm.QMM_OK
    assert qmm.qmm_debug_inject_stall(1, 200) == qmm.QMM_OK
    try:
        run()
        assert qmm.qmm_sync_status(st) == qmm.QMM_ETIMEOUT
    finally:
        qmm.qmm_debug_inject_stall(0, 0)
    got = run().cpu().numpy()
    assert qmm.qmm_sync_status(st) == qmm.QMM_OK
    assert_close_rows(got, ref, f"{route} nt={nt} after timeout")


@pytest.mark.parametrize("od,K,nt", [(300, 11008, 1), (300, 11008, 2), (300, 11008, 8), (300, 11008, 64),
                                     (257, 2304, 1), (257, 2304, 8), (257, 2304, 64), (129, 256, 70),
                                     (64, 768, 130), (33, 768, 5), (4096, 11008, 1)])
def test_q6k_any_k(od, K, nt):
    """Q6_K rows whose pitch (210*K/256 bytes) is not a multiple of 16 -- K %
    2048 != 0, e.g. K = 11008, a Llama-7B FFN-down width -- cannot be a TMA
    tensor map; every route stages them row by row (16-byte-aligned windows,
    the last row's tail by ordinary loads): the fused dp4a MMVQ at nt = 1, the
    warp-MMA MMVQ for a few tokens, the tensor-core GEMM beyond.  Outputs
    within tolerance, q8_1 bit-exact, the exact block sums of the route's dot
    code, and a deterministic repeat."""
    route = qmm.qmm_matmul_path(Q6_K, od, K, nt)
    assert route == (qmm.QMM_PATH_MMQ if nt > 16 else qmm.QMM_PATH_FUSED_MMVQ if nt == 1 else qmm.QMM_PATH_MMVQ)
    W, x = _case(Q6_K, od, K, nt, outliers=True, seed=K + nt)
    Wd, xd = dev(W, torch), dev(x, torch)
    out, xq, xds = qmm.matmul(Q6_K, Wd, xd, od, return_q8=True)
    oq, ods = ora().quantize_q8_1(x)
    assert np.array_equal(xq.cpu().numpy(), oq)
    ref = ora().matmul_q8_1(Q6_K, W, oq, ods, od, nthreads=threads())
    got = out.cpu().numpy()
    assert_close_rows(got, ref, f"q6k {od}x{K} nt={nt}")
    again = qmm.matmul(Q6_K, Wd, xd, od).cpu().numpy()
    assert np.array_equal(again.view(np.uint32), got.view(np.uint32))
    if route == qmm.QMM_PATH_MMQ:
        d = qmm.block_dots(Q6_K, Wd, dev(oq, torch), dev(ods, torch), od, path=1)
        want = _tc_dots_expected(Q6_K, W, oq, od)
    else:
        d = qmm.block_dots(Q6_K, Wd, dev(oq, torch), dev(ods, torch), od, path=0 if nt == 1 else 2)
        want = ora().block_dots(Q6_K, W, oq, od)
    torch.cuda.synchronize()
    assert qmm.qmm_sync_status(0) == qmm.QMM_OK
    assert np.array_equal(d.cpu().numpy().astype(np.int64), want.astype(np.int64))
