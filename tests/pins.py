"""Pins for the CPU oracle: facts fixed by the format definitions and by
arithmetic, independent of the oracle's own code.

Every ``pin_*`` function takes an ``oracle.Oracle`` (the real one, or a
deliberately broken build in the mutation tests) and raises AssertionError when
the oracle disagrees with the fact it checks.  Sources are cited by page title
and section:

* "llama.cpp MMQ" sec. 4 (Q4_K/Q6_K block layouts), sec. 6 (the (scale, min)
  unpack, d*sc*q - dmin*m) and sec. 7 (the IMMA count of the q-proj GEMM);
* mojo-dllm "The quantized GEMM", "The GPU path" (q8_1: one f32 scale per 32
  and scale*sum(q); nibble placement; 16-byte header) and "Weights" (the Q6_K
  zero point 32);
* minfer ch. 04 sec. 3.4 (quantize = max, scale, round).
"""
from __future__ import annotations

import os

import numpy as np

import brute
from quantized_weight_matmul_gb300 import synth

Q4_K, Q6_K = 12, 14
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def f32(v):
    return np.float32(v)


def read_golden(name: str) -> dict:
    """key = integer value lines from a golden fixture (comments start with #)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            out[k] = int(v)
    return out


def _q4k_block(d=1.0, dmin=0.0, sc=None, m=None, qs=None) -> np.ndarray:
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = np.array([d], dtype="<f2").view(np.uint8)
    blk[2:4] = np.array([dmin], dtype="<f2").view(np.uint8)
    sc = np.ones(8, np.int64) if sc is None else sc
    m = np.zeros(8, np.int64) if m is None else m
    blk[4:16] = brute.pack_q4k_codes(sc, m)
    if qs is not None:
        blk[16:144] = qs
    return blk


def _q6k_block(d=1.0, scales=None, ql=0, qh=0) -> np.ndarray:
    blk = np.zeros(210, dtype=np.uint8)
    blk[0:128] = ql
    blk[128:192] = qh
    blk[192:208] = (np.ones(16, np.int8) if scales is None
                    else np.asarray(scales, np.int8)).view(np.uint8)
    blk[208:210] = np.array([d], dtype="<f2").view(np.uint8)
    return blk


# ------------------------------------------------------------------ sizes ---

def pin_block_sizes(o):
    """144 B per Q4_K super-block and 210 B per Q6_K one, per 256 weights."""
    g = read_golden("page_numbers.txt")
    assert o.weight_bytes(Q4_K, 1, 256) == g["q4_k_block_bytes"]
    assert o.weight_bytes(Q6_K, 1, 256) == g["q6_k_block_bytes"]
    assert o.weight_bytes(Q4_K, 3584, 3584) == 3584 * 14 * g["q4_k_block_bytes"]
    assert o.weight_bytes(Q4_K, 16, 300) == 0  # K not a multiple of 256
    assert o.weight_bytes(99, 16, 256) == 0


# ------------------------------------------------------------------- q8_1 ---

def pin_q8_1_closed_forms(o):
    """Zero, constant and one-hot blocks have closed-form q8_1 encodings."""
    K = 128
    x = np.zeros((4, K), np.float32)
    x[1, :] = 0.75                      # constant block
    x[2, :32] = -3.0                    # negative constant block
    x[3, 40] = 2.5                      # one-hot inside block 1
    xq, xds = o.quantize_q8_1(x)
    # all-zero blocks: d = q = s = 0
    assert not xq[0].any() and not xds[0].any()
    d = f32(0.75) / f32(127.0)
    assert (xq[1] == 127).all()
    assert (xds[1, :, 0] == d).all() and (xds[1, :, 1] == d * f32(127 * 32)).all()
    d = f32(3.0) / f32(127.0)
    assert (xq[2, :32] == -127).all() and xds[2, 0, 0] == d
    assert xds[2, 0, 1] == d * f32(-127 * 32)
    assert not xq[2, 32:].any()
    assert xq[3, 40] == 127 and np.count_nonzero(xq[3]) == 1
    d = f32(2.5) / f32(127.0)
    assert xds[3, 1, 0] == d and xds[3, 1, 1] == d * f32(127)
    assert xds[3, 0, 0] == 0 and xds[3, 2, 0] == 0


def pin_q8_1_ties_to_even(o):
    """q = round-half-even of the true quotient x/d.

    With amax = 127 the scale is exactly 1; with amax = 889 it is exactly 7 and
    x = 7*(k + 1/2) gives a quotient of exactly k + 1/2, so true division must
    land on the even neighbour (multiplying by a rounded 1/7 would not).
    """
    x = np.zeros((2, 32), np.float32)
    vals = [127.0, 0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 126.5, -126.5, 4.49999952]
    x[0, :len(vals)] = vals
    want0 = [127, 0, 2, 2, 4, 0, -2, -2, 126, -126, 4]
    ks = [6, 12, 14, 22, 24, 26, 28, 30, 44, 86, 88]
    x[1, 0] = 889.0
    for i, k in enumerate(ks):
        x[1, 1 + i] = 7.0 * (k + 0.5)
        x[1, 20 + i] = -7.0 * (k + 0.5)
    xq, xds = o.quantize_q8_1(x)
    assert xds[0, 0, 0] == 1.0 and xds[1, 0, 0] == 7.0
    assert list(xq[0, :len(vals)]) == want0
    assert xq[1, 0] == 127
    assert list(xq[1, 1:1 + len(ks)]) == ks
    assert list(xq[1, 20:20 + len(ks)]) == [-k for k in ks]


def pin_q8_1_invariants(o):
    """Rounding to nearest: |x - d q| <= d/2; the block max maps to +-127;
    s is the correctly rounded product d * sum(q)."""
    rng = np.random.default_rng(123)
    x = synth.activations(6, 1024, rng, outliers=True)
    x[5, 64:96] = 0.0
    xq, xds = o.quantize_q8_1(x)
    d = np.repeat(xds[..., 0].astype(np.float64), 32, axis=1)
    err = np.abs(x.astype(np.float64) - d * xq)
    assert (err <= d * 0.5 * (1 + 1e-6)).all()
    assert (np.abs(xq.astype(np.int64)) <= 127).all()
    blocks = np.abs(xq.astype(np.int64)).reshape(6, -1, 32).max(axis=2)
    nonzero = xds[..., 0] != 0
    assert (blocks[nonzero] == 127).all() and (blocks[~nonzero] == 0).all()
    qsum = xq.astype(np.int64).reshape(6, -1, 32).sum(axis=2)
    exact = xds[..., 0].astype(np.float64) * qsum
    s = xds[..., 1].astype(np.float64)
    ulp = np.spacing(np.abs(xds[..., 1])).astype(np.float64)
    assert (np.abs(s - exact) <= 0.5 * ulp).all()
    amax = np.abs(x.reshape(6, -1, 32)).max(axis=2)
    assert np.array_equal(xds[..., 0], amax / np.float32(127.0))


# ------------------------------------------------------------------- Q4_K ---

def pin_f16_fields(o):
    """d is read as IEEE binary16: 1.0, the smallest subnormal, the largest
    finite value and a negative number come through exactly."""
    for raw, val in [(0x3C00, 1.0), (0x0001, 2.0 ** -24), (0x7BFF, 65504.0), (0xC000, -2.0),
                     (0x3555, 0.333251953125)]:
        blk = _q4k_block(qs=np.full(128, 0x11, np.uint8))
        blk[0:2] = np.array([raw], "<u2").view(np.uint8)
        w = o.dequantize(Q4_K, blk.reshape(1, 144), 1, 256)
        assert (w == val).all(), (hex(raw), w[0, :4])


def pin_q4k_scale_min_roundtrip(o):
    """Pack random 6-bit (scale, min) codes; the decode gives them back."""
    rng = np.random.default_rng(7)
    for _ in range(64):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        b0 = _q4k_block(d=1.0, dmin=1.0, sc=sc, m=m, qs=np.zeros(128, np.uint8))
        b1 = _q4k_block(d=1.0, dmin=1.0, sc=sc, m=m, qs=np.full(128, 0x11, np.uint8))
        W = np.stack([b0, b1])
        w = o.dequantize(Q4_K, W, 2, 256)
        got_m = -w[0].reshape(8, 32)
        got_sc = (w[1] - w[0]).reshape(8, 32)
        assert (got_m == m[:, None]).all() and (got_sc == sc[:, None]).all()


def pin_q4k_nibble_placement(o):
    """Byte i of nibble pair p: low nibble -> element i of sub-block 2p,
    high nibble -> element i of sub-block 2p+1."""
    qs = np.zeros(128, np.uint8)
    want = np.zeros(256, np.int64)
    for p in range(4):
        for i in range(32):
            lo, hi = (i + p) % 16, (15 - i - 2 * p) % 16
            qs[32 * p + i] = lo | (hi << 4)
            want[64 * p + i] = lo
            want[64 * p + 32 + i] = hi
    blk = _q4k_block(qs=qs)
    w = o.dequantize(Q4_K, blk.reshape(1, 144), 1, 256)
    assert (w[0] == want).all()


def pin_q4k_integer_matmul(o):
    """d=1, dmin=0, sc=1, m=0 makes W the raw nibbles; integer activations whose
    block maximum is 127 quantize to themselves (d = 1).  The output is then an
    exact integer matmul."""
    rng = np.random.default_rng(11)
    od, K, nt = 6, 512, 3
    blocks = []
    for r in range(od * K // 256):
        blocks.append(_q4k_block(qs=rng.integers(0, 256, 128, dtype=np.uint8)))
    W = np.stack(blocks).reshape(od, -1)
    nib = brute.q4k_nibbles(W.reshape(od, K // 256, 144)).reshape(od, K)
    x = rng.integers(-127, 128, size=(nt, K)).astype(np.float32)
    x.reshape(nt, -1, 32)[:, :, 0] = 127.0
    want = x.astype(np.int64) @ nib.T
    out = o.matmul(Q4_K, W, x, od)
    assert np.array_equal(out.astype(np.int64), want)
    xq, _ = o.quantize_q8_1(x)
    dots = o.block_dots(Q4_K, W, xq, od)
    want_dots = np.einsum("tjk,rjk->trj", x.astype(np.int64).reshape(nt, -1, 32),
                          nib.reshape(od, -1, 32))
    assert np.array_equal(dots, want_dots)


def pin_q4k_min_term(o):
    """All-zero nibbles leave only the min term: out = -sum_j dmin*m_j*s_j."""
    rng = np.random.default_rng(5)
    m = rng.integers(0, 64, 8)
    blk = _q4k_block(d=0.5, dmin=0.25, m=m, qs=np.zeros(128, np.uint8))
    x = rng.standard_normal((2, 256)).astype(np.float32)
    xq, xds = o.quantize_q8_1(x)
    out = o.matmul_q8_1(Q4_K, blk.reshape(1, 144), xq, xds, 1)
    want = -(0.25 * m[None, :] * xds[:, :, 1].astype(np.float64)).sum(axis=1)
    assert np.allclose(out[:, 0], want, rtol=1e-6, atol=0)


def _onehot_probe(o, qtype, seed):
    od, K = 8, 512
    W = synth.weights(qtype, od, K, np.random.default_rng(seed))
    x = np.eye(K, dtype=np.float32)
    out = o.matmul(qtype, W, x, od)                    # [K tokens][od]
    dx = np.float64(np.float32(1.0) / np.float32(127.0))
    want = brute.dequantize(qtype, W, od, K).T * (127 * dx)
    scale = np.abs(want).max()
    assert np.allclose(out, want, rtol=1e-6, atol=1e-6 * scale)


def pin_q4k_onehot_columns(o):
    """x = e_k reads back column k of the dequantized matrix, for every k."""
    _onehot_probe(o, Q4_K, 21)


def pin_q6k_onehot_columns(o):
    _onehot_probe(o, Q6_K, 22)


# ------------------------------------------------------------------- Q6_K ---

def pin_q6k_extremes(o):
    """q = 0 gives -32*d*sc, q = 63 gives +31*d*sc, with signed int8 scales."""
    scales = np.array([1, -1, 2, -2, 127, -128, 0, 5, 1, 1, 1, 1, 1, 1, 1, -3], np.int8)
    lo = _q6k_block(d=0.5, scales=scales, ql=0, qh=0)
    hi = _q6k_block(d=0.5, scales=scales, ql=0xFF, qh=0xFF)
    w = o.dequantize(Q6_K, np.stack([lo, hi]), 2, 256)
    s = np.repeat(scales.astype(np.float64), 16)
    assert (w[0] == -32 * 0.5 * s).all()
    assert (w[1] == 31 * 0.5 * s).all()


def pin_q6k_integer_matmul(o):
    """d=1, scales=1 makes W = q - 32; the output is an exact integer matmul and
    the per-16 block dots are exact."""
    rng = np.random.default_rng(13)
    od, K, nt = 5, 512, 3
    blocks = [_q6k_block(ql=rng.integers(0, 256, 128, dtype=np.uint8),
                         qh=rng.integers(0, 256, 64, dtype=np.uint8))
              for _ in range(od * K // 256)]
    W = np.stack(blocks).reshape(od, -1)
    q = brute.q6k_values(W.reshape(od, K // 256, 210)).reshape(od, K) - 32
    x = rng.integers(-127, 128, size=(nt, K)).astype(np.float32)
    x.reshape(nt, -1, 32)[:, :, 3] = -127.0
    out = o.matmul(Q6_K, W, x, od)
    assert np.array_equal(out.astype(np.int64), x.astype(np.int64) @ q.T)
    xq, _ = o.quantize_q8_1(x)
    dots = o.block_dots(Q6_K, W, xq, od)
    want = np.einsum("tgk,rgk->trg", x.astype(np.int64).reshape(nt, -1, 16),
                     q.reshape(od, -1, 16))
    assert np.array_equal(dots, want)


# ----------------------------------------------------- whole-method checks ---

def _random_case(qtype, seed, od=48, K=768, nt=5):
    rng = np.random.default_rng(seed)
    return synth.weights(qtype, od, K, rng), synth.activations(nt, K, rng, outliers=True), od


def pin_matmul_vs_dense_f64(o):
    """Dequantize-then-dense-f64 matmul over the same q8_1 activations agrees
    with the oracle's integer-dot + rescale form (only s's single f32 rounding
    differs)."""
    for qtype, seed in [(Q4_K, 1), (Q6_K, 2), (Q4_K, 3)]:
        W, x, od = _random_case(qtype, seed)
        xq, xds = o.quantize_q8_1(x)
        out = o.matmul_q8_1(qtype, W, xq, xds, od)
        want = brute.matmul_from_q8_1(qtype, W, xq, xds, od)
        norm = np.linalg.norm(want, axis=1, keepdims=True)
        assert (np.abs(out - want) <= 1e-6 * norm).all()
        d_all = brute.dequantize(qtype, W, od, x.shape[1])
        assert np.array_equal(o.dequantize(qtype, W, od, x.shape[1]), d_all)


def pin_block_dots_vs_dense(o):
    """Block dots equal the integer dots of the decoded codes."""
    for qtype, seed in [(Q4_K, 4), (Q6_K, 5)]:
        W, x, od = _random_case(qtype, seed, od=16, K=512, nt=3)
        xq, _ = o.quantize_q8_1(x)
        dots = o.block_dots(qtype, W, xq, od)
        nsb = 512 // 256
        if qtype == Q4_K:
            codes = brute.q4k_nibbles(W.reshape(od, nsb, 144)).reshape(od, -1, 32)
            want = np.einsum("tjk,rjk->trj", xq.astype(np.int64).reshape(3, -1, 32), codes)
        else:
            codes = brute.q6k_values(W.reshape(od, nsb, 210)).reshape(od, -1, 16) - 32
            want = np.einsum("tgk,rgk->trg", xq.astype(np.int64).reshape(3, -1, 16), codes)
        assert np.array_equal(dots, want)


def pin_quantization_error_bound(o):
    """Against the raw f32 activations the result is off by at most the
    activation rounding: sum_k |w| * d_x / 2."""
    for qtype, seed in [(Q4_K, 8), (Q6_K, 9)]:
        W, x, od = _random_case(qtype, seed)
        out = o.matmul(qtype, W, x, od).astype(np.float64)
        wd = brute.dequantize(qtype, W, od, x.shape[1])
        exact = x.astype(np.float64) @ wd.T
        _, xds = o.quantize_q8_1(x)
        dx = np.repeat(xds[..., 0].astype(np.float64), 32, axis=1)
        bound = (dx / 2) @ np.abs(wd).T
        # plus the final f32 rounding of each output
        assert (np.abs(out - exact) <= bound * (1 + 1e-6) + np.abs(exact) * 2.0 ** -23 + 1e-9).all()


def pin_threads_do_not_change_results(o):
    W, x, od = _random_case(Q4_K, 10, od=37)
    xq, xds = o.quantize_q8_1(x)
    a = o.matmul_q8_1(Q4_K, W, xq, xds, od, nthreads=1)
    b = o.matmul_q8_1(Q4_K, W, xq, xds, od, nthreads=5)
    assert np.array_equal(a, b)


def pin_mac_count_golden(o):
    """The page's IMMA count for the nt=512, od=K=3584 GEMM is one m16n8k32 per
    4096 MACs: it pins the MAC count used for TOPS."""
    g = read_golden("page_numbers.txt")
    c = synth.Case(Q4_K, 3584, 3584, 512)
    assert c.macs // (16 * 8 * 32) == g["qproj_nt512_3584_imma_count"]
    assert c.macs % (16 * 8 * 32) == 0
    assert o.weight_bytes(Q4_K, 3584, 3584) == c.weight_bytes


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
