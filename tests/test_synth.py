"""The seeded input generator (quantized_weight_matmul_gb300/synth.py): the
recipe every parity test, the oracle tests and the benchmark draw from.

Pins the recipe itself -- field ranges, byte uniformity, the exact outlier
count, the draw order and the workload families -- on the CPU, so that a
change to the generator cannot pass unnoticed through tests that only
compare two consumers of the same inputs.
"""
import numpy as np
import pytest

from quantized_weight_matmul_gb300 import synth
from quantized_weight_matmul_gb300.synth import Q4_K, Q6_K

F16_LO, F16_HI = float(np.float16(0.001)), float(np.float16(0.02))


def _f16_field(blocks, lo):
    return blocks[..., lo:lo + 2].copy().view("<f2")[..., 0].astype(np.float64)


def test_seeded_and_deterministic():
    a = synth.Case(Q4_K, 64, 1024, 3, outliers=True, seed=5).generate()
    b = synth.Case(Q4_K, 64, 1024, 3, outliers=True, seed=5).generate()
    c = synth.Case(Q4_K, 64, 1024, 3, outliers=True, seed=6).generate()
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert not np.array_equal(a[0], c[0]) and not np.array_equal(a[1], c[1])


def test_weights_drawn_before_activations():
    """Case.generate draws the weight bytes first, then x, from one stream."""
    case = synth.Case(Q6_K, 48, 512, 4, outliers=True, seed=11)
    W, x = case.generate()
    rng = np.random.default_rng(11)
    W2 = synth.weights(Q6_K, 48, 512, rng)
    x2 = synth.activations(4, 512, rng, outliers=True)
    assert np.array_equal(W, W2) and np.array_equal(x, x2)


@pytest.mark.parametrize("qtype", [Q4_K, Q6_K])
def test_shapes_and_dtypes(qtype):
    case = synth.Case(qtype, 40, 768, 5)
    W, x = case.generate()
    assert W.dtype == np.uint8 and W.shape == (40, 3 * synth.BLOCK_BYTES[qtype])
    assert W.nbytes == case.weight_bytes
    assert x.dtype == np.float32 and x.shape == (5, 768)
    assert case.macs == 5 * 40 * 768
    with pytest.raises(ValueError):
        synth.weights(qtype, 4, 300, np.random.default_rng(0))


def test_q4k_fields():
    """d and dmin are f16(U(0.001, 0.02)); every other byte is uniform, so
    the 6-bit scales and mins span [0, 63] and the nibbles [0, 15]."""
    W = synth.Case(Q4_K, 64, 1024, 1, seed=1).generate()[0].reshape(64, 4, 144)
    for lo in (0, 2):
        v = _f16_field(W, lo)
        assert v.min() >= F16_LO and v.max() <= F16_HI
        assert v.max() - v.min() > 0.015  # spread over the interval
    rest = W[:, :, 4:].astype(np.int64)
    assert abs(rest.mean() - 127.5) < 2.0
    assert np.unique(rest).size == 256
    nib = np.concatenate([(rest[:, :, 12:] & 15).ravel(), (rest[:, :, 12:] >> 4).ravel()])
    assert np.bincount(nib, minlength=16).min() > 0.8 * nib.size / 16


def test_q6k_fields():
    """d is f16(U(0.001, 0.02)) at bytes 208-209; ql, qh and the int8 scales
    are uniform bytes."""
    W = synth.Case(Q6_K, 64, 1024, 1, seed=2).generate()[0].reshape(64, 4, 210)
    d = _f16_field(W, 208)
    assert d.min() >= F16_LO and d.max() <= F16_HI
    body = W[:, :, :208].astype(np.int64)
    assert abs(body.mean() - 127.5) < 2.0
    sc = W[:, :, 192:208].view(np.int8).astype(np.int64)
    assert sc.min() < -100 and sc.max() > 100


def test_activations_standard_normal():
    x = synth.activations(1, 1 << 16, np.random.default_rng(3))
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02


@pytest.mark.parametrize("nt,K", [(1, 4096), (3, 1024), (5, 512), (8, 512), (1, 256)])
def test_outliers_exact_count(nt, K):
    """With outliers, exactly round(0.001 * nt * K) distinct entries of the
    same N(0, 1) draw are multiplied by 20; all others are unchanged."""
    plain = synth.activations(nt, K, np.random.default_rng(9), outliers=False)
    out = synth.activations(nt, K, np.random.default_rng(9), outliers=True)
    scaled = out != plain
    assert int(scaled.sum()) == int(round(0.001 * nt * K))
    assert np.array_equal(out[scaled], plain[scaled] * np.float32(20.0))


def test_workload_families():
    """The five families and their shapes, nt values and outlier settings."""
    want = {
        "tiny_q4k": {(Q4_K, 256, 512, nt, False) for nt in (1, 8)},
        "decode_gemv_q4k": {(Q4_K, od, 4096, 1, True) for od in (4096, 11008)},
        "mmvq_q4k": {(Q4_K, od, K, nt, False) for od, K in ((14336, 4096), (4096, 14336)) for nt in (2, 4, 8)},
        "prefill_gemm_q4k": {(Q4_K, od, K, nt, True) for od, K in ((4096, 4096), (14336, 4096), (4096, 14336))
                             for nt in (128, 512, 2048)},
        "skinny_q6k": {(Q6_K, od, 4096, nt, False) for od in (4096, 32000) for nt in (32, 64, 80, 256)},
    }
    assert set(synth.WORKLOADS) == set(want)
    for name, w in synth.WORKLOADS.items():
        got = {(c.qtype, c.od, c.K, c.nt, c.outliers) for c in w.cases}
        assert got == want[name], name
        assert len(w.cases) == len(got)
