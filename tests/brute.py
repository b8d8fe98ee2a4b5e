"""Brute-force f64 reference pieces, written separately from the C oracle.

These are whole-array numpy restatements of the block formats, used only to
pin the oracle on small inputs (dequantize-then-dense-f64-matmul).  They read
the formats from the same sources as the oracle but share none of its code:

* Q4_K ("llama.cpp MMQ" sec. 4 and sec. 6; mojo-dllm "The quantized GEMM",
  "The GPU path"): bytes 0-1 d, 2-3 dmin (f16), 4-15 the packed 6-bit
  (scale, min) codes, 16-143 the nibbles; byte i of nibble pair p holds element
  i of sub-block 2p (low nibble) and element i of sub-block 2p+1 (high nibble);
  weight = d*sc*nibble - dmin*m.
* Q6_K: ql (128 B), qh (64 B), 16 signed int8 scales, f16 d; weight =
  d*scale[e/16]*(q-32), with the public GGUF bit placement of ql/qh.
"""
from __future__ import annotations

import numpy as np

Q4_K = 12
Q6_K = 14


def f16_field(blocks: np.ndarray, off: int) -> np.ndarray:
    """f16 little-endian field at byte offset `off` of each block, as f64."""
    lo = blocks[..., off].astype(np.uint16)
    hi = blocks[..., off + 1].astype(np.uint16)
    return (lo | (hi << 8)).view(np.float16).astype(np.float64)


def q4k_codes(blocks: np.ndarray):
    """(sc, m) arrays [..., 8] from the 12 packed scale bytes."""
    s = blocks[..., 4:16].astype(np.int64)
    first, second, third = s[..., 0:4], s[..., 4:8], s[..., 8:12]
    sc = np.concatenate([first & 63, (third & 15) | ((first >> 6) << 4)], axis=-1)
    m = np.concatenate([second & 63, (third >> 4) | ((second >> 6) << 4)], axis=-1)
    return sc, m


def q4k_nibbles(blocks: np.ndarray) -> np.ndarray:
    """Nibbles [..., 256] in element order."""
    qs = blocks[..., 16:144].reshape(*blocks.shape[:-1], 4, 32)
    both = np.stack([qs & 15, qs >> 4], axis=-2)  # [..., pair, half(lo/hi), 32]
    return both.reshape(*blocks.shape[:-1], 256).astype(np.int64)


def q6k_values(blocks: np.ndarray) -> np.ndarray:
    """q in [0, 63], [..., 256] in element order (GGUF bit placement)."""
    ql = blocks[..., 0:128].astype(np.int64).reshape(*blocks.shape[:-1], 2, 64)
    qh = blocks[..., 128:192].astype(np.int64).reshape(*blocks.shape[:-1], 2, 32)
    out = np.empty((*blocks.shape[:-1], 2, 4, 32), dtype=np.int64)
    low = [ql[..., 0:32] & 15, ql[..., 32:64] & 15, ql[..., 0:32] >> 4, ql[..., 32:64] >> 4]
    for quad in range(4):
        out[..., quad, :] = low[quad] | (((qh >> (2 * quad)) & 3) << 4)
    return out.reshape(*blocks.shape[:-1], 256)


def q6k_scales(blocks: np.ndarray) -> np.ndarray:
    return blocks[..., 192:208].view(np.int8).astype(np.int64)


def dequantize(qtype: int, W: np.ndarray, od: int, K: int) -> np.ndarray:
    nsb = K // 256
    if qtype == Q4_K:
        blocks = W.reshape(od, nsb, 144)
        d, dmin = f16_field(blocks, 0), f16_field(blocks, 2)
        sc, m = q4k_codes(blocks)
        nib = q4k_nibbles(blocks).reshape(od, nsb, 8, 32)
        w = (d[..., None, None] * sc[..., None] * nib
             - dmin[..., None, None] * m[..., None])
        return w.reshape(od, K)
    blocks = W.reshape(od, nsb, 210)
    d = f16_field(blocks, 208)
    sc = q6k_scales(blocks)
    q = q6k_values(blocks).reshape(od, nsb, 16, 16)
    w = d[..., None, None] * sc[..., None] * (q - 32)
    return w.reshape(od, K)


def matmul_from_q8_1(qtype: int, W: np.ndarray, xq: np.ndarray, xds: np.ndarray, od: int):
    """f64 dense reference: W_deq . (dx * q)^T with the exact activation value dx*q."""
    nt, K = xq.shape
    wd = dequantize(qtype, W, od, K)
    dx = np.repeat(xds[..., 0].astype(np.float64), 32, axis=1)
    xv = dx * xq.astype(np.float64)
    return xv @ wd.T


def pack_q4k_codes(sc: np.ndarray, m: np.ndarray) -> np.ndarray:
    """Inverse of the 6-bit unpack: 12 bytes holding eight (sc, m) pairs.

    Scales/mins 0-3 sit in the low 6 bits of bytes 0-3 / 4-7; scales/mins 4-7
    keep their low 4 bits in the low / high nibble of bytes 8-11 and their top
    2 bits in the top 2 bits of bytes 0-3 / 4-7.
    """
    sc = np.asarray(sc, dtype=np.int64)
    m = np.asarray(m, dtype=np.int64)
    b = np.zeros(12, dtype=np.int64)
    for j in range(4):
        b[j] = (sc[j] & 63) | ((sc[j + 4] >> 4) << 6)
        b[j + 4] = (m[j] & 63) | ((m[j + 4] >> 4) << 6)
        b[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return b.astype(np.uint8)
