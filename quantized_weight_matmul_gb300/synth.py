"""Seeded synthetic inputs: raw GGUF K-quant weight bytes and f32 activations.

This module only draws random numbers; it holds none of the matmul's
arithmetic (no decode, no quantization, no dot products).  The CUDA tests, the
CPU oracle tests and the benchmark all take their inputs from here.

Recipe (numpy ``default_rng(seed)``, PCG64; the weight bytes are drawn first,
then the activations):

* Q4_K super-block (144 B): all 144 bytes uniform in [0, 255] (so the 6-bit
  scales and mins are uniform in [0, 63] and the nibbles uniform in [0, 15]);
  then ``d`` and ``dmin`` are overwritten with f16(U(0.001, 0.02)) -- first
  every ``d`` of the matrix, then every ``dmin``.
* Q6_K super-block (210 B): all bytes uniform (so q is uniform in [0, 63] and
  the int8 scales uniform in [-128, 127]); then ``d`` = f16(U(0.001, 0.02)).
* Activations: f32 N(0, 1); with outliers, exactly round(0.001 * nt * K)
  distinct positions, chosen uniformly, are multiplied by 20.

The block layouts are the ones described in "llama.cpp MMQ" sec. 4 and the
mojo-dllm "The quantized GEMM" page (section "The GPU path").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

Q4_K = 12
Q6_K = 14
BLOCK_BYTES = {Q4_K: 144, Q6_K: 210}
QTYPE_NAMES = {Q4_K: "Q4_K", Q6_K: "Q6_K"}


def _f16_bytes(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a.astype("<f2")).view(np.uint8).reshape(*a.shape, 2)


def weights(qtype: int, od: int, K: int, rng: np.random.Generator) -> np.ndarray:
    """Random weight matrix [od][K] as raw super-block bytes, shape (od, K/256*bytes)."""
    if K % 256:
        raise ValueError("K must be a multiple of 256")
    nsb = K // 256
    bb = BLOCK_BYTES[qtype]
    raw = rng.integers(0, 256, size=(od, nsb, bb), dtype=np.uint8)
    if qtype == Q4_K:
        d = rng.uniform(0.001, 0.02, size=(od, nsb))
        dmin = rng.uniform(0.001, 0.02, size=(od, nsb))
        raw[:, :, 0:2] = _f16_bytes(d)
        raw[:, :, 2:4] = _f16_bytes(dmin)
    elif qtype == Q6_K:
        d = rng.uniform(0.001, 0.02, size=(od, nsb))
        raw[:, :, 208:210] = _f16_bytes(d)
    else:
        raise ValueError(f"unknown qtype {qtype}")
    return raw.reshape(od, nsb * bb)


def activations(nt: int, K: int, rng: np.random.Generator, outliers: bool = False) -> np.ndarray:
    """f32 N(0,1) activations [nt][K]; optionally 0.1% of entries scaled by 20."""
    x = rng.standard_normal(size=(nt, K), dtype=np.float32)
    if outliers and nt * K > 0:
        n = int(round(0.001 * nt * K))
        if n:
            idx = rng.choice(nt * K, size=n, replace=False)
            x.reshape(-1)[idx] *= np.float32(20.0)
    return x


@dataclass(frozen=True)
class Case:
    """One matmul problem: out[nt][od] = W[od][K] . x[nt][K]^T."""
    qtype: int
    od: int
    K: int
    nt: int
    outliers: bool = False
    seed: int = 0

    @property
    def name(self) -> str:
        o = "+outliers" if self.outliers else ""
        return f"{QTYPE_NAMES[self.qtype]}_od{self.od}_K{self.K}_nt{self.nt}{o}"

    @property
    def weight_bytes(self) -> int:
        return self.od * (self.K // 256) * BLOCK_BYTES[self.qtype]

    @property
    def macs(self) -> int:
        return self.nt * self.od * self.K

    def generate(self):
        """(W bytes [od][rowbytes] uint8, x [nt][K] f32), weights drawn first."""
        rng = np.random.default_rng(self.seed)
        W = weights(self.qtype, self.od, self.K, rng)
        x = activations(self.nt, self.K, rng, self.outliers)
        return W, x


@dataclass(frozen=True)
class Workload:
    name: str
    description: str
    cases: tuple = field(default_factory=tuple)


def _cases(qtype, shapes, nts, outliers):
    return tuple(Case(qtype, od, K, nt, outliers) for (od, K) in shapes for nt in nts)


# The five workload families the benchmark and the parity tests use
# (Llama-7B / LLaDA-8B shaped projections; sizes as named).
WORKLOADS = {
    "tiny_q4k": Workload(
        "tiny_q4k", "Q4_K od=256 K=512, nt in {1, 8}",
        _cases(Q4_K, [(256, 512)], [1, 8], False)),
    "decode_gemv_q4k": Workload(
        "decode_gemv_q4k", "Q4_K decode GEMV nt=1: 4096x4096 and 11008x4096, x with 0.1% x20 outliers",
        _cases(Q4_K, [(4096, 4096), (11008, 4096)], [1], True)),
    "mmvq_q4k": Workload(
        "mmvq_q4k", "Q4_K small-batch MMVQ nt in {2,4,8}: 14336x4096 and 4096x14336",
        _cases(Q4_K, [(14336, 4096), (4096, 14336)], [2, 4, 8], False)),
    "prefill_gemm_q4k": Workload(
        "prefill_gemm_q4k",
        "Q4_K prefill GEMM nt=512 (+128, 2048): 4096x4096, 14336x4096, 4096x14336, x with outliers",
        _cases(Q4_K, [(4096, 4096), (14336, 4096), (4096, 14336)], [512, 128, 2048], True)),
    "skinny_q6k": Workload(
        "skinny_q6k", "Q6_K skinny GEMM nt in {32,64,80,256}: 4096x4096 and LM head 32000x4096",
        _cases(Q6_K, [(4096, 4096), (32000, 4096)], [32, 64, 80, 256], False)),
}
