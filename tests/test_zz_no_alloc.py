"""qmm_gemm_builtin_workspace: the tensor-core GEMM on the library's fixed
built-in scratch array instead of a caller workspace.

Called through the C ABI (the binding's same-named function) and compared with
qmm_gemm on a workspace of the caller's, within the parity tolerance of the
other GPU tests (1e-4 of each output row's L2 norm), on two calls in a row per
shape.  The file sorts last so that it runs both alone and after every other
test file in one session.
"""
import ctypes

import numpy as np
import pytest

import quantized_weight_matmul_gb300 as qmm
from gpu_helpers import REL_TOL, dev
from quantized_weight_matmul_gb300 import synth

Q4_K, Q6_K = qmm.Q4_K, qmm.Q6_K


def test_size_limit_is_refused_before_any_device_work():
    """A problem whose scratch exceeds the built-in array is refused with
    QMM_EWORKSPACE (no GPU needed: the check comes before any CUDA call)."""
    buf = ctypes.create_string_buffer(4096 + 16)
    p = (ctypes.addressof(buf) + 15) & ~15
    big = (Q4_K, 4096, 14336, 512)
    assert qmm.qmm_gemm_workspace_bytes(*big) > qmm.QMM_BUILTIN_WORKSPACE_BYTES
    assert qmm.qmm_gemm_builtin_workspace(Q4_K, p, p, p, p, 4096, 14336, 512, 0) == qmm.QMM_EWORKSPACE
    # nt = 832 at K = 4096 fills the array exactly; one token more does not fit
    assert qmm.qmm_gemm_workspace_bytes(Q4_K, 4096, 4096, 832) == qmm.QMM_BUILTIN_WORKSPACE_BYTES
    assert qmm.qmm_gemm_builtin_workspace(Q4_K, p, p, p, p, 4096, 4096, 833, 0) == qmm.QMM_EWORKSPACE
    assert qmm.qmm_gemm_builtin_workspace(Q4_K, p, p, p, p, 4096, 300, 8, 0) == qmm.QMM_EINVAL_SHAPE
    # refusals of a misaligned pointer also come before any device work
    assert qmm.qmm_gemm_builtin_workspace(Q6_K, p, p + 2, p, p, 4096, 512, 8, 0) == qmm.QMM_EALIGN
    assert qmm.qmm_gemm_builtin_workspace(Q4_K, 0, p, p, p, 4096, 4096, 8, 0) == qmm.QMM_ENULL
    assert qmm.qmm_gemm_builtin_workspace(9, p, p, p, p, 4096, 4096, 8, 0) == qmm.QMM_EINVAL_QTYPE


def _rel_err(a, ref):
    norm = np.linalg.norm(ref.astype(np.float64), axis=1)
    err = np.abs(a.astype(np.float64) - ref.astype(np.float64)).max(axis=1)
    return float((err / np.maximum(norm, 1e-30)).max())


@pytest.mark.gpu
def test_builtin_workspace_matches_qmm_gemm():
    torch = pytest.importorskip("torch")
    # the largest shape first, so the later, smaller ones run on scratch that
    # holds another layout's leftovers
    shapes = [(Q4_K, 4096, 4096, 832), (Q4_K, 300, 512, 70), (Q6_K, 4096, 4096, 64), (Q4_K, 1000, 2048, 9)]
    assert qmm.qmm_gemm_workspace_bytes(*shapes[0]) == qmm.QMM_BUILTIN_WORKSPACE_BYTES
    st = torch.cuda.current_stream().cuda_stream
    for qtype, od, K, nt in shapes:
        c = synth.Case(qtype, od, K, nt, True)
        W, x = (dev(a, torch) for a in c.generate())
        xq, xds = qmm.quantize_q8_1(x)
        ref = qmm.gemm(qtype, W, xq, xds, od).cpu().numpy()
        for call in range(2):
            out = torch.full((nt, od), float("nan"), dtype=torch.float32, device=x.device)
            rc = qmm.qmm_gemm_builtin_workspace(qtype, W.data_ptr(), xq.data_ptr(), xds.data_ptr(),
                                                out.data_ptr(), od, K, nt, st)
            assert rc == qmm.QMM_OK, qmm.qmm_strerror(rc)
            got = out.cpu().numpy()
            assert np.isfinite(got).all(), (c.name, call)
            assert _rel_err(got, ref) <= REL_TOL, (c.name, call, _rel_err(got, ref))
    assert qmm.qmm_sync_status(st) == qmm.QMM_OK
