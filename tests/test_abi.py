"""Host-side checks of the C ABI: the library loads, exports every function the
header declares, and its size helpers / argument checks behave (no GPU work)."""
import ctypes

import pytest

import quantized_weight_matmul_gb300 as qmm


@pytest.fixture(scope="module")
def lib():
    return qmm.load()


def test_exports_every_header_function(lib):
    names = qmm.header_functions()
    assert len(names) >= 13
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the Python binding carries the same names
    assert all(hasattr(qmm, n) for n in names)


def test_weight_and_activation_sizes():
    assert qmm.qmm_weight_bytes(qmm.Q4_K, 4096, 4096) == 9437184
    assert qmm.qmm_weight_bytes(qmm.Q4_K, 11008, 4096) == 25362432
    assert qmm.qmm_weight_bytes(qmm.Q4_K, 14336, 4096) == 33030144
    assert qmm.qmm_weight_bytes(qmm.Q6_K, 4096, 4096) == 13762560
    assert qmm.qmm_weight_bytes(qmm.Q6_K, 32000, 4096) == 107520000
    assert qmm.qmm_weight_bytes(qmm.Q4_K, 16, 300) == 0
    assert qmm.qmm_weight_bytes(7, 16, 256) == 0
    assert qmm.qmm_xq_bytes(3, 512) == 1536
    assert qmm.qmm_q8_1_bytes(3, 512) == 1536 and qmm.qmm_q8_1_bytes(-1, 512) == 0
    assert qmm.qmm_xds_bytes(3, 512) == 3 * 16 * 8
    assert qmm.qmm_gemv_max_nt() == 16
    assert qmm.qmm_matmul_workspace_bytes(qmm.Q4_K, 4096, 4096, 8) == 0
    ws = qmm.qmm_gemm_workspace_bytes(qmm.Q4_K, 4096, 4096, 512)
    assert ws >= 512 * 4096 * 2 + 4096 // 32 * 512 * 8
    assert qmm.qmm_matmul_workspace_bytes(qmm.Q4_K, 4096, 4096, 512) == ws
    assert qmm.qmm_gemm_workspace_bytes(qmm.Q4_K, 4096, 4000, 512) == 0


def test_argument_checks_need_no_device():
    """Bad arguments are refused before any CUDA call."""
    buf = ctypes.create_string_buffer(4096 + 16)
    p = (ctypes.addressof(buf) + 15) & ~15
    assert qmm.qmm_gemv(5, p, p, p, p, 256, 256, 1, 0) == qmm.QMM_EINVAL_QTYPE
    assert qmm.qmm_gemv(qmm.Q4_K, 0, p, p, p, 256, 256, 1, 0) == qmm.QMM_ENULL
    assert qmm.qmm_gemv(qmm.Q4_K, p, p, p, p, 256, 300, 1, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_gemv(qmm.Q4_K, p, p, p, p, 256, 256, 17, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_gemv(qmm.Q4_K, p, p, p, p, 0, 256, 1, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_gemv(qmm.Q6_K, p, p, p, p, 256, 1000, 1, 0) == qmm.QMM_EINVAL_SHAPE  # K % 256
    assert qmm.qmm_gemv(qmm.Q4_K, p + 1, p, p, p, 256, 256, 1, 0) == qmm.QMM_EALIGN
    assert qmm.qmm_quantize_q8_1(p, 1, 48, p, p, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_gemm(qmm.Q4_K, p, p, p, p, 256, 256, 0, p, 4096, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_debug_inject_stall(1, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_debug_inject_stall(0, 0) == qmm.QMM_OK


def test_every_entry_point_refuses_bad_arguments_first():
    """Each compute entry point checks type, pointers, shape, alignment and
    flags before it touches the device, so these refusals need no GPU."""
    buf = ctypes.create_string_buffer(4096 + 16)
    p = (ctypes.addressof(buf) + 15) & ~15
    Q4, Q6 = qmm.Q4_K, qmm.Q6_K
    # quantizer: pointers, shape (nt >= 1, K a multiple of 32), alignment
    assert qmm.qmm_quantize_q8_1(0, 1, 64, p, p, 0) == qmm.QMM_ENULL
    assert qmm.qmm_quantize_q8_1(p, 0, 64, p, p, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_quantize_q8_1(p + 4, 1, 64, p, p, 0) == qmm.QMM_EALIGN
    assert qmm.qmm_quantize_q8_1(p, 1, 64, p, p + 8, 0) == qmm.QMM_EALIGN
    # the whole path: type, pointers, shape, alignment, unknown flag bits
    args = [p, p, p, p, p, 256, 256, 1, 0, 0]
    assert qmm.qmm_matmul(3, *args, 0, 0) == qmm.QMM_EINVAL_QTYPE
    assert qmm.qmm_matmul(Q4, p, 0, p, p, p, 256, 256, 1, 0, 0, 0, 0) == qmm.QMM_ENULL
    assert qmm.qmm_matmul(Q6, p, p, p, p, p, 256, 300, 1, 0, 0, 0, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_matmul(Q4, p, p, p, p, p, 256, 256, 0, 0, 0, 0, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_matmul(Q4, p, p, p, p, p + 8, 256, 256, 1, 0, 0, 0, 0) == qmm.QMM_EALIGN
    assert qmm.qmm_matmul(Q4, *args, 2, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_matmul(Q4, *args, 0xFFFFFFFE, 0) == qmm.QMM_EINVAL_SHAPE
    # GEMM on caller-quantized input
    assert qmm.qmm_gemm(9, p, p, p, p, 256, 256, 32, p, 4096, 0) == qmm.QMM_EINVAL_QTYPE
    assert qmm.qmm_gemm(Q4, p, p, p, 0, 256, 256, 32, p, 4096, 0) == qmm.QMM_ENULL
    assert qmm.qmm_gemm(Q6, p, p, p + 4, p, 256, 256, 32, p, 4096, 0) == qmm.QMM_EALIGN
    # block-dot test hook
    assert qmm.qmm_debug_block_dots(9, p, p, p, 256, 256, 1, p, 0, 0, 0, 0) == qmm.QMM_EINVAL_QTYPE
    assert qmm.qmm_debug_block_dots(Q4, p, p, p, 256, 256, 1, 0, 0, 0, 0, 0) == qmm.QMM_ENULL
    assert qmm.qmm_debug_block_dots(Q4, p, p, p, 256, 512 + 32, 1, p, 0, 0, 0, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_debug_block_dots(Q6, p + 2, p, p, 256, 256, 1, p, 0, 0, 0, 0) == qmm.QMM_EALIGN


def test_valid_call_without_a_gpu_fails_loudly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    buf = ctypes.create_string_buffer(4096 + 16)
    p = (ctypes.addressof(buf) + 15) & ~15
    assert qmm.qmm_gemv(qmm.Q4_K, p, p, p, p, 256, 256, 1, 0) == qmm.QMM_EDEVICE
    assert qmm.qmm_matmul(qmm.Q4_K, p, p, p, p, p, 256, 256, 1, 0, 0, qmm.QMM_FLAG_STATIC_WEIGHTS, 0) == \
        qmm.QMM_EDEVICE
    assert qmm.qmm_quantize_q8_1(p, 1, 64, p, p, 0) == qmm.QMM_EDEVICE


def test_strerror_covers_codes():
    for code in range(0, -10, -1):
        assert qmm.qmm_strerror(code) != "unknown status"
    assert qmm.qmm_strerror(-99) == "unknown status"


def test_matmul_route_query():
    """qmm_matmul_path names the route the dispatch takes: the fused
    quantize + dp4a MMVQ kernel for few tokens (nt = 1, and Q4_K up to 4)
    while the activations leave room for its weight ring, quantize + the
    warp-MMA MMVQ from 5 tokens (Q4_K) or 2 (Q6_K) up to 16 where it fits,
    quantize + the dp4a MMVQ for the other nt <= 8, the tensor-core GEMM
    beyond; workspace is needed exactly on the GEMM route."""
    Q4, Q6 = qmm.Q4_K, qmm.Q6_K
    F, V, G = qmm.QMM_PATH_FUSED_MMVQ, qmm.QMM_PATH_MMVQ, qmm.QMM_PATH_MMQ
    cases = [((Q4, 4096, 4096, 1), F), ((Q4, 11008, 4096, 1), F), ((Q4, 256, 512, 4), F),
             ((Q4, 4096, 4096, 4), F), ((Q4, 4096, 4096, 5), V), ((Q4, 4096, 4096, 8), V),
             ((Q4, 4096, 14336, 2), F), ((Q4, 4096, 14336, 4), V), ((Q4, 4096, 14336, 8), V),
             ((Q4, 14336, 16384, 3), V), ((Q4, 4096, 4096, 9), V), ((Q4, 4096, 4096, 16), V),
             ((Q4, 4096, 4096, 17), G), ((Q4, 4096, 4096, 512), G), ((Q6, 4096, 4096, 1), F),
             ((Q6, 32000, 4096, 2), V), ((Q6, 4096, 4096, 8), V), ((Q6, 4096, 4096, 9), V),
             ((Q6, 4096, 4096, 17), G), ((Q6, 32000, 4096, 80), G),
             # Q6_K rows whose pitch is not a multiple of 16 bytes (K % 2048 != 0)
             # are staged row by row, on every route
             ((Q6, 4096, 768, 32), G), ((Q6, 4096, 11008, 1), F), ((Q6, 4096, 2304, 8), V),
             ((Q6, 300, 256, 64), G), ((Q6, 4096, 11008, 2), V)]
    for args, path in cases:
        assert qmm.qmm_matmul_path(*args) == path, args
        assert (qmm.qmm_matmul_workspace_bytes(*args) > 0) == (path == qmm.QMM_PATH_MMQ), args
    assert qmm.qmm_matmul_path(Q4, 4096, 300, 1) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_matmul_path(Q4, 4096, 4096, 0) == qmm.QMM_EINVAL_SHAPE
    assert qmm.qmm_matmul_path(3, 4096, 4096, 1) == qmm.QMM_EINVAL_QTYPE
