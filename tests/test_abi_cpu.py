"""The C ABI without a GPU: the library builds, loads and exports every symbol
include/qm.h declares, and argument errors are caught on the host before any
CUDA call (so they are testable here)."""
import os
import re

import pytest

import bit_block_quantized_qm_gb300 as qm
from bit_block_quantized_qm_gb300 import build as qm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qm_build.build()
    return qm.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "qm.h")).read()
    return set(re.findall(r"QM_API\s+[\w\s\*]+?\b(qm_\w+)\s*\(", text))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert names == set(qm.EXPORTED_SYMBOLS)
    for name in names:
        assert getattr(lib, name) is not None


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", qm.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T qm_" in line}
    assert exported == declared_symbols()


def test_version_and_status_strings(lib):
    assert qm.qm_version() >= 100
    for code in range(-9, 1):
        assert qm.qm_status_string(code) != "unknown status"
    assert qm.qm_status_string(-99) == "unknown status"


# Fake, well-aligned addresses: every check below fails before the library
# asks CUDA anything, so no address is ever dereferenced.
A_ADDR, W_ADDR, C_ADDR = 0x10000000, 0x20000000, 0x30000000


def test_shape_errors(lib):
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, C_ADDR, -1, 4, 32) == qm.QM_ERR_SHAPE
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, C_ADDR, 1, -4, 32) == qm.QM_ERR_SHAPE
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, C_ADDR, 1, 4, -32) == qm.QM_ERR_SHAPE
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, C_ADDR, 1, 4, 33) == qm.QM_ERR_SHAPE
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, C_ADDR, 1 << 40, 1 << 40, 32) == qm.QM_ERR_SHAPE
    assert qm.qm_dequant_q4_0_ptr(W_ADDR, -1, C_ADDR) == qm.QM_ERR_SHAPE
    assert qm.qm_dequant_q4_0_ptr(W_ADDR, 1 << 62, C_ADDR) == qm.QM_ERR_SHAPE
    assert qm.qm_matmul_q4_0_algo_ptr(A_ADDR, W_ADDR, C_ADDR, 1, 4, 32, 99) == qm.QM_ERR_SHAPE


def test_empty_shapes_enqueue_nothing(lib):
    assert qm.qm_matmul_q4_0_ptr(0, 0, 0, 0, 4, 32) == qm.QM_OK
    assert qm.qm_matmul_q4_0_ptr(0, 0, 0, 4, 0, 32) == qm.QM_OK
    assert qm.qm_dequant_q4_0_ptr(0, 0, 0) == qm.QM_OK


def test_null_pointers(lib):
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, 0, 1, 4, 32) == qm.QM_ERR_NULL
    assert qm.qm_matmul_q4_0_ptr(0, W_ADDR, C_ADDR, 1, 4, 32) == qm.QM_ERR_NULL
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, 0, C_ADDR, 1, 4, 32) == qm.QM_ERR_NULL
    assert qm.qm_dequant_q4_0_ptr(0, 3, C_ADDR) == qm.QM_ERR_NULL
    assert qm.qm_dequant_q4_0_ptr(W_ADDR, 3, 0) == qm.QM_ERR_NULL


def test_alignment(lib):
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR + 1, C_ADDR, 1, 4, 32) == qm.QM_ERR_ALIGN
    assert qm.qm_matmul_q4_0_ptr(A_ADDR + 2, W_ADDR, C_ADDR, 1, 4, 32) == qm.QM_ERR_ALIGN
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, C_ADDR + 2, 1, 4, 32) == qm.QM_ERR_ALIGN
    assert qm.qm_dequant_q4_0_ptr(W_ADDR + 1, 3, C_ADDR) == qm.QM_ERR_ALIGN
    assert qm.qm_dequant_q4_0_ptr(W_ADDR, 3, C_ADDR + 1) == qm.QM_ERR_ALIGN


def test_aliasing(lib):
    # C (4 x 4 floats = 64 B) starting inside A (4 x 32 floats)
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, A_ADDR + 64, 4, 4, 32) == qm.QM_ERR_ALIAS
    # C overlapping the tail of the weight stream (4 rows x 1 block = 72 B)
    assert qm.qm_matmul_q4_0_ptr(A_ADDR, W_ADDR, W_ADDR + 68, 4, 4, 32) == qm.QM_ERR_ALIAS
    assert qm.qm_dequant_q4_0_ptr(W_ADDR, 4, W_ADDR + 64) == qm.QM_ERR_ALIAS
    # adjacent, not overlapping: passes the alias check (and fails later only
    # for want of a device, or because the fake address is not device memory)
    rc = qm.qm_dequant_q4_0_ptr(W_ADDR, 4, W_ADDR + 72)
    assert rc in (qm.QM_ERR_CUDA, qm.QM_ERR_POINTER)


def test_forced_algorithm_limits(lib):
    assert qm.qm_matmul_q4_0_algo_ptr(A_ADDR, W_ADDR, C_ADDR, 9, 4, 32,
                                      qm.QM_ALGO_GEMV) == qm.QM_ERR_UNSUPPORTED
    assert qm.qm_matmul_q4_0_algo_ptr(A_ADDR, W_ADDR, C_ADDR, 3, 4, 32,
                                      qm.QM_ALGO_GEMV_PK) == qm.QM_ERR_UNSUPPORTED
    assert qm.qm_matmul_q4_0_algo_ptr(A_ADDR, W_ADDR, C_ADDR, 1, 4, 32, 6) == qm.QM_ERR_SHAPE


def test_python_wrappers_validate_tensors():
    torch = pytest.importorskip("torch")
    with pytest.raises(TypeError):
        qm.qm_dequant_q4_0(torch.zeros(18, dtype=torch.float32))
    with pytest.raises(ValueError):
        qm.qm_dequant_q4_0(torch.zeros(18, dtype=torch.uint8))  # not a CUDA tensor


def test_q8_0_argument_errors(lib):
    # shapes: negative counts, quantize element counts not a multiple of 32,
    # byte counts that overflow
    assert qm.qm_dequant_q8_0_ptr(W_ADDR, -1, C_ADDR) == qm.QM_ERR_SHAPE
    assert qm.qm_dequant_q8_0_ptr(W_ADDR, 1 << 62, C_ADDR) == qm.QM_ERR_SHAPE
    assert qm.qm_quantize_q8_0_ptr(A_ADDR, -32, W_ADDR) == qm.QM_ERR_SHAPE
    assert qm.qm_quantize_q8_0_ptr(A_ADDR, 33, W_ADDR) == qm.QM_ERR_SHAPE
    assert qm.qm_quantize_q8_0_ptr(A_ADDR, 1 << 62, W_ADDR) == qm.QM_ERR_SHAPE
    # empty inputs enqueue nothing
    assert qm.qm_dequant_q8_0_ptr(0, 0, 0) == qm.QM_OK
    assert qm.qm_quantize_q8_0_ptr(0, 0, 0) == qm.QM_OK
    # null pointers
    assert qm.qm_dequant_q8_0_ptr(0, 3, C_ADDR) == qm.QM_ERR_NULL
    assert qm.qm_dequant_q8_0_ptr(W_ADDR, 3, 0) == qm.QM_ERR_NULL
    assert qm.qm_quantize_q8_0_ptr(0, 64, W_ADDR) == qm.QM_ERR_NULL
    assert qm.qm_quantize_q8_0_ptr(A_ADDR, 64, 0) == qm.QM_ERR_NULL
    # alignment: dequant output and quantize input need 4 bytes; the block
    # streams take any alignment
    assert qm.qm_dequant_q8_0_ptr(W_ADDR, 3, C_ADDR + 2) == qm.QM_ERR_ALIGN
    assert qm.qm_quantize_q8_0_ptr(A_ADDR + 2, 64, W_ADDR) == qm.QM_ERR_ALIGN
    assert qm.qm_dequant_q8_0_ptr(W_ADDR + 1, 3, C_ADDR) in (qm.QM_ERR_CUDA, qm.QM_ERR_POINTER)
    assert qm.qm_quantize_q8_0_ptr(A_ADDR, 64, W_ADDR + 1) in (qm.QM_ERR_CUDA, qm.QM_ERR_POINTER)
    # aliasing: 4 blocks = 136 bytes in, 512 bytes out; 64 floats = 256 bytes
    # in, 68 bytes out
    assert qm.qm_dequant_q8_0_ptr(W_ADDR, 4, W_ADDR + 132) == qm.QM_ERR_ALIAS
    assert qm.qm_quantize_q8_0_ptr(A_ADDR, 64, A_ADDR + 252) == qm.QM_ERR_ALIAS
    assert qm.qm_dequant_q8_0_ptr(W_ADDR, 4, W_ADDR + 136) in (qm.QM_ERR_CUDA, qm.QM_ERR_POINTER)


def test_q8_0_python_wrappers_validate_tensors():
    torch = pytest.importorskip("torch")
    with pytest.raises(TypeError):
        qm.qm_dequant_q8_0(torch.zeros(34, dtype=torch.float32))
    with pytest.raises(ValueError):
        qm.qm_dequant_q8_0(torch.zeros(34, dtype=torch.uint8))  # not a CUDA tensor
    with pytest.raises(TypeError):
        qm.qm_quantize_q8_0(torch.zeros(32, dtype=torch.float64))


# ---------------------------------------------------------- qm_gemv_q4_0_list

def _p(A, W, C, N=64, K=256, wait_for=-1):
    return (A, W, C, N, K, wait_for)


def test_list_empty_and_shape_errors(lib):
    assert qm.qm_gemv_q4_0_list_ptr([], 1) == qm.QM_OK
    assert qm.qm_gemv_q4_0_list_ptr([_p(A_ADDR, W_ADDR, C_ADDR)], 0) == qm.QM_OK
    assert qm.qm_gemv_q4_0_list_ptr([_p(A_ADDR, W_ADDR, C_ADDR)], -1) == qm.QM_ERR_SHAPE
    # wait_for must name an earlier problem (or be -1)
    assert qm.qm_gemv_q4_0_list_ptr([_p(A_ADDR, W_ADDR, C_ADDR, wait_for=0)], 1) == qm.QM_ERR_SHAPE
    assert qm.qm_gemv_q4_0_list_ptr([_p(A_ADDR, W_ADDR, C_ADDR, wait_for=-2)], 1) == qm.QM_ERR_SHAPE
    # each problem follows the qm_matmul_q4_0 rules
    assert qm.qm_gemv_q4_0_list_ptr([_p(A_ADDR, W_ADDR, C_ADDR, K=33)], 1) == qm.QM_ERR_SHAPE
    assert qm.qm_gemv_q4_0_list_ptr([_p(A_ADDR, W_ADDR, 0)], 1) == qm.QM_ERR_NULL
    assert qm.qm_gemv_q4_0_list_ptr([_p(A_ADDR, W_ADDR, C_ADDR + 2)], 1) == qm.QM_ERR_ALIGN
    assert qm.qm_gemv_q4_0_list_ptr([_p(A_ADDR, W_ADDR, C_ADDR)], 1, counters=0x40000002) == qm.QM_ERR_ALIGN


def test_list_reserved_field_must_be_zero(lib):
    import ctypes
    arr = (qm.QmGemvProblem * 1)()
    arr[0] = qm.QmGemvProblem(A_ADDR, W_ADDR, C_ADDR, 64, 256, -1, 7)
    rc = lib.qm_gemv_q4_0_list(ctypes.cast(arr, ctypes.c_void_p), 1, 1, None, None)
    assert rc == qm.QM_ERR_SHAPE


def test_list_ordering_rules(lib):
    # Problem 1 reads problem 0's output: allowed only when it waits for 0.
    p0 = _p(A_ADDR, W_ADDR, C_ADDR, N=256, K=256)
    p1_nowait = _p(C_ADDR, W_ADDR + 0x100000, C_ADDR + 0x100000, N=64, K=256)
    assert qm.qm_gemv_q4_0_list_ptr([p0, p1_nowait], 1) == qm.QM_ERR_ALIAS
    # Problem 1 overwrites what problem 0 reads, without waiting: rejected.
    p1_war = _p(A_ADDR + 0x100000, W_ADDR + 0x100000, A_ADDR, N=64, K=256)
    assert qm.qm_gemv_q4_0_list_ptr([p0, p1_war], 1) == qm.QM_ERR_ALIAS
    # Two outputs on the same bytes without an order: rejected.
    p1_waw = _p(A_ADDR + 0x100000, W_ADDR + 0x100000, C_ADDR, N=64, K=256)
    assert qm.qm_gemv_q4_0_list_ptr([p0, p1_waw], 1) == qm.QM_ERR_ALIAS
    # An output over another problem's weights: always rejected.
    p1_w = _p(A_ADDR + 0x100000, W_ADDR + 0x100000, W_ADDR, N=64, K=256, wait_for=0)
    assert qm.qm_gemv_q4_0_list_ptr([p0, p1_w], 1) == qm.QM_ERR_ALIAS
    # Counters over an operand: rejected.
    assert qm.qm_gemv_q4_0_list_ptr([p0], 1, counters=C_ADDR) == qm.QM_ERR_ALIAS
    # With the wait the same list passes the host checks (and then needs a
    # device, which this machine does not have: the status is not an
    # argument error).
    p1_wait = _p(C_ADDR, W_ADDR + 0x100000, C_ADDR + 0x100000, N=64, K=256, wait_for=0)
    rc = qm.qm_gemv_q4_0_list_ptr([p0, p1_wait], 1)
    assert rc not in (qm.QM_ERR_ALIAS, qm.QM_ERR_SHAPE, qm.QM_ERR_NULL, qm.QM_ERR_ALIGN)


def test_list_prebuilt_problem_array_takes_the_same_checks(lib):
    # gemv_problem_array builds the C array once (for callers that pass the
    # same list every step); the call then checks it exactly as a tuple list.
    p0 = _p(A_ADDR, W_ADDR, C_ADDR, N=256, K=256)
    bad = [p0, _p(C_ADDR, W_ADDR + 0x100000, C_ADDR + 0x100000, N=64, K=256)]
    arr = qm.gemv_problem_array(bad)
    assert len(arr) == 2 and arr[1].A == C_ADDR and arr[1].wait_for == -1 and arr[1].reserved == 0
    assert qm.qm_gemv_q4_0_list_ptr(arr, 1) == qm.qm_gemv_q4_0_list_ptr(bad, 1) == qm.QM_ERR_ALIAS
    assert qm.qm_gemv_q4_0_list_ptr(qm.gemv_problem_array([]), 1) == qm.QM_OK
    assert qm.qm_gemv_q4_0_list_ptr(qm.gemv_problem_array([_p(A_ADDR, W_ADDR, C_ADDR, K=33)]), 1) == \
        qm.QM_ERR_SHAPE
