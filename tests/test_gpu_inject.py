"""The host-side failure path: a copy of the library built with its test
hooks (``build_test_hooks()``, ``include/qm_test.h``) makes the next calls of
entry points that would enqueue work fail with QM_ERR_CUDA, as a failed CUDA
call in them would.  Checked: the failing call returns QM_ERR_CUDA, enqueues
nothing (no launch counted, the output keeps its sentinel), leaves the device
error word clear, and the next call works and matches the oracle; the count
covers every kind of entry point; the product library has no such hook.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

QM_OK, QM_ERR_SHAPE, QM_ERR_CUDA = 0, -2, -5


@pytest.fixture(scope="module")
def hooked():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_block_quantized_qm_gb300 import build as qm_build
    lib = ctypes.CDLL(qm_build.build_test_hooks())
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.qm_matmul_q4_0.argtypes = [p, p, p, i64, i64, i64, p]
    lib.qm_dequant_q4_0.argtypes = [p, i64, p, p]
    lib.qm_quantize_q8_0.argtypes = [p, i64, p, p]
    lib.qm_matmul_q4_0_q8act.argtypes = [p, p, p, i64, i64, i64, p]
    lib.qm_device_status.argtypes = [p, i32]
    lib.qm_launch_count.restype = ctypes.c_uint64
    lib.qm_test_inject_error.argtypes = [i32]
    torch.cuda.set_device(0)
    return lib, oracle.load()


def operands(M, N, K, seed):
    A = synth.activations(M, K, seed)
    blob = synth.q4_0_weights(N, K, seed + 1)
    dev = torch.device("cuda", 0)
    return A, blob, torch.from_numpy(A).to(dev), torch.from_numpy(blob).to(dev), \
        torch.full((M, N), float("nan"), device=dev)


def test_product_library_has_no_hook():
    from bit_block_quantized_qm_gb300 import build as qm_build
    lib = ctypes.CDLL(qm_build.build())
    with pytest.raises(AttributeError):
        lib.qm_test_inject_error


def test_injected_failure_enqueues_nothing_and_the_next_call_works(hooked):
    lib, o = hooked
    M, N, K = 1, 1024, 4096
    A, blob, a, w, c = operands(M, N, K, 960)
    s = torch.cuda.current_stream().cuda_stream
    assert lib.qm_test_inject_error(1) == QM_OK
    before = lib.qm_launch_count()
    assert lib.qm_matmul_q4_0(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, s) == QM_ERR_CUDA
    torch.cuda.synchronize()
    assert lib.qm_launch_count() == before, "a failed call launched a kernel"
    assert torch.isnan(c).all(), "a failed call wrote its output"
    assert lib.qm_device_status(s, 1) == QM_OK
    assert lib.qm_matmul_q4_0(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, s) == QM_OK
    torch.cuda.synchronize()
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    assert oracle.within_tolerance(c.cpu().numpy(), C_ref, S_ref).all()


def test_injection_counts_every_kind_of_call(hooked):
    lib, _ = hooked
    M, N, K = 2, 64, 256
    A, blob, a, w, c = operands(M, N, K, 970)
    s = torch.cuda.current_stream().cuda_stream
    n_blocks = N * K // 32
    deq = torch.empty(n_blocks * 32, device="cuda")
    q8 = torch.empty(M * K // 32 * 34, dtype=torch.uint8, device="cuda")
    calls = [
        lambda: lib.qm_matmul_q4_0(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, s),
        lambda: lib.qm_dequant_q4_0(w.data_ptr(), n_blocks, deq.data_ptr(), s),
        lambda: lib.qm_quantize_q8_0(a.data_ptr(), M * K, q8.data_ptr(), s),
        lambda: lib.qm_matmul_q4_0_q8act(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, s),
    ]
    assert lib.qm_test_inject_error(len(calls)) == QM_OK
    for call in calls:
        assert call() == QM_ERR_CUDA
    for call in calls:
        assert call() == QM_OK
    torch.cuda.synchronize()
    assert lib.qm_device_status(s, 1) == QM_OK
    # Argument errors still come first; a pending injection can be cleared.
    assert lib.qm_test_inject_error(-1) == QM_ERR_SHAPE
    assert lib.qm_test_inject_error(5) == QM_OK
    assert lib.qm_matmul_q4_0(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, 100, s) == QM_ERR_SHAPE
    assert lib.qm_test_inject_error(0) == QM_OK
    assert calls[0]() == QM_OK
    torch.cuda.synchronize()
