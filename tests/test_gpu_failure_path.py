"""The failure path of the bounded waits, on a GPU, without a fault or a hang.

qm_selftest_wait_timeout runs a kernel whose bounded wait on an mbarrier that
nothing completes runs out.  The error word it sets must reach the host as
QM_ERR_TIMEOUT, stay set until cleared, clear on request, and leave the
context usable: a matmul right after still matches the oracle.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_block_quantized_qm_gb300 import build as qm_build
    qm_build.build()
    import bit_block_quantized_qm_gb300 as qm
    qm.load_library()
    torch.cuda.set_device(0)
    return qm, oracle.load()


def test_wait_that_runs_out_is_reported_and_cleared(env):
    qm, o = env
    assert qm.qm_device_status(clear=True) == qm.QM_OK
    launches = qm.qm_launch_count()
    assert qm.qm_selftest_wait_timeout() == qm.QM_OK
    assert qm.qm_launch_count() == launches + 1
    assert qm.qm_device_status(clear=False) == qm.QM_ERR_TIMEOUT
    assert qm.qm_device_status(clear=False) == qm.QM_ERR_TIMEOUT, "the word stays set"
    assert qm.qm_device_status(clear=True) == qm.QM_ERR_TIMEOUT
    assert qm.qm_device_status(clear=True) == qm.QM_OK

    # The context is still usable: a split-K GEMV (which uses the arrival
    # counters the clear reset) and a GEMM, both against the oracle.
    for (M, N, K) in ((1, 4096, 14336), (16, 300, 1024)):
        blob = synth.q4_0_weights(N, K, 21 + M)
        A = synth.activations(M, K, 22 + M)
        C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
        C = qm.qm_matmul_q4_0(torch.from_numpy(A).cuda(), torch.from_numpy(blob).cuda(), N)
        torch.cuda.synchronize()
        assert qm.qm_device_status(clear=True) == qm.QM_OK
        assert oracle.within_tolerance(C.cpu().numpy(), C_ref, S_ref, 1e-5, 1e-7).all()


def test_timeout_on_another_stream(env):
    qm, _ = env
    s = torch.cuda.Stream()
    assert qm.qm_selftest_wait_timeout(stream=s) == qm.QM_OK
    assert qm.qm_device_status(stream=s, clear=True) == qm.QM_ERR_TIMEOUT
    assert qm.qm_device_status(stream=s, clear=True) == qm.QM_OK
    assert np.isfinite(torch.ones(4, device="cuda").sum().item())
