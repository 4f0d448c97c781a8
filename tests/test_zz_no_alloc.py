"""qm_matmul_q4_0_noalloc: the GEMV for callers that cannot allocate.

Some callers cannot call cudaMalloc at call time (a custom allocator or
memory-pool callback, a process under a hard device-memory cap, a runtime that
owns all device memory).  qm_matmul_q4_0 gives each stream a workspace on
first use; qm_matmul_q4_0_noalloc uses a fixed array inside the library
instead.  This test calls it through the C ABI twice in a row on shapes whose
K is split (so the fixed scratch is really used, and its second use starts
from whatever the first left) and checks each result against qm_matmul_q4_0
within the parity tolerance.  It lives in its own file, collected last.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

REL, ABS = 1e-5, 1e-7


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


# (M, N, K): shapes whose launch plan splits K on GB300 (152 SMs), so the
# fixed scratch holds partial sums and arrival counters; the last is ragged.
SHAPES = [(1, 1024, 4096), (8, 4096, 14336), (3, 300, 3840)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_noalloc_matches_regular_entry_point_twice(env, shape):
    qm, o = env
    M, N, K = shape
    blob = synth.q4_0_weights(N, K, 70 + M)
    A = synth.activations(M, K, 71 + M)
    wq = torch.from_numpy(blob).cuda()
    a = torch.from_numpy(A).cuda()
    s = int(torch.cuda.current_stream().cuda_stream)
    ref = torch.empty((M, N), device="cuda")
    assert qm.qm_matmul_q4_0_ptr(a.data_ptr(), wq.data_ptr(), ref.data_ptr(), M, N, K, s) == qm.QM_OK
    torch.cuda.synchronize()
    ref = ref.cpu().numpy().astype(np.float64)
    g = synth.rng(72, shape)
    mi = np.concatenate([np.zeros(N, np.int64), g.integers(0, M, 256)])
    ni = np.concatenate([np.arange(N), g.integers(0, N, 256)])
    _, S = o.matmul_q4_0_entries(A, blob, N, K, mi, ni)
    for call in range(2):
        out = torch.full((M, N), float("nan"), device="cuda")
        rc = qm.qm_matmul_q4_0_noalloc_ptr(a.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K, s)
        assert rc == qm.QM_OK, qm.qm_status_string(rc)
        torch.cuda.synchronize()
        assert qm.qm_device_status(clear=True) == qm.QM_OK
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"call {call}: unwritten entries"
        assert np.all(np.abs(got[mi, ni] - ref[mi, ni]) <= REL * S + ABS), f"call {call} differs"


def test_noalloc_rejects_prefill_sizes(env):
    qm, _ = env
    a = torch.zeros((9, 64), device="cuda")
    wq = torch.zeros(2 * 2 * 18, dtype=torch.uint8, device="cuda")
    out = torch.zeros((9, 2), device="cuda")
    rc = qm.qm_matmul_q4_0_noalloc_ptr(a.data_ptr(), wq.data_ptr(), out.data_ptr(), 9, 2, 64, 0)
    assert rc == qm.QM_ERR_TOO_LARGE
    assert "fixed scratch" in qm.qm_status_string(rc)
