"""qm_matmul_q4_0_noalloc: the GEMV for callers that cannot allocate.

Some callers cannot call cudaMalloc at call time (a custom allocator or
memory-pool callback, a process under a hard device-memory cap, a runtime that
owns all device memory).  qm_matmul_q4_0_noalloc meets the partial sums of a
split K in a fixed array inside the library (qm_matmul_q4_0 adds them up
inside thread-block clusters).  This test calls it through the C ABI twice in
a row on shapes whose K is split (checked against its launch plan, so the
fixed scratch really holds partial sums and counters, and its second use
starts from whatever the first left), checks each result against
qm_matmul_q4_0 and against the oracle within the parity tolerance, and checks
that a first call on a fresh stream leaves the device's free memory
unchanged.  It lives in its own file, collected last.
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


# The fixed array: 1 MB of partial sums (262144 floats) and 4096 counters.
ARRAY_FLOATS, ARRAY_COUNTERS = 262144, 4096


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_noalloc_matches_regular_entry_point_twice(env, shape):
    qm, o = env
    M, N, K = shape
    # The shape splits K on this device, and the split fits the fixed array,
    # so the allocation-free call takes the same split through the array.
    props = torch.cuda.get_device_properties(0)
    if K % 256 == 0:
        plan = qm.qm_gemv_plan(M, N, K, packed=False, sm_count=props.multi_processor_count, noalloc=True)
        assert plan is not None and plan["S"] > 1, f"no K split for {shape}: {plan}"
        assert plan["RG"] * plan["S"] * M * 16 <= ARRAY_FLOATS and plan["RG"] <= ARRAY_COUNTERS
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
    mi = np.concatenate([np.repeat(np.arange(M), N), g.integers(0, M, 256)])
    ni = np.concatenate([np.tile(np.arange(N), M), g.integers(0, N, 256)])
    C_or, S = o.matmul_q4_0_entries(A, blob, N, K, mi, ni)
    for call in range(2):
        out = torch.full((M, N), float("nan"), device="cuda")
        rc = qm.qm_matmul_q4_0_noalloc_ptr(a.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K, s)
        assert rc == qm.QM_OK, qm.qm_status_string(rc)
        torch.cuda.synchronize()
        assert qm.qm_device_status(clear=True) == qm.QM_OK
        got = out.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"call {call}: unwritten entries"
        assert np.all(np.abs(got[mi, ni] - ref[mi, ni]) <= REL * S + ABS), f"call {call} differs"
        assert np.all(np.abs(got[mi, ni] - C_or) <= REL * S + ABS), f"call {call} misses the oracle"


def test_noalloc_first_call_on_a_fresh_stream_allocates_nothing(env):
    qm, _ = env
    M, N, K = 1, 1024, 4096
    blob = synth.q4_0_weights(N, K, 75)
    wq = torch.from_numpy(blob).cuda()
    a = torch.from_numpy(synth.activations(M, K, 76)).cuda()
    out = torch.empty((M, N), device="cuda")
    # One call first, so that loading the kernel's code (which the driver may
    # do at a kernel's first launch) is not counted; then a call on a stream
    # the library has never seen.
    rc = qm.qm_matmul_q4_0_noalloc_ptr(a.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K, 0)
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    rc = qm.qm_matmul_q4_0_noalloc_ptr(a.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K,
                                       int(stream.cuda_stream))
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_noalloc_rejects_prefill_sizes(env):
    qm, _ = env
    a = torch.zeros((9, 64), device="cuda")
    wq = torch.zeros(2 * 2 * 18, dtype=torch.uint8, device="cuda")
    out = torch.zeros((9, 2), device="cuda")
    rc = qm.qm_matmul_q4_0_noalloc_ptr(a.data_ptr(), wq.data_ptr(), out.data_ptr(), 9, 2, 64, 0)
    assert rc == qm.QM_ERR_TOO_LARGE
    assert "fixed scratch" in qm.qm_status_string(rc)
