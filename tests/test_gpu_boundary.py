"""The boundary allocates nothing and synchronizes nothing: after the library
has run once on a device, the first calls on a stream it has never seen (a
split-K GEMV, a split-K GEMM, a list GEMV) leave the device's free memory
unchanged, and the same first calls on another fresh stream can be captured
into a CUDA graph (each call leaves the stream capturing, as a call that
allocated or synchronized would not) whose replays match the oracle."""
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


# (M, N, K): a GEMV and a GEMM whose launch plans split K on a GB300, and a
# GEMV without a split.
SHAPES = [(1, 1024, 4096), (512, 1024, 4096), (8, 4096, 4096)]


def operands(shapes, seed):
    dev = torch.device("cuda", 0)
    out = []
    for i, (M, N, K) in enumerate(shapes):
        blob = synth.q4_0_weights(N, K, seed + i)
        A = synth.activations(M, K, seed + 50 + i)
        out.append((A, blob, torch.from_numpy(A).to(dev), torch.from_numpy(blob).to(dev),
                    torch.empty((M, N), device=dev)))
    return out


def enqueue(qm, ops, stream, check_capturing=False):
    s = int(stream.cuda_stream)
    for (A, blob, a, w, c) in ops:
        M, K = A.shape
        N = c.shape[1]
        assert qm.qm_matmul_q4_0_ptr(a.data_ptr(), w.data_ptr(), c.data_ptr(), M, N, K, s) == qm.QM_OK
        if check_capturing:
            assert torch.cuda.is_current_stream_capturing(), "a call ended the capture"
    # A two-problem list GEMV (M = 1) on the first operands' activations.
    (A, blob, a, w, c) = ops[0]
    lst = [(a.data_ptr(), w.data_ptr(), c.data_ptr(), c.shape[1], A.shape[1], -1)]
    assert qm.qm_gemv_q4_0_list_ptr(lst, 1, 0, s) == qm.QM_OK
    if check_capturing:
        assert torch.cuda.is_current_stream_capturing(), "the list call ended the capture"


def check(o, ops):
    for (A, blob, a, w, c) in ops:
        N, K = c.shape[1], A.shape[1]
        C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
        assert oracle.within_tolerance(c.cpu().numpy(), C_ref, S_ref, REL, ABS).all(), A.shape


def test_splits_are_taken(env):
    qm, _ = env
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    if sm != 152:
        pytest.skip("split expectations are for a 152-SM GB300")
    assert qm.qm_gemv_plan(1, 1024, 4096, sm_count=sm)["S"] > 1
    assert qm.qm_gemm_plan(512, 1024, 4096, sm)["s_rem"] > 1


def test_first_calls_on_a_fresh_stream_allocate_nothing(env):
    qm, o = env
    ops = operands(SHAPES, 800)
    # The library's first calls on this device (kernel loading, attributes,
    # cluster queries) happen on the default stream.
    enqueue(qm, ops, torch.cuda.current_stream())
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    free0, _ = torch.cuda.mem_get_info()
    with torch.cuda.stream(stream):
        enqueue(qm, ops, stream)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert qm.qm_device_status(clear=True) == qm.QM_OK
    check(o, ops)


def test_first_calls_on_a_fresh_stream_can_be_captured(env):
    qm, o = env
    ops = operands(SHAPES, 900)
    enqueue(qm, ops, torch.cuda.current_stream())  # the device is warm, the stream is not
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        enqueue(qm, ops, stream, check_capturing=True)
    for _ in range(2):
        for (_, _, _, _, c) in ops:
            c.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert qm.qm_device_status(clear=True) == qm.QM_OK
        check(o, ops)
