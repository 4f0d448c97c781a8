"""Back-to-back launches of different kernels on one stream, captured into a
CUDA graph and replayed: the fast kernels start early under programmatic
dependent launch, one GEMV reads the output of another, and the split-K
launches add their K ranges up inside thread-block clusters, so this checks
that every result still matches the oracle after several replays (no kernel
reads an input before the kernel that writes it has finished)."""
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


def test_mixed_sequence_in_a_cuda_graph(env):
    qm, o = env
    # (M, N, K): split-K GEMVs of different plans, one chained on the output
    # of the previous (C of one is A of the next), and a split-K GEMM.
    mm = [(1, 4096, 14336), (8, 1024, 4096), (4, 4096, 4096), (40, 1024, 4096), (1, 2048, 1024)]
    blobs = [synth.q4_0_weights(N, K, 300 + i) for i, (M, N, K) in enumerate(mm)]
    a0 = synth.activations(1, 14336, 301)
    dev = torch.device("cuda", 0)
    W = [torch.from_numpy(b).to(dev) for b in blobs]
    A0 = torch.from_numpy(a0).to(dev)
    A1 = torch.from_numpy(synth.activations(8, 4096, 302)).to(dev)
    A2 = torch.from_numpy(synth.activations(4, 4096, 303)).to(dev)
    A3 = torch.from_numpy(synth.activations(40, 4096, 304)).to(dev)
    C = [torch.empty((M, N), dtype=torch.float32, device=dev) for (M, N, K) in mm]
    x8 = torch.from_numpy(synth.activations(1, 32 * 1000, 305).ravel()).to(dev)
    q8 = torch.empty(1000 * 34, dtype=torch.uint8, device=dev)
    deq = torch.empty(blobs[1].size // 18 * 32, dtype=torch.float32, device=dev)

    def run(stream):
        s = int(stream.cuda_stream)
        ins = [A0, A1, A2, A3, None]
        for i, (M, N, K) in enumerate(mm):
            # The last GEMV reads the first 1024 outputs of the first one as its
            # A (M = 1, so a prefix of C[0]): a true producer -> consumer edge.
            a = ins[i] if ins[i] is not None else C[0]
            assert qm.qm_matmul_q4_0_ptr(a.data_ptr(), W[i].data_ptr(), C[i].data_ptr(),
                                         M, N, K, s) == qm.QM_OK
        assert qm.qm_dequant_q4_0_ptr(W[1].data_ptr(), blobs[1].size // 18, deq.data_ptr(), s) == qm.QM_OK
        assert qm.qm_quantize_q8_0_ptr(x8.data_ptr(), x8.numel(), q8.data_ptr(), s) == qm.QM_OK

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        run(stream)  # first use of each kernel (module load, attributes) outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run(stream)
    for _ in range(3):
        for c in C:
            c.fill_(float("nan"))
        q8.fill_(0xA5)
        deq.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert qm.qm_device_status(clear=True) == qm.QM_OK
        host_in = [a0, A1.cpu().numpy(), A2.cpu().numpy(), A3.cpu().numpy(), None]
        for i, (M, N, K) in enumerate(mm):
            A = host_in[i] if i < 4 else C[0].cpu().numpy()[:, :K]
            C_ref, S_ref = o.matmul_q4_0(np.ascontiguousarray(A, dtype=np.float32), blobs[i], N, K)
            got = C[i].cpu().numpy()
            assert np.all(oracle.within_tolerance(got, C_ref, S_ref, REL, ABS)), f"matmul {i} {mm[i]}"
        want = o.dequant_q4_0(blobs[1])
        assert np.array_equal(deq.cpu().numpy().view(np.uint32), want.view(np.uint32)), "dequant"
        assert np.array_equal(q8.cpu().numpy(), o.quantize_q8_0(x8.cpu().numpy())), "quantize"
