"""GPU parity of qm_matmul_q4_0_q8act (the GEMV fused with a preceding Q8_0
activation quantization) against the oracle's composition
C = dequant_q8_0(quantize_q8_0(A)) x dequant(W)^T, through the C ABI.

* the staged integer kernel (K % 256 == 0, aligned) and the generic one
  (other K, a misaligned A) over M = 1..8, ragged N and K, element by element
  within |C - C'| <= 1e-5 sum_k |A'_k W_k| + 1e-7;
* the decode shapes at full size: 1 x 4096 x 4096 element by element; 8 x
  (14336 x 4096) and 8 x (4096 x 14336) on every column of two rows and 1024
  sampled entries;
* activations past binary16's range (a block scale that narrows to
  infinity) and infinite weight scales: the same class (NaN, +-inf) as the
  composition gives, finite entries within tolerance;
* bitwise the same result on a second call; M > 8, empty and K = 0 shapes.
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


def run(qm, A, blob, N, K, a_offset=0):
    M = A.shape[0]
    dev = torch.device("cuda", 0)
    flat = torch.zeros(M * K + a_offset, dtype=torch.float32, device=dev)
    flat[a_offset:] = torch.from_numpy(A.ravel())
    a = flat[a_offset:]
    w = torch.from_numpy(blob).to(dev)
    out = torch.full((M, N), float("nan"), device=dev)
    rc = qm.qm_matmul_q4_0_q8act_ptr(a.data_ptr(), w.data_ptr(), out.data_ptr(), M, N, K,
                                     int(torch.cuda.current_stream().cuda_stream))
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    torch.cuda.synchronize()
    assert qm.qm_device_status(clear=True) == qm.QM_OK
    return out.cpu().numpy()


SHAPES = [(M, N, K) for M in (1, 2, 3, 5, 8)
          for (N, K) in ((4096, 4096), (1024, 4096), (300, 3840), (33, 768), (64, 14336),
                         (17, 32), (100, 96), (5, 4000))]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_q8act_matches_the_composition(env, shape):
    qm, o = env
    M, N, K = shape
    A = synth.activations(M, K, 600 + M)
    blob = synth.q4_0_weights(N, K, 610 + M)
    got = run(qm, A, blob, N, K)
    C, S = o.matmul_q4_0_q8act(A, blob, N, K)
    ok = oracle.within_tolerance(got, C, S, REL, ABS)
    assert ok.all(), f"{int((~ok).sum())} entries outside tolerance"
    again = run(qm, A, blob, N, K)
    assert np.array_equal(again.view(np.uint32), got.view(np.uint32)), "not deterministic"


@pytest.mark.parametrize("M", [1, 8])
def test_q8act_misaligned_activations_take_the_generic_kernel(env, M):
    qm, o = env
    N, K = 257, 1024
    A = synth.activations(M, K, 620 + M)
    blob = synth.q4_0_weights(N, K, 621)
    got = run(qm, A, blob, N, K, a_offset=1)
    C, S = o.matmul_q4_0_q8act(A, blob, N, K)
    assert oracle.within_tolerance(got, C, S, REL, ABS).all()


def test_q8act_gemv_config0_full(env):
    qm, o = env
    N = K = 4096
    A = synth.activations(1, K, 630)
    blob = synth.q4_0_weights(N, K, 631)
    got = run(qm, A, blob, N, K)
    C, S = o.matmul_q4_0_q8act(A, blob, N, K)
    assert oracle.within_tolerance(got, C, S, REL, ABS).all()


@pytest.mark.parametrize("NK", [(14336, 4096), (4096, 14336)], ids=["up", "down"])
def test_q8act_decode_batch_m8_sampled(env, NK):
    qm, o = env
    N, K = NK
    M = 8
    A = synth.activations(M, K, 640)
    blob = synth.q4_0_weights(N, K, 641)
    got = run(qm, A, blob, N, K)
    g = synth.rng(642, (N, K))
    rows = (0, 5)
    mi = np.concatenate([np.repeat(rows, N), g.integers(0, M, 1024)])
    ni = np.concatenate([np.tile(np.arange(N), len(rows)), g.integers(0, N, 1024)])
    C, S = o.matmul_q4_0_q8act_entries(A, blob, N, K, mi, ni)
    assert oracle.within_tolerance(got[mi, ni], C, S, REL, ABS).all()


@pytest.mark.parametrize("K", [4096, 96], ids=["staged", "generic"])
def test_q8act_non_finite_scales(env, K):
    qm, o = env
    M, N = 2, 48
    A = synth.activations(M, K, 650)
    A[0, 40] = 3.0e7            # block 1 of row 0: max / 127 narrows to binary16 infinity
    A[1, 3] = -1.0e9            # block 0 of row 1 likewise, negative
    blob = synth.q4_0_weights(N, K, 651).copy()
    off = (7 * (K // 32) + 1) * 18  # row 7, block 1: d = +inf with mixed nibbles
    blob[off:off + 2] = np.frombuffer(np.float16(np.inf).tobytes(), np.uint8)
    got = run(qm, A, blob, N, K)
    C, S = o.matmul_q4_0_q8act(A, blob, N, K)
    assert not np.isfinite(C).all(), "the case must reach non-finite results"
    ok = oracle.within_tolerance(got, C, S, REL, ABS)
    assert ok.all(), f"{int((~ok).sum())} entries differ (class or value)"


def test_q8act_shape_rules(env):
    qm, _ = env
    dev = torch.device("cuda", 0)
    a = torch.zeros((9, 64), device=dev)
    w = torch.zeros(2 * 2 * 18, dtype=torch.uint8, device=dev)
    out = torch.zeros((9, 2), device=dev)
    assert qm.qm_matmul_q4_0_q8act_ptr(a.data_ptr(), w.data_ptr(), out.data_ptr(), 9, 2, 64, 0) == \
        qm.QM_ERR_TOO_LARGE
    assert qm.qm_matmul_q4_0_q8act_ptr(a.data_ptr(), w.data_ptr(), out.data_ptr(), 1, 2, 48, 0) == \
        qm.QM_ERR_SHAPE
    assert qm.qm_matmul_q4_0_q8act_ptr(a.data_ptr(), w.data_ptr(), out.data_ptr(), 0, 2, 64, 0) == qm.QM_OK
    out.fill_(7.0)
    assert qm.qm_matmul_q4_0_q8act_ptr(a.data_ptr(), w.data_ptr(), out.data_ptr(), 2, 2, 0, 0) == qm.QM_OK
    torch.cuda.synchronize()
    assert torch.all(out[:2] == 0) and torch.all(out[2:] == 7.0)
