"""Structured inputs on the GPU: inputs whose products all round the same way.

On random inputs the rounding errors of a split-precision product take both
signs and cancel in a sum over K; on structured inputs (constant activations,
constant scales, values placed just below a bf16 rounding midpoint) they all
line up, and a per-product error that the random workloads hide shows up in
full.  Each case is checked element by element against the oracle, with the
tolerance of the matmul sections ("qmatvec_q4_0" / "matmul_q4_0_tiled" of the
quantized kernel-contract page, with |C - C_oracle| <= 1e-5 sum_k |A W| + 1e-7),
at K = 256, 512 and 1024, where a sum of f32 partials per 16- or 32-wide step
stays inside the bound on such inputs.

Activation values (f32):
  * A_MID  = 1 + 2^-8 - 2^-23: just below the bf16 midpoint above 1, so its
    bf16 hi piece is 1 and its lo piece 2^-8;
  * A_RES  = 1 + 2^-9 + 2^-17 - 2^-23: its lo piece rounds 2^-9 + 2^-17 - 2^-23
    down to 2^-9, leaving nearly the largest residual a two-piece bf16 split
    can leave (2^-17 of the value), with the same sign everywhere.
Scale values (binary16):
  * D_MID  = 1 + 3 * 2^-10: its bf16 piece is 1, the remainder 3 * 2^-10;
  * scales whose three mantissa bits past bf16 precision are 011 (just below
    the bf16 midpoint), positive.
"""
import numpy as np
import pytest

import oracle
import synth

from test_gpu_parity import assert_close, matmul_gpu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

A_MID = np.float32(1 + 2.0 ** -8 - 2.0 ** -23)
A_RES = np.float32(1 + 2.0 ** -9 + 2.0 ** -17 - 2.0 ** -23)
D_MID = np.float16(1 + 3 * 2.0 ** -10)


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


def blocks(N, K, d, nibbles):
    """A row-major [N][K/32] block stream from per-block scales d (float16,
    broadcast to [N, K/32]) and per-element nibbles (broadcast to [N, K])."""
    nb = K // 32
    d = np.broadcast_to(np.asarray(d, np.float16), (N, nb)).ravel()
    q = np.broadcast_to(np.asarray(nibbles, np.uint8), (N, K)).reshape(N * nb, 32)
    quant = (q[:, :16] | (q[:, 16:] << 4)).astype(np.uint8)
    return synth.assemble_blocks(d, quant)


def near_midpoint_acts(M, K, seed):
    """Positive f32 values b + 2^(e-8) - 2^(e-23), just below the
    bf16 midpoint above a random bf16 value b of [2^e, 2^(e+1)), e in -2..2."""
    g = synth.rng(seed, (M, K))
    e = g.integers(-2, 3, (M, K))
    k = g.integers(0, 128, (M, K))
    b = (1 + k / 128.0) * 2.0 ** e
    return (b + 2.0 ** (e - 8) - 2.0 ** (e - 23)).astype(np.float32)


def near_midpoint_scales(N, K, seed):
    """Positive binary16 scales in [2^-6, 2^-4) whose mantissa ends in 011."""
    g = synth.rng(seed, (N, K))
    nb = K // 32
    e = g.integers(9, 11, (N, nb)).astype(np.uint16)       # biased exponents 9, 10
    m = ((g.integers(0, 128, (N, nb)) << 3) | 3).astype(np.uint16)
    return ((e << 10) | m).view(np.float16)


def case_inputs(name, M, N, K):
    if name == "all_alike":           # every product A_MID * D_MID
        return np.full((M, K), A_MID, np.float32), blocks(N, K, D_MID, 9)
    if name == "largest_residual":    # every product A_RES * 7 D_MID
        return np.full((M, K), A_RES, np.float32), blocks(N, K, D_MID, 15)
    if name == "const_a_const_d":     # random nibbles, constant A and d
        g = synth.rng(81, (N, K))
        return np.full((M, K), A_MID, np.float32), blocks(N, K, D_MID, g.integers(0, 16, (N, K)))
    if name == "near_midpoints":      # positive products, every value near a midpoint
        g = synth.rng(82, (N, K))
        return near_midpoint_acts(M, K, 83), blocks(N, K, near_midpoint_scales(N, K, 84),
                                                   g.integers(9, 16, (N, K)))
    if name == "zero_weights":        # every nibble 8: C is exactly +0 or -0
        return np.full((M, K), A_MID, np.float32), blocks(N, K, D_MID, 8)
    raise ValueError(name)


CASES = ("all_alike", "largest_residual", "const_a_const_d", "near_midpoints", "zero_weights")

# (algorithm, M): the tensor-core GEMM on two 128-row tiles (the second
# ragged), the tensor-core GEMV at M = 1 and 8, the packed FP32 GEMV at M = 1.
PATHS = [("GEMM_TC", 130), ("GEMV", 1), ("GEMV", 8), ("GEMV_PK", 1)]


@pytest.mark.parametrize("K", [256, 512, 1024])
@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("path", PATHS, ids=lambda p: f"{p[0]}_m{p[1]}")
def test_structured_inputs_within_tolerance(env, path, case, K):
    qm, o = env
    algo_name, M = path
    N = 136
    A, blob = case_inputs(case, M, N, K)
    C = matmul_gpu(qm, A, blob, N, algo=getattr(qm, "QM_ALGO_" + algo_name))
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    assert_close(C, C_ref, S_ref, f"{algo_name} M={M} {case} K={K}")
    if case == "zero_weights":
        assert not np.any(C), "all-8 nibbles must give exact zeros"
