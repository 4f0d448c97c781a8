"""GPU parity of the Q8_0 dequant and quantize against the CPU oracle.

Both operations are exact functions of their inputs (the dequant by the
definition qs * d; the quantize by the readings stated in include/qm.h), so
every comparison is bit for bit: f32 outputs by their bit patterns (NaN by
class), Q8_0 blocks byte for byte.  Outputs sit between guard words that must
survive.  Block counts straddle the 32-block groups of the fast kernels, and
pointer offsets send work to the generic kernels.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle_pins import load_golden_q8_0_blocks, load_golden_q8_0_quantize

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GUARD = 0xA5


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


def dev_bytes(a: np.ndarray, offset: int, pad: int = 64):
    raw = torch.zeros(a.nbytes + offset + pad, dtype=torch.uint8, device="cuda")
    raw[offset:offset + a.nbytes] = torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).ravel()).cuda()
    return raw


def dequant_gpu(qm, blob: np.ndarray, w_off=0, o_off=0) -> np.ndarray:
    n_blocks = blob.size // 34
    w = dev_bytes(blob, w_off)
    out_bytes = n_blocks * 128
    o = torch.full((out_bytes + o_off + 64,), GUARD, dtype=torch.uint8, device="cuda")
    rc = qm.qm_dequant_q8_0_ptr(w.data_ptr() + w_off, n_blocks, o.data_ptr() + o_off, 0)
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    torch.cuda.synchronize()
    host = o.cpu().numpy()
    assert np.all(host[:o_off] == GUARD) and np.all(host[o_off + out_bytes:] == GUARD), "write outside out"
    return host[o_off:o_off + out_bytes].view(np.float32)


def quantize_gpu(qm, x: np.ndarray, x_off=0, o_off=0) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    xd = dev_bytes(x, x_off)
    out_bytes = x.size // 32 * 34
    o = torch.full((out_bytes + o_off + 64,), GUARD, dtype=torch.uint8, device="cuda")
    rc = qm.qm_quantize_q8_0_ptr(xd.data_ptr() + x_off, x.size, o.data_ptr() + o_off, 0)
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    torch.cuda.synchronize()
    host = o.cpu().numpy()
    assert np.all(host[:o_off] == GUARD) and np.all(host[o_off + out_bytes:] == GUARD), "write outside out"
    return host[o_off:o_off + out_bytes]


def assert_bits_equal(got, want):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    nan_w = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan_w), "NaN positions differ"
    bad = got.view(np.uint32)[~nan_w] != want.view(np.uint32)[~nan_w]
    assert not bad.any(), f"{bad.sum()} elements differ, first at {np.argwhere(bad)[:4].ravel()}"


def random_q8_0(n_blocks: int, seed: int, specials: bool = True) -> np.ndarray:
    g = synth.rng(seed, (81,))
    raw = g.integers(0, 256, size=(n_blocks, 34), dtype=np.uint8)
    d = (g.standard_normal(n_blocks) * np.exp(g.uniform(-14, 9, n_blocks))).astype(np.float16)
    if specials and n_blocks >= 8:
        d[:8] = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 6e-8, -65504, 1e-5], dtype=np.float16)
    raw[:, 0:2] = d.view(np.uint8).reshape(n_blocks, 2)
    return raw.ravel()


def random_f32(n: int, seed: int, kind: str) -> np.ndarray:
    g = synth.rng(seed, (82, ("normal", "wide", "outliers", "special").index(kind)))
    if kind == "normal":
        return g.standard_normal(n).astype(np.float32)
    if kind == "wide":  # per-block magnitudes from 1e-30 to 1e6
        blocks = n // 32
        scale = np.exp(g.uniform(-69, 14, blocks)).repeat(32)
        return (g.standard_normal(n) * scale).astype(np.float32)
    if kind == "outliers":
        x = (0.5 * g.standard_normal(n)).astype(np.float32)
        hit = g.random(n) < 0.01
        x[hit] = np.where(g.random(hit.sum()) < 0.5, -20.0, 20.0)
        return x
    if kind == "special":  # zeros, -0, NaN, inf, subnormal and huge blocks mixed in
        x = g.standard_normal(n).astype(np.float32)
        nb = n // 32
        sel = g.integers(0, 7, nb)
        for b in range(nb):
            blk = x[32 * b:32 * b + 32]
            if sel[b] == 0:
                blk[:] = 0.0
            elif sel[b] == 1:
                blk[:] = -0.0
            elif sel[b] == 2:
                blk[g.integers(0, 32)] = np.nan
            elif sel[b] == 3:
                blk[g.integers(0, 32)] = np.inf if g.random() < 0.5 else -np.inf
            elif sel[b] == 4:
                blk *= np.float32(1e-40)  # subnormal f32 block
            elif sel[b] == 5:
                blk *= np.float32(3e8)  # d beyond binary16
        return x
    raise ValueError(kind)


# ------------------------------------------------------------------ dequant

def test_dequant_q8_0_golden(env):
    qm, o = env
    blocks, values = load_golden_q8_0_blocks()
    got = dequant_gpu(qm, np.frombuffer(b"".join(blocks), dtype=np.uint8))
    assert_bits_equal(got, np.concatenate(values))


@pytest.mark.parametrize("n_blocks", [1, 31, 32, 33, 63, 1000, 4097])
@pytest.mark.parametrize("offs", [(0, 0), (1, 0), (2, 4), (0, 4), (16, 16)])
def test_dequant_q8_0_bit_exact(env, n_blocks, offs):
    qm, o = env
    blob = random_q8_0(n_blocks, 100 + n_blocks)
    assert_bits_equal(dequant_gpu(qm, blob, *offs), o.dequant_q8_0(blob))


def test_dequant_q8_0_full_size(env):
    qm, o = env
    blob = random_q8_0(14336 * 4096 // 32, 7, specials=False)
    assert_bits_equal(dequant_gpu(qm, blob), o.dequant_q8_0(blob))


# ------------------------------------------------------------------ quantize

def test_quantize_q8_0_golden(env):
    qm, o = env
    xs, blocks = load_golden_q8_0_quantize()
    got = quantize_gpu(qm, np.concatenate(xs)).reshape(len(xs), 34)
    for i, b in enumerate(blocks):
        assert np.array_equal(got[i], np.frombuffer(b, dtype=np.uint8)), f"golden case {i}: {got[i][:8]}"


@pytest.mark.parametrize("kind", ["normal", "wide", "outliers", "special"])
@pytest.mark.parametrize("n_blocks", [1, 32, 33, 1000, 4097])
@pytest.mark.parametrize("offs", [(0, 0), (4, 0), (0, 1), (0, 2), (16, 16)])
def test_quantize_q8_0_bit_exact(env, kind, n_blocks, offs):
    qm, o = env
    x = random_f32(32 * n_blocks, 200 + n_blocks, kind)
    got = quantize_gpu(qm, x, *offs)
    want = o.quantize_q8_0(x)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} bytes differ; first block {bad[0] // 34}"


def test_quantize_then_dequant_full_size(env):
    # 14336 x 4096 elements (58.7 M): quantize on the GPU, compare all bytes,
    # then dequantize the GPU's blocks on the GPU and compare all values.
    qm, o = env
    x = random_f32(14336 * 4096, 8, "normal")
    blob = quantize_gpu(qm, x)
    want = o.quantize_q8_0(x)
    assert np.array_equal(blob, want), "quantize differs"
    assert_bits_equal(dequant_gpu(qm, blob), o.dequant_q8_0(want))


def test_q8_0_deterministic(env):
    qm, o = env
    x = random_f32(32 * 5000, 9, "wide")
    a = quantize_gpu(qm, x)
    b = quantize_gpu(qm, x)
    assert np.array_equal(a, b)


def test_quantize_q8_0_near_half_integers(env):
    # Elements within a few ulp of (k + 1/2) * d for random block scales: the
    # quotient x / d sits at a rounding boundary, where the kernel must decide
    # exactly as rounding the correctly rounded quotient does.
    qm, o = env
    g = synth.rng(10, (83,))
    nb = 8192
    amax = np.exp(g.uniform(-20, 20, nb)).astype(np.float32)
    d = (amax / np.float32(127)).astype(np.float32)
    k = g.integers(-126, 126, size=(nb, 31)).astype(np.float32)
    x = ((k + np.float32(0.5)) * d[:, None]).astype(np.float32)
    steps = g.integers(-3, 4, size=(nb, 31))
    x = np.nextafter(x, np.where(steps >= 0, np.inf, -np.inf).astype(np.float32)) * (steps != 0) + x * (steps == 0)
    for s in range(2, 4):
        far = np.abs(steps) >= s
        x[far] = np.nextafter(x[far], np.where(steps[far] > 0, np.inf, -np.inf).astype(np.float32))
    blocks = np.concatenate([amax[:, None], x.astype(np.float32)], axis=1).astype(np.float32)
    got = quantize_gpu(qm, blocks)
    want = o.quantize_q8_0(blocks)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} bytes differ; first block {bad[0] // 34}"
