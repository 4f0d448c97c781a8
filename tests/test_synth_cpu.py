"""The seeded input generators (synth/) produce what the input recipe states:
the 18-byte block layout, the scale and nibble distributions, the activation
distributions, reproducibility by (seed, key), and the workloads' shapes."""
import numpy as np
import pytest

import synth


def split_blocks(blob):
    b = blob.reshape(-1, 18)
    d = b[:, 0:2].copy().view("<f2").ravel()
    q = b[:, 2:]
    return d, q


def test_block_layout():
    d = np.array([1.5, -0.25, 0.0], dtype=np.float16)
    q = np.arange(48, dtype=np.uint8).reshape(3, 16)
    blob = synth.assemble_blocks(d, q)
    assert blob.dtype == np.uint8 and blob.size == 3 * 18
    # Little-endian binary16 at bytes 0-1, then the 16 quant bytes.
    assert list(blob[0:2]) == [0x00, 0x3E]            # 1.5 = 0x3E00
    assert list(blob[18:20]) == [0x00, 0xB4]          # -0.25 = 0xB400
    assert np.array_equal(blob.reshape(3, 18)[:, 2:], q)
    with pytest.raises(ValueError):
        synth.assemble_blocks(d, q[:2])


def test_weights_shape_and_reproducibility():
    a = synth.q4_0_weights(7, 96, seed=3)
    assert a.size == synth.blob_bytes(7, 96) == 7 * 3 * 18
    assert np.array_equal(a, synth.q4_0_weights(7, 96, seed=3))
    assert not np.array_equal(a, synth.q4_0_weights(7, 96, seed=4))
    assert not np.array_equal(a, synth.q4_0_weights(7, 96, seed=3, key=(0, 1)))
    with pytest.raises(ValueError):
        synth.q4_0_weights(1, 33, seed=0)


def test_nibbles_are_uniform_and_independent():
    _, q = split_blocks(synth.q4_0_weights(512, 4096, seed=11))
    lo = (q & 15).ravel().astype(np.int64)
    hi = (q >> 4).ravel().astype(np.int64)
    n = lo.size
    for nib in (lo, hi):
        counts = np.bincount(nib, minlength=16)
        chi2 = ((counts - n / 16) ** 2 / (n / 16)).sum()
        assert chi2 < 60, chi2          # 15 degrees of freedom; p < 1e-6 beyond 60
    joint = np.bincount(lo * 16 + hi, minlength=256)
    chi2 = ((joint - n / 256) ** 2 / (n / 256)).sum()
    assert chi2 < 400, chi2             # 255 degrees of freedom


def test_scale_distributions():
    d, _ = split_blocks(synth.q4_0_weights(256, 4096, seed=12))
    d = d.astype(np.float64)
    assert (d >= 0).all()
    # |N(0,1)| * 0.02: mean 0.02 * sqrt(2 / pi), and f16 rounding of the draw.
    assert abs(d.mean() - 0.02 * np.sqrt(2 / np.pi)) < 2e-4
    assert abs(np.median(d) - 0.02 * 0.6744897501960817) < 3e-4
    dl, _ = split_blocks(synth.q4_0_weights(256, 4096, seed=13, scale="log_uniform"))
    dl = dl.astype(np.float64)
    assert dl.min() >= 1e-3 * (1 - 2 ** -10) and dl.max() <= 5e-2 * (1 + 2 ** -10)
    ln = np.log(dl)
    lo, hi = np.log(1e-3), np.log(5e-2)
    assert abs(ln.mean() - (lo + hi) / 2) < 0.02
    with pytest.raises(ValueError):
        synth.q4_0_weights(1, 32, seed=0, scale="nope")


def test_activation_distributions():
    a = synth.activations(64, 4096, seed=14)
    assert a.dtype == np.float32 and a.shape == (64, 4096)
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1.0) < 0.01
    o = synth.activations(64, 4096, seed=15, dist="outliers")
    out = np.abs(o) == 20.0
    frac = out.mean()
    assert abs(frac - 0.01) < 0.002, frac
    assert abs((o[out] > 0).mean() - 0.5) < 0.05
    rest = o[~out]
    assert abs(rest.std() - 0.5) < 0.01
    assert np.array_equal(o, synth.activations(64, 4096, seed=15, dist="outliers"))
    with pytest.raises(ValueError):
        synth.activations(1, 32, seed=0, dist="nope")


def test_workload_shapes():
    w0 = synth.workload(0)
    assert [(c.M, c.N, c.K, c.seed) for c in w0] == [(1, 4096, 4096, 0)]
    w1 = synth.workload(1)
    assert [(c.op, c.M, c.N, c.K, c.seed) for c in w1] == [
        ("matmul", 8, 14336, 4096, 1), ("matmul", 8, 4096, 14336, 2), ("dequant", 0, 14336, 4096, 1)]
    # The dequant is of the up projection's weight.
    assert np.array_equal(w1[2].weights()[:1800], w1[0].weights()[:1800])
    w2 = synth.workload(2)
    assert [(c.M, c.N, c.K, c.a_dist) for c in w2] == [(32, 4096, 4096, "outliers"),
                                                       (256, 4096, 4096, "outliers")]
    w3 = synth.workload(3)
    assert [(c.M, c.N, c.K, c.d_dist) for c in w3] == [(1024, 14336, 4096, "log_uniform"),
                                                       (1024, 4096, 14336, "log_uniform")]
    w4 = synth.workload(4)
    assert len(w4) == 3 * 32 * 7
    per_layer = sum(c.weight_bytes for c in w4 if c.M == 1) / 32
    assert per_layer == 122_683_392          # 122.7 MB of Q4_0 weights per layer
    shapes = {(c.N, c.K) for c in w4}
    assert shapes == {(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)}
    # One weight stream per (layer, projection), shared over M.
    a, b = (c for c in w4 if c.name in ("layer3_k_m1", "layer3_k_m512"))
    assert a.w_key == b.w_key and a.a_key != b.a_key
    with pytest.raises(ValueError):
        synth.workload(5)
