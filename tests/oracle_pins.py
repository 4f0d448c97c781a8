"""Pins that tie the CPU oracle to facts outside itself.

Each ``pin_*`` takes a loaded oracle and raises ``AssertionError`` if the
oracle disagrees with a fact that the kernel-contract page ("fuel-vulkan-kernels
— quantized (GGML) kernel contracts", sections ``dequant_q4_0``,
``qmatvec_q4_0``, ``matmul_q4_0_tiled``) or plain mathematics fixes:

* an independent binary16 decoder (numpy's), exhaustively;
* hand-built blocks and a hand-computed product (``tests/golden/``);
* closed forms (all-8 nibbles, zero scale, one-hot and all-ones activations);
* agreement with an independent dense fp64 product (numpy) on dequantized
  weights, row-independence (M=1 against a row of M=8) and invariance under a
  joint permutation of K-blocks;
* for Q8_0 (sections ``dequant_q8_0`` and ``quantize_q8_0``): hand-built
  blocks and hand-worked quantizations (``tests/golden/``), numpy's own
  float -> binary16 narrowing, an int8 x binary16 dequant written with numpy
  views, the round-trip bound |qs d - x| <= d / 2, sign symmetry and
  invariance of the quants under power-of-two scaling;
* for the product with the activations quantized first (the act-quant fusion
  of "vulkan: shader and sequencing efficiency backlog"): a hand-computed
  product (``tests/golden/``), identity with the plain product on
  activations that Q8_0 holds exactly, the block-factored integer form
  sum_b d_w d_a sum_j (q - 8) qs computed with numpy integers from the quant
  bytes, and the bound |C' - C| <= sum_k |a_k - a'_k| |W_k| against the plain
  product.

The same functions run against copies of the oracle with a planted mistake
(``test_oracle_mutants.py``); every such copy must fail at least one pin.
"""
from __future__ import annotations

import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _same_bits_or_nan(got, want) -> bool:
    """Bit equality of float32 arrays, except that NaN matches any NaN."""
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    if got.shape != want.shape:
        return False
    nan_w = np.isnan(want)
    if not np.array_equal(np.isnan(got), nan_w):
        return False
    return np.array_equal(got.view(np.uint32)[~nan_w], want.view(np.uint32)[~nan_w])


def load_golden_blocks():
    blocks, values = [], []
    with open(os.path.join(GOLDEN, "q4_0_hand_blocks.txt")) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "block":
                blocks.append(bytes(int(x, 16) for x in parts[1:]))
                assert len(blocks[-1]) == 18
            elif parts[0] == "values":
                values.append(np.array([float(x) for x in parts[1:]], dtype=np.float32))
                assert values[-1].size == 32
    assert len(blocks) == len(values) and blocks
    return blocks, values


def load_golden_matmul(name="q4_0_hand_matmul.txt"):
    rec = {"wrow": [], "arow": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            key, rest = parts[0], parts[1:]
            if key in ("M", "N", "K"):
                rec[key] = int(rest[0])
            elif key == "wrow":
                rec["wrow"].append(bytes(int(x, 16) for x in rest))
            elif key == "arow":
                rec["arow"].append([float(x) for x in rest])
            elif key in ("C", "S"):
                rec[key] = np.array([float(x) for x in rest]).reshape(rec["M"], rec["N"])
    blob = np.frombuffer(b"".join(rec["wrow"]), dtype=np.uint8)
    A = np.array(rec["arow"], dtype=np.float32)
    return rec["M"], rec["N"], rec["K"], A, blob, rec["C"], rec["S"]


# ---------------------------------------------------------------- binary16

def _parse_float(tok: str) -> float:
    t = tok.lower()
    if t.startswith("0x") or t.startswith("-0x"):
        return float.fromhex(t)
    return float(t)


def load_golden_q8_0_blocks():
    blocks, values = [], []
    with open(os.path.join(GOLDEN, "q8_0_hand_blocks.txt")) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "block":
                blocks.append(bytes(int(x, 16) for x in parts[1:]))
                assert len(blocks[-1]) == 34
            elif parts[0] == "values":
                values.append(np.array([float(x) for x in parts[1:]], dtype=np.float32))
                assert values[-1].size == 32
    assert len(blocks) == len(values) and blocks
    return blocks, values


def load_golden_q8_0_quantize():
    xs, blocks = [], []
    with open(os.path.join(GOLDEN, "q8_0_hand_quantize.txt")) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "x":
                xs.append(np.array([_parse_float(t) for t in parts[1:]], dtype=np.float32))
                assert xs[-1].size == 32
            elif parts[0] == "block":
                blocks.append(bytes(int(x, 16) for x in parts[1:]))
                assert len(blocks[-1]) == 34
    assert len(xs) == len(blocks) and xs
    return xs, blocks


def pin_f16_exhaustive(o):
    bits = np.arange(65536, dtype=np.uint16)
    got = o.f16_to_double(bits)
    want = bits.view(np.float16).astype(np.float64)
    nan_w = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan_w), "NaN class differs"
    assert np.array_equal(got[~nan_w], want[~nan_w]), "binary16 values differ"
    assert np.array_equal(np.signbit(got[~nan_w]), np.signbit(want[~nan_w])), "zero sign differs"


# ---------------------------------------------------------------- dequant

def pin_golden_blocks(o):
    blocks, values = load_golden_blocks()
    got = o.dequant_q4_0(np.frombuffer(b"".join(blocks), dtype=np.uint8))
    want = np.concatenate(values)
    for i in range(len(blocks)):
        sl = slice(32 * i, 32 * i + 32)
        assert _same_bits_or_nan(got[sl], want[sl]), f"hand-built block {i} differs"


def pin_all8_and_zero_scale(o):
    g = synth.rng(11, (0,))
    nb = 64
    d = (g.standard_normal(nb) * 0.05).astype(np.float16)
    blob = synth.assemble_blocks(d, np.full((nb, 16), 0x88, dtype=np.uint8))
    out = o.dequant_q4_0(blob).reshape(nb, 32)
    assert np.all(out == 0), "all-8 nibbles must give zeros"
    want_sign = np.signbit(d.astype(np.float32))[:, None].repeat(32, axis=1)
    assert np.array_equal(np.signbit(out), want_sign), "zero sign must follow d"
    qb = synth.rng(11, (1,)).integers(0, 256, size=(nb, 16), dtype=np.uint8)
    zero = o.dequant_q4_0(synth.assemble_blocks(np.zeros(nb, np.float16), qb))
    assert np.all(zero == 0), "d = 0 must give zeros"
    A = synth.activations(3, 64, 12)
    C, S = o.matmul_q4_0(A, blob[: 2 * 2 * 18], 2, 64)
    assert np.all(C == 0) and np.all(S == 0), "all-8 weights must give C = 0"


def pin_extreme_nibbles(o):
    # q = 0 gives -8d and q = 15 gives 7d, for a d with all 11 significand bits.
    d = np.array([np.float16(0.0999755859375)], dtype=np.float16)  # 0x2E66
    for byte, lo, hi in ((0x00, -8.0, -8.0), (0xFF, 7.0, 7.0), (0xF0, -8.0, 7.0)):
        out = o.dequant_q4_0(synth.assemble_blocks(d, np.full((1, 16), byte, np.uint8)))
        dd = float(d[0])
        assert np.array_equal(out[:16], np.full(16, lo * dd, np.float32))
        assert np.array_equal(out[16:], np.full(16, hi * dd, np.float32))


# ---------------------------------------------------------------- matmul

def pin_golden_matmul(o):
    M, N, K, A, blob, C_want, S_want = load_golden_matmul()
    C, S = o.matmul_q4_0(A, blob, N, K)
    assert np.array_equal(C, C_want), f"hand product differs: {C} vs {C_want}"
    assert np.array_equal(S, S_want), f"hand |product| sum differs: {S} vs {S_want}"


def pin_one_hot(o):
    # A = rows of the identity picks single weights: C[m][n] = W[n][k_m].
    N, K = 5, 96
    blob = synth.q4_0_weights(N, K, 21)
    W = o.dequant_q4_0(blob).reshape(N, K).astype(np.float64)
    ks = np.array([0, 15, 16, 31, 32, 63, 64, 95])
    A = np.zeros((ks.size, K), np.float32)
    A[np.arange(ks.size), ks] = 1.0
    C, S = o.matmul_q4_0(A, blob, N, K)
    assert np.array_equal(C, W[:, ks].T), "one-hot rows must select W[n][k]"
    assert np.array_equal(S, np.abs(W[:, ks].T))


def pin_ones_closed_form(o):
    # A = 1: C[n] = sum_b d_b * (sum of the block's 32 nibbles - 256), and the
    # nibble sum of a byte is (byte & 15) + (byte >> 4) whatever the order.
    N, K = 7, 160
    blob = synth.q4_0_weights(N, K, 22)
    blocks = blob.reshape(N, K // 32, 18)
    d = blocks[:, :, 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    qb = blocks[:, :, 2:].astype(np.int64)
    nib_sum = (qb & 15).sum(-1) + (qb >> 4).sum(-1) - 256
    want = (d * nib_sum).sum(-1)
    C, _ = o.matmul_q4_0(np.ones((1, K), np.float32), blob, N, K)
    assert np.allclose(C[0], want, rtol=1e-13, atol=0), "all-ones closed form differs"


def pin_dense_equivalence(o):
    # Fused product == dense fp64 product of A and the dequantized W (numpy).
    for (M, N, K, seed) in ((3, 4, 64, 23), (9, 7, 96, 24), (1, 33, 32, 25)):
        blob = synth.q4_0_weights(N, K, seed)
        A = synth.activations(M, K, seed, dist="outliers")
        W = o.dequant_q4_0(blob).reshape(N, K).astype(np.float64)
        dense = A.astype(np.float64) @ W.T
        dense_abs = np.abs(A.astype(np.float64)) @ np.abs(W).T
        C, S = o.matmul_q4_0(A, blob, N, K)
        assert np.allclose(C, dense, rtol=0, atol=1e-12 * dense_abs.max() + 1e-300)
        assert np.allclose(S, dense_abs, rtol=1e-13, atol=0)


def pin_rows_independent(o):
    # Row r of an M=8 product equals the M=1 product of A's row r alone.
    N, K = 6, 128
    blob = synth.q4_0_weights(N, K, 26)
    A = synth.activations(8, K, 26)
    C8, S8 = o.matmul_q4_0(A, blob, N, K)
    for r in (0, 3, 7):
        C1, S1 = o.matmul_q4_0(A[r:r + 1], blob, N, K)
        assert np.array_equal(C1[0], C8[r]) and np.array_equal(S1[0], S8[r])


def pin_block_permutation(o):
    # Permuting whole K-blocks of A and W together leaves C unchanged.
    N, K = 4, 256
    nbk = K // 32
    blob = synth.q4_0_weights(N, K, 27)
    A = synth.activations(2, K, 27)
    perm = synth.rng(27, (9,)).permutation(nbk)
    blob_p = blob.reshape(N, nbk, 18)[:, perm, :].ravel()
    A_p = A.reshape(2, nbk, 32)[:, perm, :].reshape(2, K)
    C, S = o.matmul_q4_0(A, blob, N, K)
    Cp, Sp = o.matmul_q4_0(A_p, blob_p, N, K)
    assert np.allclose(C, Cp, rtol=0, atol=1e-12 * S.max())
    assert np.allclose(S, Sp, rtol=1e-13, atol=0)


def pin_entries_match_full(o):
    # The sampled-entry routine agrees exactly with the full product.
    N, K, M = 9, 64, 5
    blob = synth.q4_0_weights(N, K, 28)
    A = synth.activations(M, K, 28)
    C, S = o.matmul_q4_0(A, blob, N, K)
    mi = np.array([0, 4, 2, 4, 1])
    ni = np.array([8, 0, 3, 8, 5])
    Ce, Se = o.matmul_q4_0_entries(A, blob, N, K, mi, ni)
    assert np.array_equal(Ce, C[mi, ni]) and np.array_equal(Se, S[mi, ni])


# ---------------------------------------------------------------- Q8_0

def pin_f16_narrowing_vs_numpy(o):
    """f32 -> binary16 against numpy's conversion (round to nearest even):
    every binary16 value, every midpoint between neighbours (the ties), values
    just around the overflow threshold, and random floats over the range."""
    h = np.arange(0x7C00, dtype=np.uint16)  # +0 .. largest finite
    v = h.view(np.float16).astype(np.float32)
    mids = ((v[:-1].astype(np.float64) + v[1:].astype(np.float64)) / 2).astype(np.float32)
    g = synth.rng(13, (0,))
    rnd = (g.standard_normal(20000) * np.exp(g.uniform(-25, 12, 20000))).astype(np.float32)
    edge = np.float32([65504, 65510, 65519.996, 65520, 65536, 1e9, 2.0**-24, 2.0**-25,
                       2.0**-25 * 1.0000001, 3 * 2.0**-26, 2.0**-14, 2.0**-14 * 0.99999994])
    x = np.concatenate([v, -v, mids, -mids, rnd, edge, -edge, np.float32([np.inf, -np.inf])])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = o.float_to_f16(x)
    bad = got != want
    assert not bad.any(), f"{bad.sum()} narrowings differ, e.g. x={x[bad][:3]}"
    nan = o.float_to_f16(np.float32([np.nan]))[0]
    assert (nan & 0x7C00) == 0x7C00 and (nan & 0x3FF) != 0, "NaN must stay NaN"


def pin_q8_0_golden_blocks(o):
    blocks, values = load_golden_q8_0_blocks()
    got = o.dequant_q8_0(np.frombuffer(b"".join(blocks), dtype=np.uint8))
    want = np.concatenate(values)
    for i in range(len(blocks)):
        sl = slice(32 * i, 32 * i + 32)
        assert _same_bits_or_nan(got[sl], want[sl]), f"hand-built Q8_0 block {i} differs"


def pin_q8_0_dequant_numpy(o):
    """qs * d with numpy: the quants as an int8 view, d as a float16 view."""
    g = synth.rng(14, (0,))
    nb = 256
    raw = g.integers(0, 256, size=(nb, 34), dtype=np.uint8)
    d = (g.standard_normal(nb) * np.exp(g.uniform(-12, 8, nb))).astype(np.float16)
    raw[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    want = (raw[:, 2:].view(np.int8).astype(np.float64) *
            raw[:, 0:2].copy().view(np.float16).astype(np.float64)).astype(np.float32)
    got = o.dequant_q8_0(raw.ravel()).reshape(nb, 32)
    assert _same_bits_or_nan(got, want), "Q8_0 dequant differs from qs * d"


def pin_q8_0_golden_quantize(o):
    xs, blocks = load_golden_q8_0_quantize()
    got = o.quantize_q8_0(np.concatenate(xs)).reshape(len(xs), 34)
    for i, b in enumerate(blocks):
        want = np.frombuffer(b, dtype=np.uint8)
        assert np.array_equal(got[i], want), f"hand-worked quantization {i} differs: {got[i][:8]}"


def _q8_blocks(o, x):
    blob = o.quantize_q8_0(x).reshape(-1, 34)
    scale = blob[:, 0:2].copy().view(np.float16).ravel()
    qs = blob[:, 2:].view(np.int8)
    return blob, scale, qs


def pin_q8_0_roundtrip_bound(o):
    """For finite blocks whose scale stays in binary16's normal range: the
    largest |x| gets |qs| = 127, every |qs d - x| <= d / 2 (d = max|x| / 127,
    up to the f32 rounding of the quotient), and the stored scale is within
    half a binary16 step of d."""
    g = synth.rng(15, (0,))
    nb = 4096
    x = (g.standard_normal((nb, 32)) * np.exp(g.uniform(-4, 9, (nb, 1)))).astype(np.float32)
    x[::7, 5] *= 40.0  # some outliers
    _, scale, qs = _q8_blocks(o, x)
    amax = np.max(np.abs(x).astype(np.float64), axis=1)
    d = amax / 127.0
    err = np.abs(qs.astype(np.float64) * d[:, None] - x.astype(np.float64))
    assert np.all(err <= d[:, None] * (0.5 + 1e-6)), "a quant is more than d/2 off"
    imax = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(qs[np.arange(nb), imax]) == 127), "the largest element must map to 127"
    assert np.all(np.abs(scale.astype(np.float64) - d) <= d * 2.0**-11), "scale not near d"


def pin_q8_0_symmetry_and_scaling(o):
    """quantize(-x): same scale, negated quants; quantize(x * 2^k): same quants,
    scale times 2^k (all in binary16's normal range)."""
    g = synth.rng(16, (0,))
    nb = 512
    x = (g.standard_normal((nb, 32)) * np.exp(g.uniform(-2, 3, (nb, 1)))).astype(np.float32)
    b0, s0, q0 = _q8_blocks(o, x)
    b1, s1, q1 = _q8_blocks(o, -x)
    assert np.array_equal(b0[:, 0:2], b1[:, 0:2]), "scale depends on the sign of x"
    assert np.array_equal(q0.astype(np.int16), -q1.astype(np.int16)), "quants not odd in x"
    for k in (-3, 5):
        _, s2, q2 = _q8_blocks(o, x * np.float32(2.0**k))
        assert np.array_equal(q0, q2), f"quants change under scaling by 2^{k}"
        assert np.array_equal(s0.astype(np.float64) * 2.0**k, s2.astype(np.float64)), \
            f"scale does not scale by 2^{k}"


# ------------------------------------------ product with quantized activations

def pin_q8act_golden(o):
    M, N, K, A, blob, C_want, S_want = load_golden_matmul("q8act_hand_matmul.txt")
    C, S = o.matmul_q4_0_q8act(A, blob, N, K)
    assert np.array_equal(C, C_want), f"hand-computed product differs: {C}"
    assert np.array_equal(S, S_want), f"hand-computed absolute sums differ: {S}"


def pin_q8act_identity_on_representable(o):
    """Blocks of integers in [-127, 127] times 2^e with a +-127 in each: the
    scale is exactly 2^e and the quants are the integers, so A' = A and the
    product equals the plain one bit for bit."""
    g = synth.rng(21, (0,))
    M, N, K = 3, 40, 256
    ints = g.integers(-127, 128, (M, K // 32, 32))
    ints[:, :, 0] = np.where(g.integers(0, 2, (M, K // 32)) == 1, 127, -127)
    e = g.integers(-10, 6, (M, K // 32, 1))
    A = (ints * np.exp2(e)).astype(np.float32).reshape(M, K)
    blob = synth.q4_0_weights(N, K, 22)
    C1, S1 = o.matmul_q4_0_q8act(A, blob, N, K)
    C0, S0 = o.matmul_q4_0(A, blob, N, K)
    assert np.array_equal(C1, C0) and np.array_equal(S1, S0), "A' differs from an exactly representable A"


def pin_q8act_integer_form(o):
    """sum_b d_w(b) d_a(b) sum_j (q_j - 8) qs_j from the quant bytes with
    numpy integers equals the product to fp64 rounding."""
    g = synth.rng(23, (0,))
    M, N, K = 4, 24, 512
    A = (g.standard_normal((M, K)) * np.exp(g.uniform(-3, 3, (M, 1)))).astype(np.float32)
    blob = synth.q4_0_weights(N, K, 24)
    C, S = o.matmul_q4_0_q8act(A, blob, N, K)
    nb = K // 32
    q8 = o.quantize_q8_0(A.ravel()).reshape(M, nb, 34)
    da = q8[:, :, 0:2].copy().view(np.float16).reshape(M, nb).astype(np.float64)
    qs = q8[:, :, 2:].view(np.int8).astype(np.int64)                       # [M, nb, 32]
    w = blob.reshape(N, nb, 18)
    dw = w[:, :, 0:2].copy().view(np.float16).reshape(N, nb).astype(np.float64)
    qb = w[:, :, 2:].astype(np.int64)
    qw = np.concatenate([qb & 0xF, qb >> 4], axis=2) - 8                     # [N, nb, 32]
    isum = np.einsum("mbj,nbj->mnb", qs, qw)                                  # exact integers
    want = np.einsum("mnb,mb,nb->mn", isum.astype(np.float64), da, dw)
    assert np.all(np.abs(C - want) <= 1e-12 * S + 1e-300), "block-factored integer form differs"


def pin_q8act_bound_against_plain(o):
    """|C' - C| <= sum_k |a_k - a'_k| |W_k|, with |a - a'| at most half a
    quantization step plus the binary16 narrowing of the scale."""
    g = synth.rng(25, (0,))
    M, N, K = 2, 32, 1024
    A = g.standard_normal((M, K)).astype(np.float32)
    blob = synth.q4_0_weights(N, K, 26)
    C1, _ = o.matmul_q4_0_q8act(A, blob, N, K)
    C0, _ = o.matmul_q4_0(A, blob, N, K)
    W = o.dequant_q4_0(blob).reshape(N, K).astype(np.float64)
    amax = np.abs(A.astype(np.float64)).reshape(M, K // 32, 32).max(axis=2)
    step = np.repeat(amax / 127.0, 32, axis=1)                                # d per element
    da = step * (0.5 + 127 * 2.0**-11) * (1 + 1e-6)
    bound = da @ np.abs(W).T
    assert np.all(np.abs(C1 - C0) <= bound), "quantized product strays past the quantization bound"


ALL_PINS = (pin_f16_exhaustive, pin_golden_blocks, pin_all8_and_zero_scale,
            pin_extreme_nibbles, pin_golden_matmul, pin_one_hot,
            pin_ones_closed_form, pin_dense_equivalence, pin_rows_independent,
            pin_block_permutation, pin_entries_match_full,
            pin_f16_narrowing_vs_numpy, pin_q8_0_golden_blocks, pin_q8_0_dequant_numpy,
            pin_q8_0_golden_quantize, pin_q8_0_roundtrip_bound, pin_q8_0_symmetry_and_scaling,
            pin_q8act_golden, pin_q8act_identity_on_representable, pin_q8act_integer_form,
            pin_q8act_bound_against_plain)
