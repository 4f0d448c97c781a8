"""The exactness arguments of the GPU kernels' arithmetic, checked by brute
force on the host (numpy emulation of IEEE round-to-nearest-even; no kernel
code and no oracle involved).

* Nibble decode, bf16 form (GEMV tensor-core consumer): the bf16 with bits
  0x43 << 8 | q is 128 + q, and subtracting 136 leaves q - 8 exactly.
* Nibble decode, f32 form (packed GEMV consumer, GEMM decode): the f32 with
  bits 0x43000000 | q << 16 is 128 + q, and one fused multiply-add
  x * d - f32(136 d) gives (q - 8) * d exactly, for every finite binary16 d.
* Weight split (GEMM): every (q - 8) * d with a finite binary16 d equals
  bf16(W) + bf16(W - bf16(W)) exactly.
* Activation split (GEMV and GEMM): |a - hi - lo| <= 2^-17 |a| for normal f32
  a, with hi = bf16(a), lo = bf16(a - hi).  The GEMV keeps both pieces against
  the exact (q - 8), so 2^-17 is its whole per-product error.
* GEMM products: the GEMM takes all four bf16 piece products (hi W_hi +
  hi W_lo + lo W_hi + lo W_lo), which miss a * W by the activation residual
  alone, at most 2^-17 |a W|.  Three products (dropping lo W_lo, up to 2^-16
  |a W|) would miss by up to (2^-16 + 2^-17) |a W|, more than the 1e-5
  tolerance, and that bound is nearly reached.
* Accumulation: on a constant input (every product the same, so every
  rounding error has the same sign) f32 sums over K = 4096 miss the 1e-5
  relative tolerance whichever way they are formed, including the plain
  sequential FMA chain; the tolerance holds for inputs whose rounding errors
  do not line up, such as the random workloads the parity tests use.
"""
import numpy as np

Q = np.arange(16)


def bf16_rne(x):
    """f32 -> bf16 (round to nearest even), returned as f32.  Finite inputs."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return r.astype(np.uint32).view(np.float32)


def finite_f16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    h = bits.view(np.float16)
    return h[np.isfinite(h)].astype(np.float64)


def test_bf16_rne_helper():
    # Ties go to even, halfway above a mantissa step rounds up, exact values stay.
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -8 + 2 ** -20, -2.5],
                 dtype=np.float32)
    want = np.array([1.0, 1.0, 1.0 + 2 ** -6, 1.0 + 2 ** -7, -2.5], dtype=np.float32)
    assert np.array_equal(bf16_rne(x), want)


def test_bf16_nibble_decode():
    v = ((0x4300 | Q).astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(v, 128.0 + Q)
    # 128 + q - 136 in bf16 arithmetic: exact small integers.
    assert np.array_equal(bf16_rne(v - np.float32(136)), (Q - 8).astype(np.float32))


def test_f32_nibble_decode_fma_is_exact_for_every_scale():
    v = (np.uint32(0x43000000) | (Q.astype(np.uint32) << 16)).view(np.float32)
    assert np.array_equal(v, 128.0 + Q)
    d = finite_f16()
    bias = (np.float32(-136.0) * d.astype(np.float32)).astype(np.float64)  # f32 product
    assert np.array_equal(bias, -136.0 * d), "136 d is exact in f32"
    exact = v.astype(np.float64)[None, :] * d[:, None] + bias[:, None]     # the FMA before rounding
    want = (Q - 8)[None, :] * d[:, None]
    assert np.array_equal(exact, want)
    # One rounding to f32 leaves it unchanged: (q - 8) d is representable.
    assert np.array_equal(exact.astype(np.float32).astype(np.float64), want)


def test_weight_splits_exactly_into_two_bf16():
    d = finite_f16().astype(np.float32)
    W = ((Q - 8).astype(np.float32)[None, :] * d[:, None]).ravel()
    hi = bf16_rne(W)
    rest = (W.astype(np.float64) - hi.astype(np.float64))
    assert np.array_equal(rest.astype(np.float32).astype(np.float64), rest), "W - hi exact in f32"
    lo = bf16_rne(rest.astype(np.float32))
    assert np.array_equal(hi.astype(np.float64) + lo.astype(np.float64), W.astype(np.float64))


def test_activation_split_bound():
    g = np.random.default_rng(0)
    mant = g.integers(0, 1 << 23, 400_000, dtype=np.uint32)
    expo = g.integers(1, 255, 400_000, dtype=np.uint32)
    sign = g.integers(0, 2, 400_000, dtype=np.uint32)
    a = ((sign << 31) | (expo << 23) | mant).view(np.float32)
    # Add the values next to bf16 rounding boundaries of a few binades.
    edges = []
    for e in (-100, -10, 0, 10, 100):
        base = np.float32(2.0 ** e)
        step = np.float32(2.0 ** (e - 8))
        for k in range(1, 256):
            t = np.float32(base + k * step)
            edges += [t, np.nextafter(t, np.float32(np.inf)), np.nextafter(t, np.float32(-np.inf))]
    a = np.concatenate([a, np.array(edges, dtype=np.float32)])
    a = a[np.isfinite(a) & (np.abs(a) >= np.float32(2.0 ** -100)) & (np.abs(a) < np.float32(2.0 ** 126))]
    hi = bf16_rne(a)
    rest = (a.astype(np.float64) - hi.astype(np.float64)).astype(np.float32)
    assert np.array_equal(rest.astype(np.float64), a.astype(np.float64) - hi.astype(np.float64))
    lo = bf16_rne(rest)
    err = np.abs(a.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
    assert (err <= 2.0 ** -17 * np.abs(a.astype(np.float64))).all()


def gemm_kept(a, W):
    """Three of the four piece products (lo W_lo dropped), for activation a and weight W."""
    hi = bf16_rne(a).astype(np.float64)
    lo = bf16_rne((np.float64(a) - hi).astype(np.float32)).astype(np.float64)
    W_hi = bf16_rne(W).astype(np.float64)
    W_lo = bf16_rne((np.float64(W) - W_hi).astype(np.float32)).astype(np.float64)
    return hi * W_hi + hi * W_lo + lo * W_hi


def test_gemm_three_product_bound():
    g = np.random.default_rng(1)
    a = g.standard_normal(200_000).astype(np.float32) * np.float32(3.0)
    d = g.choice(finite_f16()[finite_f16() > 0], 200_000).astype(np.float32)
    W = (g.integers(0, 16, 200_000) - 8).astype(np.float32) * d
    keep = (a != 0) & (W != 0)
    a, W = a[keep], W[keep]
    exact = a.astype(np.float64) * W.astype(np.float64)
    err = np.abs(gemm_kept(a, W) - exact)
    bound = (2.0 ** -16 + 2.0 ** -17) * np.abs(exact)
    assert (err <= bound).all()
    # Nearly reached: a just below the bf16 midpoint above 1, and d likewise.
    a1 = np.float32(1 + 2 ** -8 - 2 ** -23)
    W1 = np.float32(np.float16(1.0029296875))      # q = 9
    e1 = abs(gemm_kept(a1, W1) - np.float64(a1) * np.float64(W1)) / (np.float64(a1) * np.float64(W1))
    assert 1.1e-5 < e1 <= 2.0 ** -16 + 2.0 ** -17


def gemm_four(a, W):
    """The four products the GEMM takes for activation a and weight W."""
    hi = bf16_rne(a).astype(np.float64)
    lo = bf16_rne((np.float64(a) - hi).astype(np.float32)).astype(np.float64)
    W_hi = bf16_rne(W).astype(np.float64)
    W_lo = bf16_rne((np.float64(W) - W_hi).astype(np.float32)).astype(np.float64)
    return hi * W_hi + hi * W_lo + lo * W_hi + lo * W_lo


def test_gemm_four_product_bound():
    g = np.random.default_rng(2)
    a = g.standard_normal(200_000).astype(np.float32) * np.float32(3.0)
    d = g.choice(finite_f16()[finite_f16() > 0], 200_000).astype(np.float32)
    W = (g.integers(0, 16, 200_000) - 8).astype(np.float32) * d
    keep = (a != 0) & (W != 0)
    a, W = a[keep], W[keep]
    exact = a.astype(np.float64) * W.astype(np.float64)
    assert (np.abs(gemm_four(a, W) - exact) <= 2.0 ** -17 * np.abs(exact)).all()
    # The input that defeats three products is exact to 2^-23 with four.
    a1 = np.float32(1 + 2 ** -8 - 2 ** -23)
    W1 = np.float32(np.float16(1.0029296875))
    p1 = np.float64(a1) * np.float64(W1)
    assert abs(gemm_four(a1, W1) - p1) / p1 <= 2.0 ** -22


def test_constant_inputs_defeat_any_f32_sum():
    # Every product alike: the sequential f32 FMA chain, and the GEMM's
    # 16-wide MMA steps with three products, both miss the tolerance at
    # K = 4096; four products with the small ones summed apart do not.
    K = 4096
    a = np.float32(1 + 2 ** -8 - 2 ** -23)
    W = np.float32(np.float16(1.0029296875))
    exact = K * np.float64(a) * np.float64(W)
    tol = 1e-5 * abs(exact) + 1e-7
    s = np.float32(0)
    for _ in range(K):
        s = np.float32(np.float64(s) + np.float64(a) * np.float64(W))  # one rounding per FMA
    assert abs(np.float64(s) - exact) > tol
    hi = bf16_rne(a).astype(np.float64)
    lo = bf16_rne(np.float32(np.float64(a) - hi)).astype(np.float64)
    W_hi = bf16_rne(W).astype(np.float64)
    W_lo = bf16_rne(np.float32(np.float64(W) - W_hi)).astype(np.float64)
    D3 = np.float32(0)
    for _ in range(K // 16):
        for t in (hi * W_hi, hi * W_lo, lo * W_hi):
            D3 = np.float32(np.float64(D3) + 16 * t)   # a 16-wide MMA adds its exact dot once
    assert abs(np.float64(D3) - exact) > tol
    Dm, Ds = np.float32(0), np.float32(0)
    for _ in range(K // 16):
        Dm = np.float32(np.float64(Dm) + 16 * hi * W_hi)
        for t in (hi * W_lo, lo * W_hi, lo * W_lo):
            Ds = np.float32(np.float64(Ds) + 16 * t)
    assert abs(np.float64(np.float32(np.float64(Dm) + np.float64(Ds))) - exact) < 0.05 * tol
