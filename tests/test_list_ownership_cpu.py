"""Host-side check of the list GEMV's fragment ownership (no GPU).

The list kernel's consumer warps take the CTA's unit sequence of a problem
16 units at a time: warp w takes position s0 + w of every stage (s0 = 0, 16,
32, ...), which is unit (s0 + w) mod U of tile (s0 + w) div U, U = K / 256.
Warp w converts units w, w + 16, w + 32, ... < U of new activations.  The
kernel then synchronises a warp only with its partner (w xor 8), or with
nobody when U is a multiple of 16.  That is safe exactly when

* every unit a warp reads is converted by itself or its partner (any U that
  is a multiple of 8, any number of tiles), and
* for U a multiple of 16, every unit a warp reads is converted by itself.

This test replays that index arithmetic for every K the kernel takes (2048
.. 14336 in steps of 2048) and 1..9 tiles per CTA, and plants the
arithmetic's two likely slips (a stage of 8 units, conversion by unit % 8)
to show that the check catches them.
"""
import pytest

WARPS = 16
KS = list(range(2048, 14336 + 1, 2048))


def reads(U, n, stage=WARPS):
    """Units each warp reads over n tiles (positions s0 + w, s0 += stage)."""
    out = {w: set() for w in range(WARPS)}
    total = n * U
    for s0 in range(0, total, stage):
        for w in range(WARPS):
            i = s0 + w
            if w < stage and i < total:
                out[w].add(i % U)
    return out


def converts(U, by_mod=WARPS):
    out = {w: set() for w in range(WARPS)}
    for u in range(U):
        out[u % by_mod].add(u)
    return out


def ownership_ok(U, n, stage=WARPS, by_mod=WARPS):
    r, c = reads(U, n, stage), converts(U, by_mod)
    own = U % 16 == 0
    for w in range(WARPS):
        mine = c[w] if own else c[w] | c[w ^ 8]
        if not r[w] <= mine:
            return False
    return True


@pytest.mark.parametrize("K", KS)
def test_every_unit_read_is_converted_by_the_warp_or_its_partner(K):
    U = K // 256
    assert U % 8 == 0
    for n in range(1, 10):
        assert ownership_ok(U, n), (K, n)


@pytest.mark.parametrize("K", KS)
def test_every_unit_is_converted_once(K):
    U = K // 256
    c = converts(U)
    units = sorted(u for w in range(WARPS) for u in c[w])
    assert units == list(range(U))


def test_shapes_with_u_a_multiple_of_16_need_no_partner():
    for K in KS:
        U = K // 256
        if U % 16:
            continue
        r, c = reads(U, 5), converts(U)
        assert all(r[w] == c[w] for w in range(WARPS)), K


def test_planted_slips_are_caught():
    # A stage of 8 units (warps 8..15 idle) breaks the mod-16 ownership that
    # a 16-unit problem relies on.
    assert not all(ownership_ok(K // 256, n, stage=8) for K in KS for n in range(1, 6))
    # Converting by unit % 8 assigns units w + 8 to warp w: warp w + 8 of a
    # 16-unit problem (no partner barrier) then reads a unit it did not write.
    assert not ownership_ok(16, 3, by_mod=8)
