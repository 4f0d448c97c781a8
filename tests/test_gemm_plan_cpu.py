"""The prefill GEMM's work items, checked on the host (qm_gemm_plan).

For a GEMM of M x N x K the library picks a tile width (128 or 256 columns),
fills whole waves of CTAs with whole tiles and splits the tiles of the last,
partial wave: into two 128-column halves, or into s_rem = 2, 4 or 8 K ranges
whose sums meet through a thread-block cluster, when the split tiles' clusters
can all be resident at once (else the last wave stays whole).  This test
replays the kernel's decoding of its 1-D grid for the returned plans and checks
that every (tile, k-step, column half) is computed exactly once, that K ranges
are whole 256-wide units, that a cluster never straddles whole and split
tiles, and that nothing spills into a second wave that a split was meant to
avoid.
"""
import numpy as np
import pytest

import bit_block_quantized_qm_gb300 as qm


@pytest.fixture(scope="module")
def lib():
    from bit_block_quantized_qm_gb300 import build as qm_build
    qm_build.build()
    return qm.load_library()


def replay(plan, M, N, K):
    """Count visits of each (tile, k-step of 64, column half) by the grid."""
    bn, nt, tiles, n_full = plan["BN"], plan["nt"], plan["tiles"], plan["n_full"]
    s_rem, hw, items = plan["s_rem"], plan["hw"], plan["items"]
    ksteps = K // 64
    count = np.zeros((tiles, ksteps, 2), dtype=np.int64)
    for b in range(items):
        half_item = bn == 256 and hw and b >= n_full
        tile = b if b < n_full else n_full + (b - n_full) // (2 if hw else s_rem)
        split = 0 if (b < n_full or hw) else (b - n_full) % s_rem
        S = 1 if (b < n_full or hw) else s_rem
        kt = ksteps // S
        halves = [(b - n_full) & 1] if half_item else [0, 1]
        for hh in halves:
            count[tile, split * kt:(split + 1) * kt, hh] += 1
    return count


SHAPES = [(130, 8000, 512), (9, 7, 256), (32, 4096, 4096), (130, 257, 512), (200, 130, 1024), (256, 4096, 4096),
          (260, 300, 8192), (300, 9800, 512), (256, 19500, 512), (512, 1024, 4096),
          (512, 4096, 4096), (512, 14336, 4096), (512, 4096, 14336), (1024, 14336, 4096),
          (130, 10200, 1024), (4096, 4096, 256), (96, 64, 14336)]


@pytest.mark.parametrize("sm_count", [152, 132, 20])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_work_items_cover_every_tile_once(lib, shape, sm_count):
    M, N, K = shape
    plan = qm.qm_gemm_plan(M, N, K, sm_count)
    bn = plan["BN"]
    assert bn in (112, 128, 256)
    assert plan["nt"] == -(-N // bn) and plan["tiles"] == plan["nt"] * -(-M // 128)
    assert (K // 256) % plan["s_rem"] == 0, "K ranges are whole 256-wide units"
    assert not (plan["hw"] and plan["s_rem"] > 1)
    if plan["hw"]:
        assert bn == 256 and 2 * (plan["tiles"] - plan["n_full"]) <= sm_count
    if plan["s_rem"] > 1 or plan["hw"]:
        assert plan["tiles"] - plan["n_full"] == plan["tiles"] % sm_count
        assert plan["items"] - plan["n_full"] <= sm_count, "the split last wave fits the SMs"
    assert plan["cl"] == (plan["s_rem"] > 1)
    if plan["cl"]:
        assert plan["s_rem"] in (2, 4, 8) and plan["n_full"] % plan["s_rem"] == 0
        assert plan["tiles"] - plan["n_full"] <= {2: 76, 4: 38, 8: 19}[plan["s_rem"]]
    count = replay(plan, M, N, K)
    assert count.min() == 1 and count.max() == 1


def test_tile_widths(lib):
    # 130 x 8000: 126 tiles of 128 columns, 144 of 112, both without a K split.
    plan = qm.qm_gemm_plan(130, 8000, 512, 152)
    assert plan["BN"] == 112 and plan["tiles"] == 144 and plan["items"] == 144
    # M >= 256 with N >= 2048 takes 256-column tiles (512 x 4096: 64 tiles,
    # K split in two through clusters); 512 x 1024 splits K with 128 columns.
    plan = qm.qm_gemm_plan(512, 4096, 4096, 152)
    assert plan["BN"] == 256 and plan["s_rem"] == 2 and plan["items"] == 128
    assert qm.qm_gemm_plan(1024, 14336, 4096, 152)["BN"] == 256
    assert qm.qm_gemm_plan(512, 1024, 4096, 152)["BN"] == 128


def test_cluster_split_needs_resident_clusters(lib):
    # 32 tiles split 4 ways only when 32 clusters of 4 fit at once; else 2
    # ways when 32 clusters of 2 do; else not at all.
    plan = qm.qm_gemm_plan(512, 1024, 4096, 152, fit=(76, 38, 19))
    assert plan["s_rem"] == 4 and plan["cl"] == 1
    plan = qm.qm_gemm_plan(512, 1024, 4096, 152, fit=(76, 31, 19))
    assert plan["s_rem"] == 2 and plan["cl"] == 1
    plan = qm.qm_gemm_plan(512, 1024, 4096, 152, fit=(31, 15, 7))
    assert plan["s_rem"] == 1 and plan["cl"] == 0 and plan["items"] == plan["tiles"]


def test_plan_rejects_unsupported_shapes(lib):
    for args in ((1, 4096, 4000), (0, 4096, 4096), (1, 0, 4096)):
        with pytest.raises(qm.QMError):
            qm.qm_gemm_plan(*args)


def random_shapes(n, seed):
    g = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(g.choice([int(g.integers(9, 300)), int(g.integers(300, 4100))]))
        N = int(g.choice([int(g.integers(1, 600)), int(g.integers(600, 30000))]))
        K = 256 * int(g.integers(1, 65))
        out.append((M, N, K))
    return out


@pytest.mark.parametrize("sm_count", [152, 132, 20, 8])
def test_work_items_random_shapes(lib, sm_count):
    # Seeded random shapes: the same invariants as above, over ragged M and N,
    # K from 256 to 16384, and devices of several sizes.
    for (M, N, K) in random_shapes(40, 1000 + sm_count):
        plan = qm.qm_gemm_plan(M, N, K, sm_count)
        bn = plan["BN"]
        assert bn in (112, 128, 256), (M, N, K)
        assert plan["nt"] == -(-N // bn) and plan["tiles"] == plan["nt"] * -(-M // 128)
        assert (K // 256) % plan["s_rem"] == 0, (M, N, K)
        if plan["s_rem"] > 1 or plan["hw"]:
            assert plan["items"] - plan["n_full"] <= sm_count, (M, N, K)
        assert plan["cl"] == (plan["s_rem"] > 1)
        if plan["cl"]:
            assert plan["s_rem"] in (2, 4, 8) and plan["n_full"] % plan["s_rem"] == 0
        count = replay(plan, M, N, K)
        assert count.min() == 1 and count.max() == 1, (M, N, K, plan)
