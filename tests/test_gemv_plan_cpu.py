"""The decode GEMV's launch planner, checked on the host (qm_gemv_plan).

The planner chooses the stage shape (rps row groups x c units, hs warps per
tile), the K split S and the ring depth for one CTA per SM.  Whatever it
chooses, the kernel must visit every (row group, unit) of the matrix exactly
once, each half of a unit once, stay inside the opt-in shared memory and keep
TMA boxes at most 256 rows high.  A split K adds up through thread-block
clusters on the regular path: S is then 2, 4 or 8, a cluster is S consecutive
CTAs of one row-block range, and all of the launch's clusters are resident at
once; on the allocation-free path the split partial sums fit its fixed
scratch array.  This test replays the kernel's work assignment for the
returned plans in numpy and checks all of that, for a GB300 (152 SMs, 227 KB)
and for smaller devices.
"""
import numpy as np
import pytest

import bit_block_quantized_qm_gb300 as qm

UNIT = 256
NOALLOC_PART_FLOATS, NOALLOC_COUNTERS = 262144, 4096
FIT = {152: (76, 36, 18), 132: (66, 32, 16), 48: (24, 12, 6)}  # resident clusters of 2, 4, 8


def check_split(plan, M, rows, sm_count, noalloc):
    S = plan["S"]
    if S == 1:
        assert plan["cl"] == 0
        return
    if noalloc:
        assert plan["cl"] == 0
        assert plan["RG"] * S * M * rows <= NOALLOC_PART_FLOATS and plan["RG"] <= NOALLOC_COUNTERS
    else:
        assert plan["cl"] == 1 and S in (2, 4, 8)
        assert plan["grid"] // S <= FIT[sm_count][{2: 0, 4: 1, 8: 2}[S]], "every cluster resident"


@pytest.fixture(scope="module")
def lib():
    from bit_block_quantized_qm_gb300 import build as qm_build
    qm_build.build()
    return qm.load_library()


def covered(plan, packed):
    """How often the kernel visits each (row group, unit, half) under `plan`."""
    RG, U, S, rps, c, hs = (plan[k] for k in ("RG", "U", "S", "rps", "c", "hs"))
    rbpc, grid, W = plan["rbpc"], plan["grid"], plan["W"]
    RB = -(-RG // rps)
    count = np.zeros((RG, U, 2), dtype=np.int64)
    w = np.arange(W)
    h, rgl, ul = w % hs, (w // hs) % rps, w // (hs * rps)
    for b in range(grid):
        split = b % S
        u0 = split * U // S
        nu = (split + 1) * U // S - u0
        rb0 = (b // S) * rbpc
        nrb = max(0, min(rbpc, RB - rb0))
        spr = -(-nu // c)
        rbi, sc, ww = np.meshgrid(np.arange(nrb), np.arange(spr), w, indexing="ij")
        j = sc * c + ul[ww]
        rg = (rb0 + rbi) * rps + rgl[ww]
        ok = (j < nu) & (rg < RG)
        rg, j, hh = rg[ok], j[ok], h[ww][ok]
        if hs == 1:
            np.add.at(count, (rg, u0 + j, 0), 1)
            np.add.at(count, (rg, u0 + j, 1), 1)
        else:
            np.add.at(count, (rg, u0 + j, hh), 1)
    return count


SHAPES = [(1, 4096, 4096), (1, 14336, 4096), (1, 4096, 14336), (1, 1024, 4096), (1, 28672, 4096),
          (1, 80000, 256), (1, 1, 256), (1, 16, 256), (1, 33, 768), (1, 300, 3840), (2, 1000, 2048),
          (4, 4096, 4096), (5, 257, 768), (8, 4096, 4096), (8, 14336, 4096), (8, 4096, 14336),
          (8, 1000, 2048), (3, 64, 14336), (7, 6144, 4096)]
DEVICES = [(152, 232448), (132, 232448), (48, 101376)]


@pytest.mark.parametrize("noalloc", [False, True], ids=["regular", "noalloc"])
@pytest.mark.parametrize("dev", DEVICES, ids=lambda d: f"{d[0]}sm")
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("packed", [False, True], ids=["mma", "packed"])
def test_plan_invariants(lib, shape, packed, dev, noalloc):
    M, N, K = shape
    if packed and M > 2:
        pytest.skip("the packed consumer serves M = 1..2")
    sm_count, smem_optin = dev
    plan = qm.qm_gemv_plan(M, N, K, packed, sm_count, smem_optin, FIT[sm_count], noalloc)
    if plan is None:
        return  # no plan fits: the library runs the generic GEMV instead
    rows = 32 if packed else 16
    assert plan["RG"] == -(-N // rows) and plan["U"] == K // UNIT
    assert plan["W"] == plan["rps"] * plan["c"] * plan["hs"]
    assert 8 <= plan["W"] <= (24 if packed else 16)
    assert plan["hs"] == (2 if packed else 1)
    assert plan["rps"] * rows <= 256, "TMA box height"
    assert plan["smem"] <= smem_optin
    assert plan["stages"] >= 2
    assert plan["grid"] % plan["S"] == 0 and plan["grid"] <= sm_count
    assert plan["nu_max"] == -(-plan["U"] // plan["S"])
    check_split(plan, M, rows, sm_count, noalloc)
    count = covered(plan, packed)
    assert count.min() == 1 and count.max() == 1, "every (row group, unit, half) exactly once"


def test_plan_rejects_bad_arguments(lib):
    with pytest.raises(qm.QMError):
        qm.qm_gemv_plan(9, 4096, 4096)
    with pytest.raises(qm.QMError):
        qm.qm_gemv_plan(3, 4096, 4096, packed=True)
    with pytest.raises(qm.QMError):
        qm.qm_gemv_plan(1, 4096, 4000)
    with pytest.raises(qm.QMError):
        qm.qm_gemv_plan(1, 0, 4096)


@pytest.mark.parametrize("dev", DEVICES, ids=lambda d: f"{d[0]}sm")
def test_plan_invariants_random_shapes(lib, dev):
    # Seeded random shapes over M = 1..8, ragged N up to 60000 and K up to
    # 32768, both consumers.
    sm_count, smem_optin = dev
    g = np.random.default_rng(7 + sm_count)
    for _ in range(40):
        M = int(g.integers(1, 9))
        N = int(g.choice([int(g.integers(1, 700)), int(g.integers(700, 60000))]))
        K = 256 * int(g.integers(1, 129))
        for packed, noalloc in ((False, False), (True, False), (False, True)) if M <= 2 else ((False, False), (False, True)):
            plan = qm.qm_gemv_plan(M, N, K, packed, sm_count, smem_optin, FIT[sm_count], noalloc)
            if plan is None:
                continue
            rows = 32 if packed else 16
            assert plan["RG"] == -(-N // rows) and plan["U"] == K // UNIT
            assert plan["W"] == plan["rps"] * plan["c"] * plan["hs"]
            assert plan["rps"] * rows <= 256 and plan["smem"] <= smem_optin
            assert plan["grid"] % plan["S"] == 0 and plan["grid"] <= sm_count
            check_split(plan, M, rows, sm_count, noalloc)
            count = covered(plan, packed)
            assert count.min() == 1 and count.max() == 1, (M, N, K, packed, plan)


def test_cluster_split_follows_resident_clusters(lib):
    # 1 x 1024 x 4096 has 64 row groups for 152 SMs: it splits K, through
    # clusters that fit; with no cluster resident it cannot split at all.
    plan = qm.qm_gemv_plan(1, 1024, 4096, fit=(76, 36, 18))
    assert plan["S"] > 1 and plan["cl"] == 1
    plan = qm.qm_gemv_plan(1, 1024, 4096, fit=(0, 0, 0))
    assert plan["S"] == 1 and plan["cl"] == 0
