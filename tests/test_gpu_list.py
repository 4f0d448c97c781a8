"""GPU parity of qm_gemv_q4_0_list (a list of GEMVs in one persistent launch)
against the oracle, through the C ABI.

* independent problems of mixed shapes (ragged N, K from 256 to 16384) in one
  list, every entry within |C - C_oracle| <= 1e-5 sum_k |A W| + 1e-7
  (the matmul sections of the quantized kernel-contract page), and bitwise the
  same on a second run;
* dependent problems: a decoder-shaped chain (q, k, v; o reads q's output
  after q, k, v; gate and up read o's; down reads up's), with weights that
  have one non-zero element per row, so that every output is exactly one
  earlier value (or its negative) and the chain is exact on both sides: any
  stale read of an activation shows up as a wrong entry.  Run with counters
  (one launch) and without (one launch per dependency), twice in a row;
* lists that the persistent kernel does not take (M = 2, K not a multiple of
  2048) run problem by problem and still match the oracle;
* a row with an infinite scale over all-8 nibbles comes out NaN, as the
  definition gives it;
* activation hand-overs: a list whose K alternates between sizes whose
  fragments each warp keeps alone and sizes whose fragments warp pairs
  share, with runs of K = 4096 problems (activations copied ahead), with
  distinct, shared and repeated activation vectors and problems too small
  to reach every CTA, both products, checked entry by entry;
* the 32-layer decoder sweep at M = 1 (224 GEMVs, every one with its own
  activation vector) through one call, sampled rows of every problem against
  the oracle;
* the act-quant list (qm_gemv_q4_0_q8act_list) against the oracle's
  composition dequant_q8_0(quantize_q8_0(A)) x dequant(W)^T: mixed shapes,
  the decoder chain (exact with one-hot weights), a non-finite scale and a
  shape that runs outside the persistent kernel.
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


def run_list(qm, problems, M, counters=None):
    """problems: (A tensor, wq tensor, C tensor, N, K, wait_for)."""
    s = int(torch.cuda.current_stream().cuda_stream)
    raw = [(A.data_ptr(), w.data_ptr(), C.data_ptr(), N, K, wf) for (A, w, C, N, K, wf) in problems]
    rc = qm.qm_gemv_q4_0_list_ptr(raw, M, counters.data_ptr() if counters is not None else 0, s)
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    torch.cuda.synchronize()
    assert qm.qm_device_status(clear=True) == qm.QM_OK


# (N, K): the persistent kernel takes K = 2048, 4096, 6144, 8192, 14336 (boxes of
# 8 or 16 units); the others run through the fallback path in list order.
MIXED = [(4096, 4096), (1024, 4096), (1000, 4096), (17, 256), (300, 14336), (64, 16384),
         (4096, 512), (1, 1024), (2049, 2304), (700, 2048), (96, 6144), (513, 8192)]


def test_list_independent_mixed_shapes(env):
    qm, o = env
    host, problems = [], []
    for i, (N, K) in enumerate(MIXED):
        blob = synth.q4_0_weights(N, K, 200 + i)
        A = synth.activations(1, K, 300 + i)
        host.append((A, blob))
        problems.append((torch.from_numpy(A).cuda(), torch.from_numpy(blob).cuda(),
                         torch.full((1, N), float("nan"), device="cuda"), N, K, -1))
    run_list(qm, problems, 1)
    first = [p[2].cpu().numpy() for p in problems]
    for (A, blob), (N, K), C in zip(host, MIXED, first):
        C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
        ok = oracle.within_tolerance(C, C_ref, S_ref, REL, ABS)
        assert ok.all(), f"N={N} K={K}: {int((~ok).sum())} entries outside tolerance"
    for p in problems:
        p[2].fill_(float("nan"))
    run_list(qm, problems, 1)
    for p, C in zip(problems, first):
        assert np.array_equal(p[2].cpu().numpy().view(np.uint32), C.view(np.uint32)), "not deterministic"


def one_hot_weights(N, K, seed):
    """A block stream with exactly one non-zero weight per row, +1 or -1
    (d = 1, nibble 9 or 7, every other nibble 8), at a random column; returns
    the stream and (column, sign) per row."""
    g = synth.rng(seed, (N, K))
    cols = g.integers(0, K, N)
    signs = np.where(g.integers(0, 2, N) == 1, 1, -1)
    q = np.full((N, K), 8, np.uint8)
    q[np.arange(N), cols] = np.where(signs > 0, 9, 7)
    nb = K // 32
    qb = q.reshape(N * nb, 32)
    quant = (qb[:, :16] | (qb[:, 16:] << 4)).astype(np.uint8)
    d = np.ones(N * nb, np.float16)
    return synth.assemble_blocks(d, quant)


# Decoder-shaped chain: (name, N, K, input, wait_for); input -1 is the
# external activation, else the index of the problem whose output it reads.
CHAIN = [("q", 4096, 4096, -1, -1), ("k", 1024, 4096, -1, -1), ("v", 1024, 4096, -1, -1),
         ("o", 4096, 4096, 0, 2), ("gate", 14336, 4096, 3, 3), ("up", 14336, 4096, 3, 3),
         ("down", 4096, 14336, 5, 5)]


@pytest.mark.parametrize("with_counters", [True, False], ids=["counters", "no_counters"])
def test_list_dependent_chain_exact(env, with_counters):
    qm, o = env
    g = synth.rng(401, (0,))
    x = g.integers(-1000, 1001, (1, 4096)).astype(np.float32)   # exact in bf16 hi + lo
    blobs = [one_hot_weights(N, K, 410 + i) for i, (_, N, K, _, _) in enumerate(CHAIN)]
    # The oracle runs the chain on its own outputs (exact integers here).
    ref = []
    for (name, N, K, src, _), blob in zip(CHAIN, blobs):
        A = x if src < 0 else ref[src].astype(np.float32).reshape(1, -1)
        C_ref, _ = o.matmul_q4_0(A, blob, N, K)
        ref.append(C_ref)
    xs = torch.from_numpy(x).cuda()
    outs = [torch.empty((1, N), device="cuda") for (_, N, _, _, _) in CHAIN]
    ws = [torch.from_numpy(b).cuda() for b in blobs]
    problems = []
    for i, (name, N, K, src, wf) in enumerate(CHAIN):
        A = xs if src < 0 else outs[src]
        problems.append((A, ws[i], outs[i], N, K, wf))
    counters = torch.full((len(CHAIN),), 12345, dtype=torch.int32, device="cuda") if with_counters else None
    for rep in range(2):
        for c in outs:
            c.fill_(float("nan"))
        run_list(qm, problems, 1, counters)
        for (name, N, K, _, _), C, C_ref in zip(CHAIN, outs, ref):
            got = C.cpu().numpy().ravel().astype(np.float64)
            bad = got != C_ref.ravel()
            assert not bad.any(), f"run {rep} {name}: {int(bad.sum())} entries differ (stale input?)"


@pytest.mark.parametrize("M,K", [(2, 4096), (1, 4000 // 32 * 32)])
def test_list_fallback_problem_by_problem(env, M, K):
    qm, o = env
    shapes = [(300, K), (64, K)]
    host, problems = [], []
    for i, (N, KK) in enumerate(shapes):
        blob = synth.q4_0_weights(N, KK, 500 + i)
        A = synth.activations(M, KK, 510 + i)
        host.append((A, blob))
        problems.append((torch.from_numpy(A).cuda(), torch.from_numpy(blob).cuda(),
                         torch.full((M, N), float("nan"), device="cuda"), N, KK, -1))
    run_list(qm, problems, M)
    for (A, blob), (N, KK), p in zip(host, shapes, problems):
        C_ref, S_ref = o.matmul_q4_0(A, blob, N, KK)
        assert oracle.within_tolerance(p[2].cpu().numpy(), C_ref, S_ref, REL, ABS).all()


def test_list_nonfinite_scale_row_recomputed(env):
    qm, o = env
    N, K = 40, 2048                    # a shape the persistent kernel takes
    blob = synth.q4_0_weights(N, K, 520).copy()
    # Row 3, block 1: d = +inf with every nibble 8: that row's entries are NaN
    # by the definition (inf * 0), which block-scaled sums would miss.
    off = (3 * (K // 32) + 1) * 18
    blob[off:off + 2] = np.frombuffer(np.float16(np.inf).tobytes(), np.uint8)
    blob[off + 2:off + 18] = 0x88
    A = synth.activations(1, K, 521)
    C = torch.full((1, N), 0.0, device="cuda")
    run_list(qm, [(torch.from_numpy(A).cuda(), torch.from_numpy(blob).cuda(), C, N, K, -1)], 1)
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    got = C.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(C_ref)) and np.isnan(got[0, 3])
    fin = np.isfinite(C_ref)
    assert oracle.within_tolerance(got[fin], C_ref[fin], S_ref[fin], REL, ABS).all()


# --------------------------------------------------- the act-quant list
# qm_gemv_q4_0_q8act_list: every problem is dequant_q8_0(quantize_q8_0(A)) x
# dequant(W)^T, checked against the oracle's composition.

def run_q8_list(qm, problems, M, counters=None):
    s = int(torch.cuda.current_stream().cuda_stream)
    raw = [(A.data_ptr(), w.data_ptr(), C.data_ptr(), N, K, wf) for (A, w, C, N, K, wf) in problems]
    rc = qm.qm_gemv_q4_0_q8act_list_ptr(raw, M, counters.data_ptr() if counters is not None else 0, s)
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    torch.cuda.synchronize()
    assert qm.qm_device_status(clear=True) == qm.QM_OK


def test_q8act_list_independent_mixed_shapes(env):
    qm, o = env
    host, problems = [], []
    for i, (N, K) in enumerate(MIXED):
        blob = synth.q4_0_weights(N, K, 700 + i)
        A = synth.activations(1, K, 710 + i)
        host.append((A, blob))
        problems.append((torch.from_numpy(A).cuda(), torch.from_numpy(blob).cuda(),
                         torch.full((1, N), float("nan"), device="cuda"), N, K, -1))
    run_q8_list(qm, problems, 1)
    first = [p[2].cpu().numpy() for p in problems]
    for (A, blob), (N, K), C in zip(host, MIXED, first):
        C_ref, S_ref = o.matmul_q4_0_q8act(A, blob, N, K)
        ok = oracle.within_tolerance(C, C_ref, S_ref, REL, ABS)
        assert ok.all(), f"N={N} K={K}: {int((~ok).sum())} entries outside tolerance"
    for p in problems:
        p[2].fill_(float("nan"))
    run_q8_list(qm, problems, 1)
    for p, C in zip(problems, first):
        assert np.array_equal(p[2].cpu().numpy().view(np.uint32), C.view(np.uint32)), "not deterministic"


@pytest.mark.parametrize("with_counters", [True, False], ids=["counters", "no_counters"])
def test_q8act_list_dependent_chain_exact(env, with_counters):
    # One-hot weights with d = 1: every output is one quantized activation,
    # qs * d_a exactly, on both sides, so the chain is exact.
    qm, o = env
    g = synth.rng(720, (0,))
    x = g.integers(-1000, 1001, (1, 4096)).astype(np.float32)
    blobs = [one_hot_weights(N, K, 730 + i) for i, (_, N, K, _, _) in enumerate(CHAIN)]
    ref = []
    for (name, N, K, src, _), blob in zip(CHAIN, blobs):
        A = x if src < 0 else ref[src].astype(np.float32).reshape(1, -1)
        C_ref, _ = o.matmul_q4_0_q8act(A, blob, N, K)
        ref.append(C_ref)
    xs = torch.from_numpy(x).cuda()
    outs = [torch.empty((1, N), device="cuda") for (_, N, _, _, _) in CHAIN]
    ws = [torch.from_numpy(b).cuda() for b in blobs]
    problems = []
    for i, (name, N, K, src, wf) in enumerate(CHAIN):
        A = xs if src < 0 else outs[src]
        problems.append((A, ws[i], outs[i], N, K, wf))
    counters = torch.full((len(CHAIN),), 777, dtype=torch.int32, device="cuda") if with_counters else None
    for rep in range(2):
        for c in outs:
            c.fill_(float("nan"))
        run_q8_list(qm, problems, 1, counters)
        for (name, N, K, _, _), C, C_ref in zip(CHAIN, outs, ref):
            got = C.cpu().numpy().ravel().astype(np.float64)
            bad = got != C_ref.ravel()
            assert not bad.any(), f"run {rep} {name}: {int(bad.sum())} entries differ"


def test_q8act_list_non_finite_and_fallback(env):
    qm, o = env
    # A shape the persistent kernel takes with an infinite weight scale, and
    # one it does not (K = 96: through qm_matmul_q4_0_q8act).
    shapes = [(40, 2048), (33, 96)]
    host, problems = [], []
    for i, (N, K) in enumerate(shapes):
        blob = synth.q4_0_weights(N, K, 740 + i).copy()
        if i == 0:
            off = (3 * (K // 32) + 1) * 18
            blob[off:off + 2] = np.frombuffer(np.float16(np.inf).tobytes(), np.uint8)
        A = synth.activations(1, K, 750 + i)
        host.append((A, blob))
        problems.append((torch.from_numpy(A).cuda(), torch.from_numpy(blob).cuda(),
                         torch.zeros((1, N), device="cuda"), N, K, -1))
    run_q8_list(qm, problems, 1)
    for (A, blob), (N, K), p in zip(host, shapes, problems):
        C_ref, S_ref = o.matmul_q4_0_q8act(A, blob, N, K)
        assert oracle.within_tolerance(p[2].cpu().numpy(), C_ref, S_ref, REL, ABS).all(), (N, K)
    assert not np.isfinite(o.matmul_q4_0_q8act(*host[0], *shapes[0])[0]).all()


# ------------------------------------------- activation hand-overs, sweep
# (N, K, activation id): ids name activation vectors; a repeated id reuses
# the same device vector.  K / 256 a multiple of 16 (each warp alone with its
# fragments) or not (warp pairs share them), runs of K = 4096 problems with
# new activations each (copied ahead into the other bank), K = 14336 after
# them and before them; N = 16 and 48 leave most CTAs without a tile.
HANDOVER = [(4096, 4096, 0), (512, 14336, 1), (2048, 14336, 2), (1024, 8192, 3),
            (16, 4096, 0), (4096, 2048, 4), (300, 14336, 5), (48, 6144, 6),
            (1024, 14336, 5), (4096, 4096, 7), (700, 8192, 8), (256, 14336, 9),
            (2048, 4096, 7), (4096, 4096, 10), (1024, 4096, 11), (16, 4096, 12),
            (4096, 4096, 13), (2048, 4096, 14), (512, 14336, 15), (4096, 4096, 16),
            (48, 4096, 17), (1000, 4096, 18)]


@pytest.mark.parametrize("q8act", [False, True], ids=["f32", "q8act"])
def test_list_activation_handovers(env, q8act):
    qm, o = env
    acts = {}
    for (N, K, a) in HANDOVER:
        if a not in acts:
            acts[a] = synth.activations(1, K, 800 + a)
    dacts = {a: torch.from_numpy(A).cuda() for a, A in acts.items()}
    blobs = [synth.q4_0_weights(N, K, 820 + i) for i, (N, K, _) in enumerate(HANDOVER)]
    outs = [torch.full((1, N), float("nan"), device="cuda") for (N, _, _) in HANDOVER]
    problems = [(dacts[a], torch.from_numpy(b).cuda(), C, N, K, -1)
                for (N, K, a), b, C in zip(HANDOVER, blobs, outs)]
    for rep in range(2):
        for C in outs:
            C.fill_(float("nan"))
        (run_q8_list if q8act else run_list)(qm, problems, 1)
        for i, ((N, K, a), blob, C) in enumerate(zip(HANDOVER, blobs, outs)):
            ref = o.matmul_q4_0_q8act if q8act else o.matmul_q4_0
            C_ref, S_ref = ref(acts[a], blob, N, K)
            ok = oracle.within_tolerance(C.cpu().numpy(), C_ref, S_ref, REL, ABS)
            assert ok.all(), f"run {rep} problem {i} (N={N} K={K}): {int((~ok).sum())} bad"


def test_list_decoder_sweep_one_call(env):
    """The 224 GEMVs of the 32-layer decoder sweep at M = 1 (hidden 4096,
    GQA), every one with its own activation vector, through one call of
    qm_gemv_q4_0_list; 24 sampled rows of every problem (the first, the last
    and 22 random ones) against the oracle, entry by entry."""
    qm, o = env
    cases = synth.workload(4, layers=32, sweep_m=(1,))
    acts = [c.acts() for c in cases]
    blobs = [c.weights() for c in cases]
    dev_w = [torch.from_numpy(b).cuda() for b in blobs]
    dev_a = [torch.from_numpy(A).cuda() for A in acts]
    outs = [torch.full((1, c.N), float("nan"), device="cuda") for c in cases]
    problems = [(A, w, C, c.N, c.K, -1) for A, w, C, c in zip(dev_a, dev_w, outs, cases)]
    run_list(qm, problems, 1)
    g = synth.rng(840, (0,))
    for c, A, blob, C in zip(cases, acts, blobs, outs):
        rows = np.unique(np.concatenate([[0, c.N - 1], g.integers(0, c.N, 22)]))
        got = C.cpu().numpy().ravel()[rows]
        C_ref, S_ref = o.matmul_q4_0_entries(A, blob, c.N, c.K, np.zeros_like(rows), rows)
        ok = oracle.within_tolerance(got, C_ref, S_ref, REL, ABS)
        assert ok.all(), f"{c.name}: rows {rows[~ok].tolist()} outside tolerance"
    del dev_w
