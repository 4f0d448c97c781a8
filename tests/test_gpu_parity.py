"""GPU parity: libqm's CUDA kernels against the CPU oracle, through the C ABI.

* dequant: bit-exact (NaN matched by class), aligned and misaligned pointers,
  ragged block counts, special scales, and the full 14336 x 4096 weight;
* matmul: per element |C - C_oracle| <= 1e-5 * sum_k |A W| + 1e-7 over tail
  shapes that span several tiles and ragged edges, every algorithm, the
  GEMV's TMA/cluster path and its generic path, guard words around C,
  determinism, K = 0, non-finite scales, and the workload shapes at full size
  (exhaustively where the oracle is fast, otherwise on sampled entries).
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

REL, ABS = 1e-5, 1e-7
GUARD_BITS = 0x7FC0DEAD  # a NaN payload no kernel produces


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


def dev(x):
    return torch.from_numpy(np.array(x, copy=True)).cuda()


def dequant_gpu(qm, blob, in_off=0, out_off=0):
    """Dequant through the C ABI with the stream and output placed at byte
    offsets in larger buffers; guard words around the output are checked."""
    nb = blob.size // 18
    raw = torch.zeros(blob.size + 32, dtype=torch.uint8, device="cuda")
    raw[in_off:in_off + blob.size] = dev(blob)
    guard = 64
    out_buf = torch.full((nb * 32 + 2 * guard + 4,), 0, dtype=torch.int32, device="cuda")
    out_buf.fill_(GUARD_BITS)
    out_base = out_buf.data_ptr() + 4 * guard + out_off
    rc = qm.qm_dequant_q4_0_ptr(raw.data_ptr() + in_off, nb, out_base, 0)
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    torch.cuda.synchronize()
    host = out_buf.cpu().numpy().view(np.uint32)
    start = guard + out_off // 4
    assert np.all(host[:start] == GUARD_BITS), "write before the output"
    assert np.all(host[start + nb * 32:] == GUARD_BITS), "write past the output"
    assert np.array_equal(raw[in_off:in_off + blob.size].cpu().numpy(), blob), "input modified"
    return host[start:start + nb * 32].view(np.float32)


def assert_bits_equal(got, want):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    nan_w = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan_w), "NaN positions differ"
    bad = got.view(np.uint32)[~nan_w] != want.view(np.uint32)[~nan_w]
    assert not bad.any(), f"{bad.sum()} elements differ, first at {np.argwhere(bad)[:4].ravel()}"


def matmul_gpu(qm, A, blob, N, algo=0, a_off=0, w_off=0, c_off=0):
    """C through the C ABI with guard words around C; A and wq may sit at byte
    offsets (multiples of 4 and 2) inside larger buffers, and C c_off floats
    past a 16-byte boundary."""
    M, K = A.shape
    a_raw = torch.zeros(A.size * 4 + 64, dtype=torch.uint8, device="cuda")
    a_raw[a_off:a_off + A.size * 4] = dev(A.view(np.uint8).ravel())
    w_raw = torch.zeros(blob.size + 64, dtype=torch.uint8, device="cuda")
    w_raw[w_off:w_off + blob.size] = dev(blob)
    guard = 32 + c_off
    c_buf = torch.empty(M * N + 2 * guard, dtype=torch.int32, device="cuda")
    c_buf.fill_(GUARD_BITS)
    rc = qm.qm_matmul_q4_0_algo_ptr(a_raw.data_ptr() + a_off, w_raw.data_ptr() + w_off,
                                    c_buf.data_ptr() + 4 * guard, M, N, K, algo, 0)
    assert rc == qm.QM_OK, qm.qm_status_string(rc)
    torch.cuda.synchronize()
    assert qm.qm_device_status(clear=True) == qm.QM_OK
    host = c_buf.cpu().numpy().view(np.uint32)
    assert np.all(host[:guard] == GUARD_BITS) and np.all(host[guard + M * N:] == GUARD_BITS), \
        "write outside C"
    return host[guard:guard + M * N].view(np.float32).reshape(M, N)


def assert_close(C, C_ref, S_ref, what=""):
    ok = oracle.within_tolerance(C, C_ref, S_ref, REL, ABS)
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        detail = [(tuple(i), float(C[tuple(i)]), float(C_ref[tuple(i)]), float(S_ref[tuple(i)]))
                  for i in idx]
        raise AssertionError(f"{what}: {int((~ok).sum())} entries outside tolerance: {detail}")


# ---------------------------------------------------------------- dequant

def test_dequant_golden_blocks(env):
    qm, o = env
    from oracle_pins import load_golden_blocks
    blocks, values = load_golden_blocks()
    blob = np.frombuffer(b"".join(blocks), dtype=np.uint8)
    got = dequant_gpu(qm, blob)
    assert_bits_equal(got, np.concatenate(values))


@pytest.mark.parametrize("nb", [1, 7, 31, 32, 33, 255, 1000, 65537])
@pytest.mark.parametrize("offs", [(0, 0), (2, 0), (0, 4), (16, 16), (6, 12)])
def test_dequant_random_bitexact(env, nb, offs):
    qm, o = env
    blob = synth.q4_0_weights(1, 32 * nb, 100 + nb)
    got = dequant_gpu(qm, blob, in_off=offs[0], out_off=offs[1])
    assert_bits_equal(got, o.dequant_q4_0(blob))


def test_dequant_special_scales(env):
    qm, o = env
    specials = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x0400, 0x7BFF, 0xFBFF,
                         0x7C00, 0xFC00, 0x7E00, 0xFE01, 0x3C00, 0xBC00, 0x3555, 0x2E66],
                        dtype=np.uint16)
    g = synth.rng(5, (3,))
    d = np.concatenate([specials, g.integers(0, 65536, 4096 - specials.size).astype(np.uint16)])
    q = g.integers(0, 256, size=(d.size, 16), dtype=np.uint8)
    q[:16, :4] = 0x88  # q = 8 against every special scale: signed zeros / NaN
    blob = synth.assemble_blocks(d.view(np.float16), q)
    got = dequant_gpu(qm, blob)
    assert_bits_equal(got, o.dequant_q4_0(blob))


def test_dequant_full_weight_14336x4096(env):
    qm, o = env
    case = [c for c in synth.workload(1) if c.op == "dequant"][0]
    blob = case.weights()
    wq = dev(blob)
    out = qm.qm_dequant_q4_0(wq)
    torch.cuda.synchronize()
    assert_bits_equal(out.cpu().numpy(), o.dequant_q4_0(blob))


# ---------------------------------------------------------------- matmul

TAIL_SHAPES = [(M, N, K) for M in (1, 2, 3, 5, 8, 9, 16, 31, 32, 33, 65, 130)
               for (N, K) in ((1, 32), (7, 96), (31, 160), (33, 288), (257, 64), (130, 1024))]


@pytest.mark.parametrize("shape", TAIL_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_matmul_tail_shapes(env, shape):
    qm, o = env
    M, N, K = shape
    blob = synth.q4_0_weights(N, K, M * 7 + N)
    A = synth.activations(M, K, K + M, dist="outliers")
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    algos = [qm.QM_ALGO_AUTO, qm.QM_ALGO_GEMM_SIMT] + \
        ([qm.QM_ALGO_GEMV, qm.QM_ALGO_GEMV_SIMT] if M <= 8 else []) + \
        ([qm.QM_ALGO_GEMV_PK] if M <= 2 else [])
    for algo in algos:
        assert_close(matmul_gpu(qm, A, blob, N, algo), C_ref, S_ref, f"algo {algo}")


# GEMV TMA path: K % 256 == 0, aligned; N ragged against 32-row groups; K
# split into 2, 4 or 8 ranges (added up inside a thread-block cluster) or not
# at all; more row groups than fit one wave of CTAs.
GEMV_FAST = [(M, N, K) for M in (1, 2, 4, 7, 8)
             for (N, K) in ((1, 256), (31, 512), (33, 768), (100, 2048), (1000, 256),
                            (64, 14336), (4096, 512), (1024, 4096), (300, 3840))] + \
            [(1, 80000, 256), (3, 4096, 4096), (8, 4096, 4096), (1, 14336, 4096),
             (1, 4096, 14336), (2, 6144, 4096), (1, 28672, 4096)]


@pytest.mark.parametrize("shape", GEMV_FAST, ids=lambda s: "x".join(map(str, s)))
def test_gemv_tma_path(env, shape):
    qm, o = env
    M, N, K = shape
    blob = synth.q4_0_weights(N, K, 11 * M + N)
    A = synth.activations(M, K, 13 * M + K)
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMV), C_ref, S_ref, "tensor cores")
    assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMV_SIMT), C_ref, S_ref, "fp32 fma")
    if M <= 2:
        assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMV_PK), C_ref, S_ref, "packed fp32")


@pytest.mark.parametrize("offs", [(4, 0), (0, 2), (0, 18), (8, 8)])
def test_gemv_misaligned_takes_generic_path(env, offs):
    qm, o = env
    M, N, K = 4, 70, 512
    blob = synth.q4_0_weights(N, K, 31)
    A = synth.activations(M, K, 32)
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMV, a_off=offs[0], w_off=offs[1]),
                 C_ref, S_ref)
    assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMM_SIMT, a_off=offs[0], w_off=offs[1]),
                 C_ref, S_ref)


# Prefill GEMM on tcgen05 tensor cores: K % 256 == 0; M and N ragged against
# the 128 x 128 tiles; K up to 14336 (long accumulations in TMEM).  These
# shapes take the 128-column tiles.
GEMM_TC = [(9, 7, 256), (128, 128, 256), (130, 257, 512), (1, 300, 768), (200, 130, 1024),
           (64, 1000, 2048), (257, 129, 4096), (96, 64, 14336),
           (130, 10200, 1024)]  # 160 tiles: 152 whole, the last 8 split in 4 K ranges


@pytest.mark.parametrize("shape", GEMM_TC, ids=lambda s: "x".join(map(str, s)))
def test_gemm_tensor_cores(env, shape):
    qm, o = env
    M, N, K = shape
    blob = synth.q4_0_weights(N, K, 3 * M + N)
    A = synth.activations(M, K, 5 * M + K, dist="outliers")
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMM_TC), C_ref, S_ref, "tcgen05")


# 112-column tiles (the 128-column kernel with N = 112 MMAs) where they fill
# more SMs without a K split: 144 tiles of 130 x 8000 against 126 of 128
# columns; a ragged last tile, a misaligned C, and non-finite scales.
@pytest.mark.parametrize("c_off", [0, 1])
def test_gemm_tensor_cores_narrow_tiles(env, c_off):
    qm, o = env
    M, N, K = 130, 8000, 512
    assert qm.qm_gemm_plan(M, N, K)["BN"] == 112
    blob = synth.q4_0_weights(N, K, 41 + c_off).reshape(N, K // 32, 18).copy()
    blob[N - 1, 2, 0:2] = np.frombuffer(np.float16(np.inf).tobytes(), np.uint8)
    blob[115, 9, 0:2] = np.frombuffer(np.float16(np.nan).tobytes(), np.uint8)
    blob = blob.ravel()
    A = synth.activations(M, K, 43 + c_off, dist="outliers")
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMM_TC, c_off=c_off), C_ref, S_ref,
                 "tcgen05, 112-column tiles")


# Shapes that take the 256-column tiles (M >= 256 and either enough 128 x 256
# tiles to fill the GPU or K >= 8192): ragged M and N, a 16-way K split, a
# misaligned C, and non-finite scales in both the split and the unsplit path.
GEMM_WIDE = [(260, 300, 8192, 0), (300, 9800, 512, 0), (300, 9800, 512, 1)]


@pytest.mark.parametrize("shape", GEMM_WIDE, ids=lambda s: "x".join(map(str, s)))
def test_gemm_tensor_cores_wide_tiles(env, shape):
    qm, o = env
    M, N, K, c_off = shape
    blob = synth.q4_0_weights(N, K, 7 * M + N).reshape(N, K // 32, 18).copy()
    blob[N - 1, 3, 0:2] = np.frombuffer(np.float16(np.inf).tobytes(), np.uint8)
    blob[N // 2, K // 64, 0:2] = np.frombuffer(np.float16(np.nan).tobytes(), np.uint8)
    blob = blob.ravel()
    A = synth.activations(M, K, 11 * M + K, dist="outliers")
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMM_TC, c_off=c_off), C_ref, S_ref,
                 "tcgen05, 256-column tiles")


@pytest.mark.parametrize("shape", [(200, 130, 1024), (64, 1000, 2048), (130, 10200, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_cluster_split_nonfinite_scales(env, shape):
    # Tiles split over 4 or 8 K ranges whose sums meet through a thread-block
    # cluster (the last shape: after 152 whole tiles); non-finite scales in
    # rows of split tiles go through the element-by-element recomputation.
    qm, o = env
    M, N, K = shape
    blob = synth.q4_0_weights(N, K, 13 * M + N).reshape(N, K // 32, 18).copy()
    blob[N - 1, 1, 0:2] = np.frombuffer(np.float16(-np.inf).tobytes(), np.uint8)
    blob[N // 3, K // 64, 0:2] = np.frombuffer(np.float16(np.nan).tobytes(), np.uint8)
    blob = blob.ravel()
    A = synth.activations(M, K, 17 * M + K, dist="outliers")
    C = matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMM_TC)
    if M * N * K <= 1e9:
        C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
        assert_close(C, C_ref, S_ref, "tcgen05, cluster split")
        return
    g = synth.rng(80, (M, N, K))
    rows = np.array([0, M - 1])
    mi = np.concatenate([np.repeat(rows, N), g.integers(0, M, 1024)])
    ni = np.concatenate([np.tile(np.arange(N), rows.size), g.integers(0, N, 1024)])
    C_ref, S_ref = o.matmul_q4_0_entries(A, blob, N, K, mi, ni)
    assert_close(C[mi, ni], C_ref, S_ref, "tcgen05, cluster split (sampled)")


def test_gemm_tensor_cores_wide_tiles_last_wave_split(env):
    # 154 tiles of 128 x 256 on 152 SMs: 152 whole tiles, the last 2 split
    # into 128-column halves (one of them wholly past N = 19500).  Checked on
    # all columns of 3 rows (first, last, one of the split tiles' rows) and
    # 1024 random entries.
    qm, o = env
    M, N, K = 256, 19500, 512
    blob = synth.q4_0_weights(N, K, 77)
    A = synth.activations(M, K, 78, dist="outliers")
    C = matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMM_TC)
    g = synth.rng(79, (M, N, K))
    rows = np.array([0, 200, M - 1])
    mi = np.concatenate([np.repeat(rows, N), g.integers(0, M, 1024)])
    ni = np.concatenate([np.tile(np.arange(N), rows.size), g.integers(0, N, 1024)])
    C_ref, S_ref = o.matmul_q4_0_entries(A, blob, N, K, mi, ni)
    assert_close(C[mi, ni], C_ref, S_ref, "tcgen05, last wave split")


@pytest.mark.parametrize("c_off", [1, 2])
def test_gemm_tensor_cores_misaligned_c(env, c_off):
    # C off a 16-byte boundary (N % 4 == 0): the epilogue's row stores fall
    # back from 16-byte to 4-byte stores.
    qm, o = env
    M, N, K = 130, 256, 512
    blob = synth.q4_0_weights(N, K, 90 + c_off)
    A = synth.activations(M, K, 91 + c_off)
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    assert_close(matmul_gpu(qm, A, blob, N, qm.QM_ALGO_GEMM_TC, c_off=c_off), C_ref, S_ref,
                 "tcgen05, misaligned C")


def test_gemm_tensor_cores_unsupported_layouts(env):
    qm, o = env
    A = torch.zeros((16, 96), device="cuda")
    wq = torch.zeros(8 * 3 * 18, dtype=torch.uint8, device="cuda")
    C = torch.zeros((16, 8), device="cuda")
    rc = qm.qm_matmul_q4_0_algo_ptr(A.data_ptr(), wq.data_ptr(), C.data_ptr(), 16, 8, 96,
                                    qm.QM_ALGO_GEMM_TC, 0)
    assert rc == qm.QM_ERR_UNSUPPORTED  # K % 256 != 0


def test_deterministic_repeat(env):
    qm, o = env
    for (M, N, K) in ((1, 4096, 4096), (8, 1000, 14336), (64, 300, 2048), (300, 500, 4096)):
        blob = synth.q4_0_weights(N, K, 41)
        A = synth.activations(M, K, 42)
        C1 = matmul_gpu(qm, A, blob, N)
        C2 = matmul_gpu(qm, A, blob, N)
        assert np.array_equal(C1.view(np.uint32), C2.view(np.uint32))


def test_k_zero_gives_positive_zeros(env):
    qm, o = env
    C = torch.full((3, 5), 7.0, device="cuda")
    A = torch.empty((3, 0), device="cuda")
    wq = torch.empty(0, dtype=torch.uint8, device="cuda")
    qm.qm_matmul_q4_0(A, wq, 5, out=C)
    torch.cuda.synchronize()
    host = C.cpu().numpy()
    assert np.all(host == 0) and not np.signbit(host).any()


def test_nonfinite_scales(env):
    qm, o = env
    M, N, K = 3, 5, 256
    blob = synth.q4_0_weights(N, K, 51).reshape(N, K // 32, 18).copy()
    blob[1, 2, 0:2] = np.frombuffer(np.float16(np.inf).tobytes(), np.uint8)
    blob[3, 5, 0:2] = np.frombuffer(np.float16(np.nan).tobytes(), np.uint8)
    blob = blob.ravel()
    A = synth.activations(M, K, 52)
    C_ref, S_ref = o.matmul_q4_0(A, blob, N, K)
    for algo in (qm.QM_ALGO_GEMV, qm.QM_ALGO_GEMV_SIMT, qm.QM_ALGO_GEMM_SIMT, qm.QM_ALGO_GEMM_TC):
        assert_close(matmul_gpu(qm, A, blob, N, algo), C_ref, S_ref, f"algo {algo}")
    for m in (1, 2):
        C_ref, S_ref = o.matmul_q4_0(A[:m], blob, N, K)
        assert_close(matmul_gpu(qm, A[:m], blob, N, qm.QM_ALGO_GEMV_PK), C_ref, S_ref, "packed fp32")


def test_m1_matches_rows_of_m8(env):
    qm, o = env
    N, K = 512, 4096
    blob = synth.q4_0_weights(N, K, 61)
    A = synth.activations(8, K, 62)
    C8 = matmul_gpu(qm, A, blob, N)
    _, S8 = o.matmul_q4_0(A[[0, 5]], blob, N, K)
    for i, r in enumerate((0, 5)):
        C1 = matmul_gpu(qm, A[r:r + 1], blob, N)
        assert np.all(np.abs(C1[0].astype(np.float64) - C8[r]) <= 2 * (REL * S8[i] + ABS))


# ------------------------------------------------------- workload shapes

def _check_case(qm, o, case, full_limit=6e8, rows=4, pairs=512, blob=None):
    """The case through qm_matmul_q4_0 against the oracle: every entry when
    M*N*K <= full_limit, else `rows` random rows x every column plus `pairs`
    random entries (the oracle's OpenMP build, bit-identical to the plain one,
    takes the large samples)."""
    blob = case.weights() if blob is None else blob
    A = case.acts()
    wq = dev(blob)
    C = qm.qm_matmul_q4_0(dev(A), wq, case.N)
    torch.cuda.synchronize()
    C = C.cpu().numpy()
    if case.M * case.N * case.K <= full_limit:
        C_ref, S_ref = o.matmul_q4_0(A, blob, case.N, case.K)
        assert_close(C, C_ref, S_ref, case.name)
        return
    g = synth.rng(99, (case.M, case.N, case.K))
    r = g.choice(case.M, size=min(rows, case.M), replace=False)
    mi = np.concatenate([np.repeat(r, case.N), g.integers(0, case.M, pairs)])
    ni = np.concatenate([np.tile(np.arange(case.N), r.size), g.integers(0, case.N, pairs)])
    C_ref, S_ref = oracle.load_parallel().matmul_q4_0_entries(A, blob, case.N, case.K, mi, ni)
    assert_close(C[mi, ni], C_ref, S_ref, case.name + " (sampled)")


@pytest.mark.parametrize("index", [0, 1, 2, 3])
def test_workload_full_size(env, index):
    # Workloads 0-2 every entry; workload 3 (M = 1024) on 16 random rows x
    # every column plus 1024 random entries.
    qm, o = env
    for case in synth.workload(index):
        if case.op == "matmul":
            _check_case(qm, o, case, rows=16, pairs=1024)


def test_decoder_layer_shapes(env):
    # One layer of the 32-layer decoder sweep at each M (sampled checks).
    qm, o = env
    cases = [c for c in synth.workload(4, layers=1)]
    for case in cases:
        _check_case(qm, o, case, full_limit=1e8, rows=2, pairs=256)


def test_decoder_sweep_every_layer_m512(env):
    # Every layer of the 32-layer decoder sweep at M = 512 (the prefill GEMM on
    # tensor cores): 4 random rows x every column of each of the 7 projections.
    qm, o = env
    for case in synth.workload(4, layers=32, sweep_m=(512,)):
        _check_case(qm, o, case, full_limit=0, rows=4, pairs=0)
