"""GGML Q4_0 x f32 quantized matmul, Q4_0 dequant and Q8_0 dequant/quantize on
GB300 (sm_103a).

A thin Python binding over the C ABI of ``libqm.so`` (``include/qm.h``): it
only marshals arguments.  Every step of the computation runs in the library's
CUDA kernels; there is no host fallback, and calls fail loudly when the
library has not been built.  PyTorch supplies device memory and streams.

Entry points (same names as the C ABI):

* ``qm_dequant_q4_0(wq, out=None, stream=None)`` -> f32 tensor ``[n_blocks*32]``
* ``qm_dequant_q8_0(wq, out=None, stream=None)`` -> f32 tensor ``[n_blocks*32]``
* ``qm_quantize_q8_0(x, out=None, stream=None)`` -> uint8 tensor ``[n/32*34]``
* ``qm_matmul_q4_0(A, wq, N, out=None, stream=None)`` -> f32 tensor ``[M, N]``
* ``qm_matmul_q4_0_algo(A, wq, N, algo, out=None, stream=None)``
* ``qm_gemv_q4_0_list(problems, M, counters=None, stream=None)``: a list of
  GEMV problems ``(A, wq, C, N, wait_for)`` in one persistent launch
* ``qm_device_status(stream=None, clear=True)``, ``qm_status_string(code)``,
  ``qm_version()``

The ``*_ptr`` variants take raw device addresses (ints) instead of tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "QMError", "load_library", "library_path", "qm_version", "qm_status_string",
    "qm_dequant_q4_0", "qm_matmul_q4_0", "qm_matmul_q4_0_algo", "qm_device_status",
    "qm_launch_count",
    "qm_dequant_q4_0_ptr", "qm_matmul_q4_0_ptr", "qm_matmul_q4_0_algo_ptr",
    "qm_dequant_q8_0", "qm_quantize_q8_0", "qm_dequant_q8_0_ptr", "qm_quantize_q8_0_ptr",
    "QM_OK", "QM_ERR_NULL", "QM_ERR_SHAPE", "QM_ERR_ALIGN", "QM_ERR_ALIAS", "QM_ERR_CUDA",
    "QM_ERR_TIMEOUT", "QM_ERR_UNSUPPORTED", "QM_ERR_POINTER", "QM_ERR_TOO_LARGE",
    "qm_matmul_q4_0_noalloc_ptr", "qm_selftest_wait_timeout",
    "qm_matmul_q4_0_q8act", "qm_matmul_q4_0_q8act_ptr", "qm_gemv_q4_0_q8act_list_ptr",
    "QM_ALGO_AUTO", "QM_ALGO_GEMV", "QM_ALGO_GEMM_SIMT", "QM_ALGO_GEMV_SIMT", "QM_ALGO_GEMM_TC",
    "QM_ALGO_GEMV_PK", "qm_gemv_plan", "GEMV_PLAN_FIELDS", "qm_gemm_plan", "GEMM_PLAN_FIELDS",
    "EXPORTED_SYMBOLS", "QmGemvProblem", "qm_gemv_q4_0_list_ptr", "qm_gemv_q4_0_list",
    "gemv_problem_array",
]

QM_OK = 0
QM_ERR_NULL = -1
QM_ERR_SHAPE = -2
QM_ERR_ALIGN = -3
QM_ERR_ALIAS = -4
QM_ERR_CUDA = -5
QM_ERR_TIMEOUT = -6
QM_ERR_UNSUPPORTED = -7
QM_ERR_POINTER = -8
QM_ERR_TOO_LARGE = -9

QM_ALGO_AUTO = 0
QM_ALGO_GEMV = 1
QM_ALGO_GEMM_SIMT = 2
QM_ALGO_GEMV_SIMT = 3
QM_ALGO_GEMM_TC = 4
QM_ALGO_GEMV_PK = 5

BLOCK_BYTES = 18
BLOCK_ELEMS = 32
Q8_0_BLOCK_BYTES = 34

# Every symbol include/qm.h declares.
EXPORTED_SYMBOLS = ("qm_version", "qm_status_string", "qm_dequant_q4_0", "qm_matmul_q4_0",
                    "qm_matmul_q4_0_algo", "qm_device_status", "qm_launch_count", "qm_gemv_plan", "qm_gemm_plan",
                    "qm_matmul_q4_0_noalloc", "qm_dequant_q8_0", "qm_quantize_q8_0",
                    "qm_selftest_wait_timeout", "qm_gemv_q4_0_list", "qm_matmul_q4_0_q8act",
                    "qm_gemv_q4_0_q8act_list")

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libqm.so")
_lock = threading.Lock()
_lib = None


class QmGemvProblem(ctypes.Structure):
    """One problem of qm_gemv_q4_0_list (the C struct qm_gemv_problem)."""
    _fields_ = [("A", ctypes.c_void_p), ("wq", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("wait_for", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class QMError(RuntimeError):
    """A negative status returned by libqm."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {qm_status_string(code)} (status {code})")


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libqm.so (built by ``bit_block_quantized_qm_gb300.build.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"libqm.so is not built ({_LIB_PATH}); run "
                    "`python -c 'import __graft_entry__ as g; g.build()'` first")
            lib = ctypes.CDLL(_LIB_PATH)
            i64, p, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            lib.qm_version.argtypes = []
            lib.qm_version.restype = i32
            lib.qm_status_string.argtypes = [i32]
            lib.qm_status_string.restype = ctypes.c_char_p
            lib.qm_dequant_q4_0.argtypes = [p, i64, p, p]
            lib.qm_dequant_q4_0.restype = i32
            lib.qm_matmul_q4_0.argtypes = [p, p, p, i64, i64, i64, p]
            lib.qm_matmul_q4_0.restype = i32
            lib.qm_matmul_q4_0_algo.argtypes = [p, p, p, i64, i64, i64, i32, p]
            lib.qm_matmul_q4_0_algo.restype = i32
            lib.qm_gemv_plan.argtypes = [i64, i64, i64, i32, i32, i32, i32, i32, i32, i32, p]
            lib.qm_gemv_plan.restype = i32
            lib.qm_gemm_plan.argtypes = [i64, i64, i64, i32, i32, i32, i32, p]
            lib.qm_gemm_plan.restype = i32
            lib.qm_device_status.argtypes = [p, i32]
            lib.qm_selftest_wait_timeout.argtypes = [p]
            lib.qm_selftest_wait_timeout.restype = i32
            lib.qm_device_status.restype = i32
            lib.qm_matmul_q4_0_noalloc.argtypes = [p, p, p, i64, i64, i64, p]
            lib.qm_matmul_q4_0_noalloc.restype = i32
            lib.qm_matmul_q4_0_q8act.argtypes = [p, p, p, i64, i64, i64, p]
            lib.qm_matmul_q4_0_q8act.restype = i32
            lib.qm_dequant_q8_0.argtypes = [p, i64, p, p]
            lib.qm_dequant_q8_0.restype = i32
            lib.qm_quantize_q8_0.argtypes = [p, i64, p, p]
            lib.qm_quantize_q8_0.restype = i32
            lib.qm_gemv_q4_0_list.argtypes = [p, i64, i64, p, p]
            lib.qm_gemv_q4_0_list.restype = i32
            lib.qm_gemv_q4_0_q8act_list.argtypes = [p, i64, i64, p, p]
            lib.qm_gemv_q4_0_q8act_list.restype = i32
            lib.qm_launch_count.argtypes = []
            lib.qm_launch_count.restype = ctypes.c_uint64
            _lib = lib
    return _lib


def qm_version() -> int:
    return load_library().qm_version()


def qm_status_string(code: int) -> str:
    return load_library().qm_status_string(int(code)).decode()


def _check(code: int, where: str) -> int:
    if code != QM_OK:
        raise QMError(code, where)
    return code


# ------------------------------------------------------------ raw pointers

def qm_dequant_q4_0_ptr(wq: int, n_blocks: int, out: int, stream: int = 0) -> int:
    return load_library().qm_dequant_q4_0(wq, n_blocks, out, stream)


def qm_dequant_q8_0_ptr(wq: int, n_blocks: int, out: int, stream: int = 0) -> int:
    return load_library().qm_dequant_q8_0(wq, n_blocks, out, stream)


def qm_quantize_q8_0_ptr(x: int, n_elements: int, out: int, stream: int = 0) -> int:
    return load_library().qm_quantize_q8_0(x, n_elements, out, stream)


def qm_matmul_q4_0_ptr(A: int, wq: int, C: int, M: int, N: int, K: int, stream: int = 0) -> int:
    return load_library().qm_matmul_q4_0(A, wq, C, M, N, K, stream)


def qm_matmul_q4_0_algo_ptr(A: int, wq: int, C: int, M: int, N: int, K: int, algo: int,
                            stream: int = 0) -> int:
    return load_library().qm_matmul_q4_0_algo(A, wq, C, M, N, K, algo, stream)


def qm_selftest_wait_timeout(stream=None) -> int:
    """Enqueue the failure-path self-test kernel (a bounded wait that runs
    out); the next qm_device_status reports QM_ERR_TIMEOUT.  Returns the C
    status."""
    return load_library().qm_selftest_wait_timeout(_stream_handle(stream))


def qm_matmul_q4_0_noalloc_ptr(A: int, wq: int, C: int, M: int, N: int, K: int,
                               stream: int = 0) -> int:
    """The allocation-free GEMV (M <= 8); see include/qm.h."""
    return load_library().qm_matmul_q4_0_noalloc(A, wq, C, M, N, K, stream)


def qm_matmul_q4_0_q8act_ptr(A: int, wq: int, C: int, M: int, N: int, K: int,
                             stream: int = 0) -> int:
    """The product with the activations quantized to Q8_0 first (M <= 8);
    see include/qm.h."""
    return load_library().qm_matmul_q4_0_q8act(A, wq, C, M, N, K, stream)


def qm_gemv_q4_0_list_ptr(problems, M: int, counters: int = 0, stream: int = 0,
                          q8act: bool = False) -> int:
    """The list GEMV on raw addresses: `problems` is a sequence of (A, wq, C, N,
    K, wait_for) tuples of ints, or an array built once by
    gemv_problem_array; `counters` the device address of len(problems)
    uint32 (0 for none).  With `q8act`, qm_gemv_q4_0_q8act_list (the
    act-quant product).  Returns the C status."""
    arr = problems if isinstance(problems, ctypes.Array) else gemv_problem_array(problems)
    fn = load_library().qm_gemv_q4_0_q8act_list if q8act else load_library().qm_gemv_q4_0_list
    return fn(ctypes.cast(arr, ctypes.c_void_p), len(problems), M, counters or None, stream)


def gemv_problem_array(problems):
    """The C array of qm_gemv_problem for a sequence of (A, wq, C, N, K,
    wait_for) tuples, for callers that pass the same list many times."""
    arr = (QmGemvProblem * len(problems))()
    for i, (A, wq, C, N, K, wait_for) in enumerate(problems):
        arr[i] = QmGemvProblem(A, wq, C, N, K, wait_for, 0)
    return arr


def qm_gemv_q4_0_q8act_list_ptr(problems, M: int, counters: int = 0, stream: int = 0) -> int:
    """qm_gemv_q4_0_q8act_list on raw addresses (see qm_gemv_q4_0_list_ptr)."""
    return qm_gemv_q4_0_list_ptr(problems, M, counters, stream, q8act=True)


# ------------------------------------------------------------ torch tensors

def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _require(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def qm_dequant_q4_0(wq, out=None, stream=None):
    """Dequantize a Q4_0 block stream (uint8 CUDA tensor, n_blocks*18 bytes)
    into f32 ``[n_blocks*32]``."""
    import torch
    _require(wq, torch.uint8, "wq")
    if wq.numel() % BLOCK_BYTES:
        raise ValueError("wq length is not a multiple of 18 bytes")
    n_blocks = wq.numel() // BLOCK_BYTES
    if out is None:
        out = torch.empty(n_blocks * BLOCK_ELEMS, dtype=torch.float32, device=wq.device)
    _require(out, torch.float32, "out")
    if out.numel() != n_blocks * BLOCK_ELEMS:
        raise ValueError("out has the wrong number of elements")
    _check(qm_dequant_q4_0_ptr(wq.data_ptr(), n_blocks, out.data_ptr(), _stream_handle(stream)),
           "qm_dequant_q4_0")
    return out


def qm_dequant_q8_0(wq, out=None, stream=None):
    """Dequantize a Q8_0 block stream (uint8 CUDA tensor, n_blocks*34 bytes)
    into f32 ``[n_blocks*32]``."""
    import torch
    _require(wq, torch.uint8, "wq")
    if wq.numel() % Q8_0_BLOCK_BYTES:
        raise ValueError("wq length is not a multiple of 34 bytes")
    n_blocks = wq.numel() // Q8_0_BLOCK_BYTES
    if out is None:
        out = torch.empty(n_blocks * BLOCK_ELEMS, dtype=torch.float32, device=wq.device)
    _require(out, torch.float32, "out")
    if out.numel() != n_blocks * BLOCK_ELEMS:
        raise ValueError("out has the wrong number of elements")
    _check(qm_dequant_q8_0_ptr(wq.data_ptr(), n_blocks, out.data_ptr(), _stream_handle(stream)),
           "qm_dequant_q8_0")
    return out


def qm_quantize_q8_0(x, out=None, stream=None):
    """Quantize f32 (a CUDA tensor of a multiple of 32 elements) into a Q8_0
    block stream (uint8 ``[n/32*34]``)."""
    import torch
    _require(x, torch.float32, "x")
    if x.numel() % BLOCK_ELEMS:
        raise ValueError("x has a number of elements that is not a multiple of 32")
    n_out = x.numel() // BLOCK_ELEMS * Q8_0_BLOCK_BYTES
    if out is None:
        out = torch.empty(n_out, dtype=torch.uint8, device=x.device)
    _require(out, torch.uint8, "out")
    if out.numel() != n_out:
        raise ValueError("out has the wrong number of bytes")
    _check(qm_quantize_q8_0_ptr(x.data_ptr(), x.numel(), out.data_ptr(), _stream_handle(stream)),
           "qm_quantize_q8_0")
    return out


def qm_matmul_q4_0_algo(A, wq, N: int, algo: int, out=None, stream=None):
    """C[M, N] = A[M, K] x dequant(W)^T with the algorithm forced."""
    import torch
    _require(A, torch.float32, "A")
    _require(wq, torch.uint8, "wq")
    if A.dim() != 2:
        raise ValueError("A must be 2-D [M, K]")
    M, K = A.shape
    if K % BLOCK_ELEMS or wq.numel() != N * (K // BLOCK_ELEMS) * BLOCK_BYTES:
        raise ValueError("wq size does not match N x K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _require(out, torch.float32, "out")
    if out.numel() != M * N:
        raise ValueError("out has the wrong number of elements")
    _check(qm_matmul_q4_0_algo_ptr(A.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K, algo,
                                   _stream_handle(stream)), "qm_matmul_q4_0")
    return out


def qm_matmul_q4_0(A, wq, N: int, out=None, stream=None):
    """C[M, N] = A[M, K] x dequant(W)^T; GEMV kernels for M <= 8, GEMM above."""
    return qm_matmul_q4_0_algo(A, wq, N, QM_ALGO_AUTO, out=out, stream=stream)


def qm_matmul_q4_0_q8act(A, wq, N: int, out=None, stream=None):
    """C[M, N] = dequant_q8_0(quantize_q8_0(A)) x dequant(W)^T for M <= 8."""
    import torch
    _require(A, torch.float32, "A")
    _require(wq, torch.uint8, "wq")
    if A.dim() != 2:
        raise ValueError("A must be 2-D [M, K]")
    M, K = A.shape
    if K % BLOCK_ELEMS or wq.numel() != N * (K // BLOCK_ELEMS) * BLOCK_BYTES:
        raise ValueError("wq size does not match N x K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _require(out, torch.float32, "out")
    if out.numel() != M * N:
        raise ValueError("out has the wrong number of elements")
    _check(qm_matmul_q4_0_q8act_ptr(A.data_ptr(), wq.data_ptr(), out.data_ptr(), M, N, K,
                                    _stream_handle(stream)), "qm_matmul_q4_0_q8act")
    return out


def qm_gemv_q4_0_list(problems, M: int = 1, counters=None, stream=None):
    """Run a list of GEMV problems ``(A, wq, C, N, wait_for)`` (A f32 [M, K], wq
    the uint8 block stream of N x K, C f32 [M, N] written in place) in one
    persistent launch where the shapes allow; ``counters`` is a uint32 or int32
    CUDA tensor of len(problems) entries, needed for launches in which a
    problem waits on another (see include/qm.h)."""
    import torch
    raw = []
    for A, wq, C, N, wait_for in problems:
        _require(A, torch.float32, "A")
        _require(wq, torch.uint8, "wq")
        _require(C, torch.float32, "C")
        K = A.shape[-1]
        if A.numel() != M * K or C.numel() != M * N or K % BLOCK_ELEMS or \
                wq.numel() != N * (K // BLOCK_ELEMS) * BLOCK_BYTES:
            raise ValueError("problem operands do not match M, N, K")
        raw.append((A.data_ptr(), wq.data_ptr(), C.data_ptr(), N, K, wait_for))
    ctr = 0
    if counters is not None:
        if not counters.is_cuda or counters.element_size() != 4 or counters.numel() < len(problems):
            raise ValueError("counters must be a CUDA tensor of len(problems) 32-bit entries")
        ctr = counters.data_ptr()
    _check(qm_gemv_q4_0_list_ptr(raw, M, ctr, _stream_handle(stream)), "qm_gemv_q4_0_list")


GEMV_PLAN_FIELDS = ("RG", "U", "S", "rps", "c", "hs", "rbpc", "nu_max", "stages", "grid", "smem", "W",
                    "cl")


def qm_gemv_plan(M: int, N: int, K: int, packed: bool = False, sm_count: int = 152,
                 smem_optin: int = 232448, fit=(76, 38, 19), noalloc: bool = False):
    """The decode GEMV's launch plan (host only, see include/qm.h) as a dict,
    or None when no plan fits; raises on invalid arguments.  `fit` = resident
    clusters of 2, 4 and 8 CTAs (the regular path's K split); with `noalloc`
    the plan of qm_matmul_q4_0_noalloc."""
    out = (ctypes.c_int64 * 13)()
    rc = load_library().qm_gemv_plan(M, N, K, 1 if packed else 0, sm_count, smem_optin, fit[0], fit[1],
                                     fit[2], 1 if noalloc else 0, ctypes.cast(out, ctypes.c_void_p))
    if rc == QM_ERR_UNSUPPORTED:
        return None
    _check(rc, "qm_gemv_plan")
    return dict(zip(GEMV_PLAN_FIELDS, (int(v) for v in out)))


GEMM_PLAN_FIELDS = ("BN", "nt", "tiles", "n_full", "s_rem", "hw", "items", "cl")


def qm_gemm_plan(M: int, N: int, K: int, sm_count: int = 152, fit=(76, 38, 19)):
    """The prefill GEMM's work items (host only, see include/qm.h) as a dict;
    `fit` = resident clusters of 2, 4 and 8 CTAs."""
    out = (ctypes.c_int64 * 8)()
    _check(load_library().qm_gemm_plan(M, N, K, sm_count, fit[0], fit[1], fit[2],
                                       ctypes.cast(out, ctypes.c_void_p)), "qm_gemm_plan")
    return dict(zip(GEMM_PLAN_FIELDS, (int(v) for v in out)))


def qm_launch_count() -> int:
    """Kernels enqueued by the library so far in this process."""
    return int(load_library().qm_launch_count())


def qm_device_status(stream=None, clear: bool = True) -> int:
    """Synchronize the stream and return the device error status (QM_OK or
    QM_ERR_TIMEOUT); see include/qm.h."""
    return load_library().qm_device_status(_stream_handle(stream), 1 if clear else 0)
