"""CPU oracle for the GGML Q4_0 x f32 quantized matmul and the Q8_0 dequant and
quantize — TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``qm_oracle.c`` (plain C99, fp64, single-threaded);
this module compiles it with gcc and exposes it to numpy through ctypes.
``load_parallel()`` binds a second build of the same source with OpenMP,
which shares independent output entries (and dequant blocks) out over the
host's cores for the multi-core CPU baseline; every entry is still one
ascending-k fp64 sum, so its results are bit-identical to ``load()``'s.
Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it.

Functions (all follow "fuel-vulkan-kernels — quantized (GGML) kernel
contracts", sections ``dequant_q4_0``, ``qmatvec_q4_0``, ``matmul_q4_0_tiled``,
``dequant_q8_0`` and ``quantize_q8_0``):

* ``f16_to_double(bits)``      — binary16 decode, elementwise;
* ``dequant_q4_0(blob)``       — block stream -> f32, ``(nibble - 8) * d``;
* ``matmul_q4_0(A, blob, N, K)`` -> ``(C, S)`` in fp64, with
  ``S = sum_k |A[m,k] * W[n,k]|`` for the tolerance;
* ``matmul_q4_0_entries(A, blob, N, K, m_idx, n_idx)`` — the same for chosen
  entries only (sampled checks at full size);
* ``float_to_f16(x)``          — f32 -> binary16 bits, round to nearest even;
* ``dequant_q8_0(blob)``       — Q8_0 block stream -> f32, ``qs * d``;
* ``quantize_q8_0(x)``         — f32 (a multiple of 32 elements) -> Q8_0 blocks,
  with the readings stated in ``qm_oracle.h``.

Every function is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_OMP_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_omp.so")

BLOCK_BYTES = 18
BLOCK_ELEMS = 32
Q8_0_BLOCK_BYTES = 34

_lock = threading.Lock()
_lib = None
_omp_lib = None

# Plain IEEE arithmetic: no contraction into fused multiply-adds, no fast-math.
_CFLAGS = ["-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra"]


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile an oracle source file into a shared library with gcc."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *_CFLAGS, *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def build_all() -> None:
    """Compile both builds of the oracle: plain, and with OpenMP."""
    build()
    build(out=_OMP_LIB_PATH, extra_flags=("-fopenmp",))


def _needs_build(path: str) -> bool:
    if not os.path.exists(path):
        return True
    src_mtime = max(os.path.getmtime(_SRC),
                    os.path.getmtime(os.path.join(_HERE, "qm_oracle.h")))
    return os.path.getmtime(path) < src_mtime


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    i64, p = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_to_double.restype = ctypes.c_double
    lib.oracle_f16_to_double_array.argtypes = [p, i64, p]
    lib.oracle_f16_to_double_array.restype = None
    lib.oracle_dequant_q4_0.argtypes = [p, i64, p]
    lib.oracle_dequant_q4_0.restype = None
    lib.oracle_matmul_q4_0.argtypes = [p, p, i64, i64, i64, p, p]
    lib.oracle_matmul_q4_0.restype = ctypes.c_int
    lib.oracle_matmul_q4_0_entries.argtypes = [p, p, i64, i64, i64, p, p, i64, p, p]
    lib.oracle_matmul_q4_0_entries.restype = ctypes.c_int
    lib.oracle_float_to_f16_array.argtypes = [p, i64, p]
    lib.oracle_float_to_f16_array.restype = None
    lib.oracle_dequant_q8_0.argtypes = [p, i64, p]
    lib.oracle_dequant_q8_0.restype = None
    lib.oracle_quantize_q8_0.argtypes = [p, i64, p]
    lib.oracle_matmul_q4_0_q8act.argtypes = [p, p, i64, i64, i64, p, p]
    lib.oracle_matmul_q4_0_q8act.restype = ctypes.c_int
    lib.oracle_matmul_q4_0_q8act_entries.argtypes = [p, p, i64, i64, i64, p, p, i64, p, p]
    lib.oracle_matmul_q4_0_q8act_entries.restype = ctypes.c_int
    lib.oracle_quantize_q8_0.restype = None
    return lib


def load(path: str | None = None) -> "Oracle":
    """Return the oracle bound to the default library (built on first use), or
    to the library at ``path`` (used by tests that compile a planted mistake)."""
    global _lib
    if path is not None:
        return Oracle(_bind(ctypes.CDLL(path)))
    with _lock:
        if _lib is None:
            if _needs_build(_LIB_PATH):
                build()
            _lib = Oracle(_bind(ctypes.CDLL(_LIB_PATH)))
    return _lib


def load_parallel() -> "Oracle":
    """The oracle built with OpenMP (threads: OMP_NUM_THREADS, else every
    core the process may run on)."""
    global _omp_lib
    with _lock:
        if _omp_lib is None:
            if _needs_build(_OMP_LIB_PATH):
                build(out=_OMP_LIB_PATH, extra_flags=("-fopenmp",))
            _omp_lib = Oracle(_bind(ctypes.CDLL(_OMP_LIB_PATH)))
    return _omp_lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """numpy-facing wrapper over one loaded copy of the C oracle."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib

    def f16_to_double(self, bits) -> np.ndarray:
        h = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16).ravel())
        out = np.empty(h.size, dtype=np.float64)
        self.lib.oracle_f16_to_double_array(_ptr(h), h.size, _ptr(out))
        return out

    def dequant_q4_0(self, blob: np.ndarray) -> np.ndarray:
        blob = np.ascontiguousarray(blob, dtype=np.uint8).ravel()
        if blob.size % BLOCK_BYTES:
            raise ValueError("blob length is not a multiple of 18 bytes")
        n_blocks = blob.size // BLOCK_BYTES
        out = np.empty(n_blocks * BLOCK_ELEMS, dtype=np.float32)
        self.lib.oracle_dequant_q4_0(_ptr(blob), n_blocks, _ptr(out))
        return out

    @staticmethod
    def _check(A, blob, N, K):
        A = np.ascontiguousarray(A, dtype=np.float32)
        if A.ndim != 2 or A.shape[1] != K:
            raise ValueError("A must be [M, K]")
        blob = np.ascontiguousarray(blob, dtype=np.uint8).ravel()
        if K % BLOCK_ELEMS or blob.size != N * (K // BLOCK_ELEMS) * BLOCK_BYTES:
            raise ValueError("blob size does not match N x K")
        return A, blob

    def matmul_q4_0(self, A: np.ndarray, blob: np.ndarray, N: int, K: int):
        A, blob = self._check(A, blob, N, K)
        M = A.shape[0]
        C = np.empty((M, N), dtype=np.float64)
        S = np.empty((M, N), dtype=np.float64)
        rc = self.lib.oracle_matmul_q4_0(_ptr(A), _ptr(blob), M, N, K, _ptr(C), _ptr(S))
        if rc != 0:
            raise ValueError("oracle rejected the sizes")
        return C, S

    def matmul_q4_0_entries(self, A, blob, N, K, m_idx, n_idx):
        A, blob = self._check(A, blob, N, K)
        M = A.shape[0]
        mi = np.ascontiguousarray(m_idx, dtype=np.int64).ravel()
        ni = np.ascontiguousarray(n_idx, dtype=np.int64).ravel()
        if mi.size != ni.size:
            raise ValueError("index arrays differ in length")
        C = np.empty(mi.size, dtype=np.float64)
        S = np.empty(mi.size, dtype=np.float64)
        rc = self.lib.oracle_matmul_q4_0_entries(_ptr(A), _ptr(blob), M, N, K,
                                                 _ptr(mi), _ptr(ni), mi.size,
                                                 _ptr(C), _ptr(S))
        if rc != 0:
            raise ValueError("oracle rejected the sizes or indices")
        return C, S


    def matmul_q4_0_q8act(self, A: np.ndarray, blob: np.ndarray, N: int, K: int):
        """C and S of A' x dequant(W)^T, A' = dequant_q8_0(quantize_q8_0(A))."""
        A, blob = self._check(A, blob, N, K)
        M = A.shape[0]
        C = np.empty((M, N), dtype=np.float64)
        S = np.empty((M, N), dtype=np.float64)
        rc = self.lib.oracle_matmul_q4_0_q8act(_ptr(A), _ptr(blob), M, N, K, _ptr(C), _ptr(S))
        if rc != 0:
            raise ValueError("oracle rejected the sizes")
        return C, S

    def matmul_q4_0_q8act_entries(self, A, blob, N, K, m_idx, n_idx):
        A, blob = self._check(A, blob, N, K)
        M = A.shape[0]
        mi = np.ascontiguousarray(m_idx, dtype=np.int64).ravel()
        ni = np.ascontiguousarray(n_idx, dtype=np.int64).ravel()
        if mi.size != ni.size:
            raise ValueError("index arrays differ in length")
        C = np.empty(mi.size, dtype=np.float64)
        S = np.empty(mi.size, dtype=np.float64)
        rc = self.lib.oracle_matmul_q4_0_q8act_entries(_ptr(A), _ptr(blob), M, N, K, _ptr(mi),
                                                       _ptr(ni), mi.size, _ptr(C), _ptr(S))
        if rc != 0:
            raise ValueError("oracle rejected the sizes or indices")
        return C, S

    def float_to_f16(self, x) -> np.ndarray:
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float32).ravel())
        out = np.empty(x.size, dtype=np.uint16)
        self.lib.oracle_float_to_f16_array(_ptr(x), x.size, _ptr(out))
        return out

    def dequant_q8_0(self, blob: np.ndarray) -> np.ndarray:
        blob = np.ascontiguousarray(blob, dtype=np.uint8).ravel()
        if blob.size % Q8_0_BLOCK_BYTES:
            raise ValueError("blob length is not a multiple of 34 bytes")
        n_blocks = blob.size // Q8_0_BLOCK_BYTES
        out = np.empty(n_blocks * BLOCK_ELEMS, dtype=np.float32)
        self.lib.oracle_dequant_q8_0(_ptr(blob), n_blocks, _ptr(out))
        return out

    def quantize_q8_0(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float32).ravel())
        if x.size % BLOCK_ELEMS:
            raise ValueError("element count is not a multiple of 32")
        n_blocks = x.size // BLOCK_ELEMS
        blob = np.empty(n_blocks * Q8_0_BLOCK_BYTES, dtype=np.uint8)
        self.lib.oracle_quantize_q8_0(_ptr(x), n_blocks, _ptr(blob))
        return blob


def within_tolerance(C_test, C_ref, S_ref, rel=1e-5, abs_=1e-7):
    """Per-element check |C_test - C_ref| <= rel * S + abs_.  Non-finite
    reference entries must be matched by class: NaN by NaN, +-Inf by the same
    Inf.  Returns a boolean array of the entries that pass."""
    C_test = np.asarray(C_test, dtype=np.float64)
    C_ref = np.asarray(C_ref, dtype=np.float64)
    S_ref = np.asarray(S_ref, dtype=np.float64)
    finite = np.isfinite(C_ref) & np.isfinite(S_ref)
    ok = np.zeros(C_ref.shape, dtype=bool)
    with np.errstate(invalid="ignore"):
        ok[finite] = np.abs(C_test[finite] - C_ref[finite]) <= rel * S_ref[finite] + abs_
    nan_ref = np.isnan(C_ref)
    ok[nan_ref] = np.isnan(C_test[nan_ref])
    inf_ref = np.isinf(C_ref)
    ok[inf_ref] = C_test[inf_ref] == C_ref[inf_ref]
    # A finite result whose absolute sum overflowed puts no bound on the error.
    odd = np.isfinite(C_ref) & ~np.isfinite(S_ref)
    ok[odd] = ~np.isnan(C_test[odd])
    return ok
