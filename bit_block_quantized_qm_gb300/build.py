"""Build libqm.so in-tree with nvcc for sm_103a (GB300).

Each CUDA source compiles to an object in parallel; the objects link into
``bit_block_quantized_qm_gb300/_build/libqm.so`` with the CUDA runtime linked
statically, so the library needs only the NVIDIA driver at run time.

``build_test_hooks()`` builds a second copy with the test-only hooks of
``include/qm_test.h`` compiled in (``-DQM_TEST_HOOKS``), into
``_build/test/libqm.so``; the product library never carries them.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libqm.so")
SOURCES = ("qm_api.cu", "dequant.cu", "q8_0.cu", "gemv.cu", "gemv_tc.cu", "gemv_list.cu", "gemv_q8act.cu", "gemm.cu",
           "gemm_tc.cu")
HEADERS = ("qm_device.cuh", "qm_internal.h")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqm")
    return path


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra, out_dir: str = BUILD) -> str:
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src), *(os.path.join(CSRC, h) for h in HEADERS),
            os.path.join(ROOT, "include", "qm.h"), os.path.join(ROOT, "include", "qm_test.h")]
    if _stale(obj, deps) or (extra and out_dir == BUILD):
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(extra_flags=(), force: bool = False) -> str:
    """Compile (if stale) and link libqm.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra_flags)
    if force:
        for s in SOURCES:
            obj = os.path.join(BUILD, os.path.splitext(s)[0] + ".o")
            if os.path.exists(obj):
                os.remove(obj)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    if _stale(LIB, objs) or extra:
        cmd = [nvcc(), *ARCH, "-shared", "-o", LIB, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    return LIB


TEST_BUILD = os.path.join(BUILD, "test")
TEST_LIB = os.path.join(TEST_BUILD, "libqm.so")


def build_test_hooks() -> str:
    """Compile (if stale) and link the test-hook copy of libqm.so; returns its path."""
    os.makedirs(TEST_BUILD, exist_ok=True)
    flags = ["-DQM_TEST_HOOKS"]
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, TEST_BUILD), SOURCES))
    if _stale(TEST_LIB, objs):
        cmd = [nvcc(), *ARCH, "-shared", "-o", TEST_LIB, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    return TEST_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
