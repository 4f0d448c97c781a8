"""Seeded synthetic inputs for the Q4_0 x f32 matmul and the Q4_0 dequant.

This module only draws random numbers and lays them out in the GGML Q4_0 byte
format; it holds none of the decode or matmul arithmetic.  Both the CUDA tests
and the oracle take their inputs from here.

Q4_0 block layout (18 bytes, 32 elements; "fuel-vulkan-kernels — quantized
(GGML) kernel contracts", section ``dequant_q4_0``): bytes 0-1 hold the scale
``d`` as little-endian IEEE binary16, bytes 2-17 the 16 quant bytes.  Because
the generators draw each quant byte uniformly from 0..255, both of its nibbles
are independent and uniform on 0..15.

Random streams: every array comes from its own ``numpy.random.Generator``
(PCG64) seeded by ``SeedSequence(seed, spawn_key=key)``, so each matrix of a
workload is reproducible on its own.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BLOCK_BYTES = 18
BLOCK_ELEMS = 32


def rng(seed: int, key: tuple = ()) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(key))))


def blob_bytes(N: int, K: int) -> int:
    return N * (K // BLOCK_ELEMS) * BLOCK_BYTES


def assemble_blocks(d_f16: np.ndarray, quant_bytes: np.ndarray) -> np.ndarray:
    """Lay out per-block scales (float16 [nb]) and quant bytes (uint8 [nb,16])
    as the 18-byte block stream (flat uint8)."""
    d_f16 = np.ascontiguousarray(d_f16, dtype="<f2").ravel()
    quant_bytes = np.ascontiguousarray(quant_bytes, dtype=np.uint8).reshape(-1, 16)
    nb = d_f16.size
    if quant_bytes.shape[0] != nb:
        raise ValueError("scale and quant counts differ")
    out = np.empty((nb, BLOCK_BYTES), dtype=np.uint8)
    out[:, 0:2] = d_f16.view(np.uint8).reshape(nb, 2)
    out[:, 2:] = quant_bytes
    return out.ravel()


def q4_0_weights(N: int, K: int, seed: int, key: tuple = (0,),
                 scale: str = "abs_normal") -> np.ndarray:
    """A row-major [N][K/32] Q4_0 block stream.

    scale="abs_normal": d = f16(|N(0,1)| * 0.02)            (round to nearest even)
    scale="log_uniform": d = f16(exp(U[ln 1e-3, ln 5e-2]))
    Quant nibbles are uniform on 0..15."""
    if K % BLOCK_ELEMS:
        raise ValueError("K must be a multiple of 32")
    nb = N * (K // BLOCK_ELEMS)
    g = rng(seed, key)
    if scale == "abs_normal":
        d = (np.abs(g.standard_normal(nb)) * 0.02).astype(np.float16)
    elif scale == "log_uniform":
        d = np.exp(g.uniform(np.log(1e-3), np.log(5e-2), nb)).astype(np.float16)
    else:
        raise ValueError(f"unknown scale distribution {scale!r}")
    q = g.integers(0, 256, size=(nb, 16), dtype=np.uint8)
    return assemble_blocks(d, q)


def activations(M: int, K: int, seed: int, key: tuple = (1,),
                dist: str = "normal") -> np.ndarray:
    """f32 [M, K].  dist="normal": N(0,1).  dist="outliers": 0.5*N(0,1), then
    each entry independently (probability 0.01) replaced by +20 or -20 with
    equal odds."""
    g = rng(seed, key)
    if dist == "normal":
        return g.standard_normal((M, K), dtype=np.float32)
    if dist == "outliers":
        a = (0.5 * g.standard_normal((M, K))).astype(np.float32)
        hit = g.random((M, K)) < 0.01
        sign = np.where(g.integers(0, 2, size=(M, K)) == 1, 20.0, -20.0).astype(np.float32)
        a[hit] = sign[hit]
        return a
    raise ValueError(f"unknown activation distribution {dist!r}")


@dataclass(frozen=True)
class Case:
    """One operation of a workload: a matmul (M>=1) or a dequant of an N x K weight."""
    name: str
    op: str            # "matmul" | "dequant"
    M: int
    N: int
    K: int
    seed: int
    w_key: tuple = (0,)
    a_key: tuple = (1,)
    a_dist: str = "normal"
    d_dist: str = "abs_normal"
    tags: tuple = field(default_factory=tuple)

    def weights(self) -> np.ndarray:
        return q4_0_weights(self.N, self.K, self.seed, self.w_key, self.d_dist)

    def acts(self) -> np.ndarray:
        return activations(self.M, self.K, self.seed, self.a_key, self.a_dist)

    @property
    def weight_bytes(self) -> int:
        return blob_bytes(self.N, self.K)


# Decoder layer shapes (hidden 4096, grouped-query attention), as (name, K, N):
# K is the input width, N the output width of each projection.
DECODER_LAYER = (("q", 4096, 4096), ("k", 4096, 1024), ("v", 4096, 1024),
                 ("o", 4096, 4096), ("gate", 4096, 14336), ("up", 4096, 14336),
                 ("down", 14336, 4096))


def workload(index: int, layers: int = 32, sweep_m=(1, 8, 512)) -> list:
    """The cases of workload `index` (0..4).

    0: GEMV M=1, K=N=4096, A ~ N(0,1), d = f16(|N(0,1)|*0.02); seed 0.
    1: GEMV M=8 at (K=4096, N=14336) seed 1 and (K=14336, N=4096) seed 2; plus
       the dequant of the 14336 x 4096 weight (the seed-1 weight).
    2: prefill M=32 and M=256, K=N=4096, A = 0.5*N(0,1) with 1% outliers of
       +-20; seed 3 (one weight, one activation draw per M).
    3: prefill M=1024 at (K=4096, N=14336) and (K=14336, N=4096); d =
       f16(log-uniform on [1e-3, 5e-2]); A ~ N(0,1); seed 4.
    4: decoder sweep: `layers` layers of DECODER_LAYER at each M in sweep_m;
       seed 5, one weight stream per (layer, projection), shared over M.
    """
    if index == 0:
        return [Case("gemv_m1_k4096_n4096", "matmul", 1, 4096, 4096, 0)]
    if index == 1:
        return [Case("gemv_m8_k4096_n14336", "matmul", 8, 14336, 4096, 1),
                Case("gemv_m8_k14336_n4096", "matmul", 8, 4096, 14336, 2),
                Case("dequant_n14336_k4096", "dequant", 0, 14336, 4096, 1)]
    if index == 2:
        return [Case(f"prefill_m{m}_k4096_n4096", "matmul", m, 4096, 4096, 3,
                     a_key=(1, m), a_dist="outliers") for m in (32, 256)]
    if index == 3:
        return [Case("prefill_m1024_k4096_n14336", "matmul", 1024, 14336, 4096, 4,
                     w_key=(0, 0), a_key=(1, 0), d_dist="log_uniform"),
                Case("prefill_m1024_k14336_n4096", "matmul", 1024, 4096, 14336, 4,
                     w_key=(0, 1), a_key=(1, 1), d_dist="log_uniform")]
    if index == 4:
        out = []
        for m in sweep_m:
            for layer in range(layers):
                for p, (proj, K, N) in enumerate(DECODER_LAYER):
                    out.append(Case(f"layer{layer}_{proj}_m{m}", "matmul", m, N, K, 5,
                                    w_key=(0, layer, p), a_key=(1, layer, p, m),
                                    tags=(("layer", layer), ("proj", proj))))
        return out
    raise ValueError(f"no workload {index}")
