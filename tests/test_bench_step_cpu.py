"""The bench step's operand layout, built on the host (no GPU).

bench.sweep_operands builds the decoder sweep's 224 GEMVs as one problem
list over one activation buffer and one output buffer per replica.  Within a
layer q, k and v must read one input vector, gate and up another, o and down
their own; every output must be its own N floats, the outputs back to back;
and the shapes must be the sweep's.  Run on CPU tensors with 2 layers (the
addresses are only recorded, never dereferenced).
"""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

torch = pytest.importorskip("torch")

import bench  # noqa: E402
import synth  # noqa: E402


def test_sweep_operands_layout():
    import bit_block_quantized_qm_gb300 as qm
    cases = synth.workload(4, layers=2, sweep_m=(1,))
    weights, a_host, c_total, reps = bench.sweep_operands(qm, torch, torch.device("cpu"), cases, 2)
    assert len(weights) == len(cases) == 14
    assert c_total == sum(c.N for c in cases)
    # 4 input vectors per layer: q (K 4096), o (4096), gate (4096), down (14336).
    assert a_host.size == 2 * (3 * 4096 + 14336)
    for rp in reps:
        arr = rp["problems"]
        A0, C0 = rp["A"].data_ptr(), rp["C"].data_ptr()
        assert len(arr) == len(cases)
        c_end = C0
        for i, (c, p) in enumerate(zip(cases, arr)):
            assert (p.N, p.K, p.wait_for, p.reserved) == (c.N, c.K, -1, 0)
            assert p.wq == weights[i].data_ptr()
            assert p.C == c_end, "outputs back to back, in problem order"
            c_end += 4 * c.N
        assert c_end == C0 + 4 * c_total
        for layer in range(2):
            a = [arr[7 * layer + j].A for j in range(7)]
            q, k, v, o, gate, up, down = a
            assert q == k == v and gate == up
            assert len({q, o, gate, down}) == 4
            for j, addr in enumerate(a):
                off = (addr - A0) // 4
                K = cases[7 * layer + j].K
                assert 0 <= off and off + K <= a_host.size
                # The vector at that offset is the layer's input for this projection.
                src = 7 * layer + bench.SHARED_INPUT[bench.DECODER_PROJS[j]]
                np.testing.assert_array_equal(a_host[off:off + K], cases[src].acts().ravel())
    # The replicas do not share activation or output buffers.
    assert reps[0]["A"].data_ptr() != reps[1]["A"].data_ptr()
    assert reps[0]["C"].data_ptr() != reps[1]["C"].data_ptr()
