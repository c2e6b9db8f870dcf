"""GPU parity across the payload sweep (workload 5) and at the largest size.

A reduced grid of the sweep: every R (2, 4, 8) x dtype x slot kind at four
payloads from 2 KiB to 16 MiB per rank, each captured as a graph of two calls
(the two slot parities) and checked bit for bit against the CPU oracle; and
the sweep's largest cell, R=8 bf16 64 MiB per rank (two-shot, HBM slots).
The full 192-cell sweep with 1000 calls per cell runs in bench.py --sweep.
"""
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, capture, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _cell(R, dtype, nbytes, slots, calls=2):
    import tensor_decode_all_gb300 as tda
    n = nbytes // 2
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    h = tda.Handle(R, tdt, n, slots)
    streams = rank_streams(R)
    xs_all = [inputs.allreduce_inputs(5, R, n, dtype, "uniform", c) for c in range(calls)]
    ins = [[to_dev(x, dtype) for x in xs] for xs in xs_all]
    outs = [[torch.empty(n, dtype=tdt, device="cuda") for _ in range(R)] for _ in range(calls)]
    g = capture(h, "allreduce", ins, outs, streams)
    g.replay()
    torch.cuda.synchronize()
    h.check()
    for c in (0, calls - 1):
        want = oracle.allreduce(xs_all[c], dtype, ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[c][r]), want, dtype, f"R={R} {dtype} {nbytes}B {slots} call {c} rank {r}")
    del g
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("nbytes", [2 << 10, 64 << 10, 1 << 20, 16 << 20])
def test_sweep_cell(nbytes, R, dtype, slots):
    _cell(R, dtype, nbytes, slots)


def test_largest_cell_r8_bf16_64MiB_hbm():
    _cell(8, "bf16", 64 << 20, "hbm", calls=1)
