"""GPU parity across the whole payload sweep (workload 5).

Every cell of the sweep -- R = 2, 4, 8 x fp16, bf16 x pinned-host and HBM
slots x the 16 payloads 2 KiB .. 64 MiB per rank (192 cells) -- is captured
as a graph of two calls (the two slot parities, each with its own inputs)
and replayed until the cell has run its calls: 1000 for payloads up to 1 MiB,
fewer for the large ones (at least 8, and about 4 GiB of payload per cell, so
that the run stays within minutes).  The first replay's two calls and the
last replay's two calls are compared bit for bit with the CPU oracle on
every rank.  Timing the same cells is bench.py --sweep's job.
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, capture, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu

SIZES = [1 << k for k in range(11, 27)]   # 2 KiB .. 64 MiB per rank


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def calls_for(R, nbytes):
    if nbytes <= (1 << 20):
        return 1000
    return max(8, min(1000, (4 << 30) // (R * nbytes)))


def _check(outs, xs_all, R, dtype, label):
    for c in range(len(xs_all)):
        want = oracle.allreduce(xs_all[c], dtype, ranks=[0], nthreads=oracle.max_threads())[0]
        got = to_bits(torch.stack(outs[c]))
        if not np.array_equal(got, np.broadcast_to(want, got.shape)):
            for r in range(R):
                assert_bits_equal(got[r], want, dtype, f"{label} call {c} rank {r}")


_last_inputs = {}


def _inputs(R, n, dtype):
    """The cell's two calls' inputs (kept for the next cell with the same
    shape: the two slot kinds of a cell share their inputs)."""
    key = (R, n, dtype)
    if key not in _last_inputs:
        _last_inputs.clear()
        _last_inputs[key] = [inputs.allreduce_inputs(5, R, n, dtype, "uniform", c) for c in range(2)]
    return _last_inputs[key]


def _cell(R, dtype, nbytes, slots):
    import tensor_decode_all_gb300 as tda
    n = nbytes // 2
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    h = tda.Handle(R, tdt, n, slots)
    streams = rank_streams(R)
    xs_all = _inputs(R, n, dtype)
    ins = [[to_dev(x, dtype) for x in xs] for xs in xs_all]
    outs = [[torch.empty(n, dtype=tdt, device="cuda") for _ in range(R)] for _ in range(2)]
    g = capture(h, "allreduce", ins, outs, streams)
    label = f"R={R} {dtype} {nbytes}B {slots}"
    total = calls_for(R, nbytes)
    g.replay()
    torch.cuda.synchronize()
    h.check()
    _check(outs, xs_all, R, dtype, label + " first replay")
    for o in outs:
        for t in o:
            t.fill_(float("nan"))
    for _ in range(total // 2 - 1):
        g.replay()
    torch.cuda.synchronize()
    h.check()
    _check(outs, xs_all, R, dtype, label + f" replay {total // 2}")
    del g
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("nbytes", SIZES)
def test_sweep_cell(nbytes, R, dtype, slots):
    _cell(R, dtype, nbytes, slots)

