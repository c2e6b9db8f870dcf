"""GPU parity of the push form (AR_ALGO_PUSH) against the CPU oracle.

Writers store their tile into a receive area of every peer and readers sum
their own area; the arithmetic is the other forms', so every output must match
the oracle bit for bit, per-rank and in one launch of every rank, in graphs,
and interleaved with the pull forms on one handle.
"""
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, capture, enqueue, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _handle(R, dtype, n, slots):
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, TORCH[dtype], n, slots)
    h.set_algo("push")
    return h


def _check(outs, xs, dtype, what):
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r, o in enumerate(outs):
        assert_bits_equal(to_bits(o), want, dtype, f"{what} rank {r}")


@pytest.mark.parametrize("R,dtype,slots", [(1, "f16", "hbm"), (2, "f16", "pinned"), (2, "bf16", "hbm"),
                                           (3, "bf16", "pinned"), (4, "f16", "hbm"), (4, "bf16", "pinned"),
                                           (8, "bf16", "hbm"), (8, "f16", "pinned")])
@pytest.mark.parametrize("n", [1, 9, 4096, 131072 + 5, 1 << 20])
def test_push_matches_oracle(R, dtype, slots, n):
    """Per-rank launches, one tile per block and stage: the 1 Mi-element calls
    run several stages per block, the odd ones have ragged tails."""
    h = _handle(R, dtype, n, slots)
    assert h.plan("allreduce", n).algo == 4
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", n % 31)
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.full_like(t, float("nan")) for t in ins]
    enqueue(h, "allreduce", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    h.check()
    _check(outs, xs, dtype, f"push R={R} n={n} {slots}")
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
def test_push_graph_replays_and_fused_launch(slots):
    """A graph of 20 per-rank push calls replayed 3 times with fresh inputs,
    then push calls as one launch of every rank."""
    R, n, C, dtype = 4, 65536 + 3, 20, "bf16"
    h = _handle(R, dtype, n, slots)
    streams = rank_streams(R)
    ins = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(C)]
    outs = [[torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)] for _ in range(C)]
    g = capture(h, "allreduce", ins, outs, streams)
    for rep in range(3):
        xs_all = [inputs.allreduce_inputs(5, R, n, dtype, "uniform", 1000 + rep * C + c) for c in range(C)]
        for c in range(C):
            for r in range(R):
                ins[c][r].copy_(to_dev(xs_all[c][r], dtype))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(C):
            _check(outs[c], xs_all[c], dtype, f"replay {rep} call {c}")
    del g
    s = torch.cuda.Stream()
    for c in range(3):
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 2000 + c)
        ins1 = [to_dev(x, dtype) for x in xs]
        outs1 = [torch.empty_like(t) for t in ins1]
        s.wait_stream(torch.cuda.current_stream())
        h.allreduce_fused(ins1, outs1, s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        h.check()
        _check(outs1, xs, dtype, f"fused push {c}")
    h.destroy()


def test_push_interleaves_with_pull_forms():
    """Push, one-shot, two-shot and tagged calls in turn on one handle: the
    shared counters keep slot parity and stage counts consistent."""
    import tensor_decode_all_gb300 as tda
    R, dtype, nmax = 4, "f16", 1 << 19
    h = tda.Handle(R, torch.float16, nmax, "hbm")
    streams = rank_streams(R)
    seq = [("push", 5000), ("oneshot", 70001), ("push", nmax), ("twoshot", 300000), ("tagged", 2048),
           ("push", 17), ("push", 4096), ("oneshot", 9)]
    for rnd in range(2):
        for i, (form, n) in enumerate(seq):
            h.set_algo(form)
            xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 3000 + 10 * rnd + i)
            ins = [to_dev(x, dtype) for x in xs]
            outs = [torch.full_like(t, float("nan")) for t in ins]
            enqueue(h, "allreduce", ins, outs, streams)
            torch.cuda.synchronize()
            h.check()
            _check(outs, xs, dtype, f"round {rnd} step {i} {form} n={n}")
    h.destroy()


def test_push_refused_for_complex64_and_reset_clears_its_flags():
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    hc = tda.Handle(2, torch.complex64, 16, "hbm")
    assert ar.ar_set_algo(hc.ptr, ar.AR_ALGO_PUSH) == ar.AR_EINVAL
    hc.destroy()
    R, n, dtype = 2, 8192, "f16"
    h = _handle(R, dtype, n, "pinned")
    streams = rank_streams(R)
    for c in range(3):
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 4000 + c)
        ins = [to_dev(x, dtype) for x in xs]
        outs = [torch.empty_like(t) for t in ins]
        enqueue(h, "allreduce", ins, outs, streams)
        torch.cuda.synchronize()
        _check(outs, xs, dtype, f"before reset {c}")
        if c == 1:
            h.reset()            # counters and push flags back to zero together
    h.destroy()
