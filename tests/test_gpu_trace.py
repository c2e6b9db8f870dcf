"""The device-side trace (ar_set_trace) on the GPU.

The exchange needs every rank's block b to run while its peers' blocks b do;
the trace shows it: for every call and block, the latest of the R start times
comes before the earliest end.  The traced calls must still be bit-exact.
"""
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, capture, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("R,dtype,n,slots,fused", [
    (2, "f16", 131072, "pinned", False),   # one-shot over the host link
    (2, "f16", 4096, "pinned", False),     # tagged words
    (8, "bf16", 393216, "hbm", False),     # two-shot
    (8, "bf16", 393216, "hbm", "flags"),   # two-shot, one cooperative launch of every rank
    (8, "bf16", 393216, "hbm", True),      # cluster form (one launch of every rank, AUTO)
    (2, "f16", 131072, "pinned", True),    # cluster form over the host link
])
def test_trace_shows_rank_kernels_overlap(R, dtype, n, slots, fused):
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import trace
    C, depth = 6, 8
    h = tda.Handle(R, TORCH[dtype], n, slots)
    if fused == "flags":
        h.set_tactics(cluster_max_bytes=0)
    buf = trace.start(h, depth)
    xs_all = [inputs.allreduce_inputs(2, R, n, dtype, "uniform", c) for c in range(C)]
    ins = [[to_dev(x, dtype) for x in xs] for xs in xs_all]
    outs = [[torch.empty_like(t) for t in row] for row in ins]
    if fused:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        for c in range(C):
            h.allreduce_fused(ins[c], outs[c], s)
        torch.cuda.current_stream().wait_stream(s)
    else:
        g = capture(h, "allreduce", ins, outs, rank_streams(R))
        g.replay()
    torch.cuda.synchronize()
    h.check()
    for c in range(C):
        want = oracle.allreduce(xs_all[c], dtype, ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[c][r]), want, dtype, f"traced call {c} rank {r}")
    rec = trace.records(buf)
    blocks = len(set(rec["block"].tolist()))
    assert 1 <= blocks <= h.info().max_blocks
    assert len(rec) == C * R * blocks
    assert sorted(set(rec["call"].tolist())) == list(range(C))
    assert set(rec["rank"].tolist()) == set(range(R))
    assert set(rec["block"].tolist()) == set(range(blocks))
    assert trace.overlap_violations(rec) == []
    assert (rec["cyc_published"] > 0).all() and (rec["cyc_peers"] >= rec["cyc_published"]).all()
    assert (rec["cyc_end"] >= rec["cyc_peers"]).all() and (rec["t_end_ns"] >= rec["t_start_ns"]).all()
    assert set(rec["algo"].tolist()) == {h.plan("allreduce_fused" if fused else "allreduce", n).algo}
    summary = trace.summarize(rec, sm_clock_mhz=2070.0)
    assert summary["overlap_violations"] == 0 and summary["ranks"] == R
    # tracing off: later calls leave the buffer as it is
    h.set_trace(None, 0)
    before = buf.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    h.allreduce_fused(ins[0], outs[0], s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(before, buf)
    h.destroy()


def test_trace_ring_keeps_the_last_depth_calls():
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import trace
    R, n, depth, calls = 2, 4096, 3, 7
    h = tda.Handle(R, torch.float16, n, "hbm")
    buf = trace.start(h, depth)
    ins = [torch.zeros(n, dtype=torch.float16, device="cuda") for _ in range(R)]
    outs = [torch.empty_like(t) for t in ins]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    for _ in range(calls):
        h.allreduce_fused(ins, outs, s)
    torch.cuda.synchronize()
    h.check()
    rec = trace.records(buf)
    assert sorted(set(rec["call"].tolist())) == list(range(calls - depth, calls))
    with pytest.raises(tda.ArError):
        h.set_trace(buf, 1)   # fewer records than one call needs
    h.destroy()
