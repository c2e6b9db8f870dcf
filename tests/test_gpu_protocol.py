"""Slot parity when calls on one handle use different grids.

The slot half a call writes is picked by its blocks' call count.  A call on a
small grid (few tiles, or a form whose tiles are larger) leaves the blocks it
did not launch behind unless they are advanced too; a later call whose tiles
map a slot region to another block index could then write that region in the
half a peer still reads from the call before.  These tests mix grids and forms
in one graph and check every output, and use the device trace to check that
every block of every call counts the same calls.
"""
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


# (elements per rank, form): a two-shot call of one 512-vector tile on one block,
# then one-shot / tagged calls of the same bytes on two blocks, and other sizes.
SEQUENCE = [(4096, "twoshot"), (4096, "oneshot"), (4096, "twoshot"), (4096, "tagged"), (2048, "oneshot"),
            (8192, "oneshot"), (4096, "twoshot"), (8192, "twoshot"), (2048, "tagged"), (8192, "oneshot"),
            (6144, "tagged"), (4096, "oneshot")]


@pytest.mark.parametrize("slots", ["pinned", "hbm"])
def test_mixed_grids_in_one_graph(slots):
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import trace
    R, dtype, nmax = 2, "f16", 8192
    h = tda.Handle(R, torch.float16, nmax, slots)
    buf = trace.start(h, len(SEQUENCE) * 2)
    streams = rank_streams(R)
    ins = [[torch.empty(n, dtype=torch.float16, device="cuda") for _ in range(R)] for n, _ in SEQUENCE]
    outs = [[torch.empty(n, dtype=torch.float16, device="cuda") for _ in range(R)] for n, _ in SEQUENCE]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            cap = torch.cuda.current_stream()
            for s in streams:
                s.wait_stream(cap)
            for c, (n, algo) in enumerate(SEQUENCE):
                h.set_algo(algo)
                for r in range(R):
                    h.allreduce(r, ins[c][r], outs[c][r], streams[r])
            for s in streams:
                cap.wait_stream(s)
    torch.cuda.current_stream().wait_stream(side)
    for rep in range(6):
        xs_all = []
        for c, (n, _) in enumerate(SEQUENCE):
            xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 1000 + rep * 100 + c)
            for r in range(R):
                ins[c][r].copy_(to_dev(xs[r], dtype))
            xs_all.append(xs)
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c, (n, algo) in enumerate(SEQUENCE):
            want = oracle.allreduce(xs_all[c], dtype, ranks=[0])[0]
            for r in range(R):
                assert_bits_equal(to_bits(outs[c][r]), want, dtype, f"{slots} rep {rep} call {c} ({algo}, n={n})")
    # Every block that ran a call counted the same calls before it: the
    # records that carry one call count all come from one call (one form, one
    # record per rank and block, the same blocks on every rank).
    rec = trace.records(buf)
    assert len(rec) > 0
    for call in set(rec["call"].tolist()):
        grp = rec[rec["call"] == call]
        assert len(set(grp["algo"].tolist())) == 1, call
        pairs = list(zip(grp["rank"].tolist(), grp["block"].tolist()))
        assert len(pairs) == len(set(pairs)), call
        blocks = [set(grp[grp["rank"] == r]["block"].tolist()) for r in range(R)]
        assert all(b == blocks[0] for b in blocks), call
    del g
    h.destroy()
