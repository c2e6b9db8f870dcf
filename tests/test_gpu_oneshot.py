"""The one-shot form's kernel that publishes one stage ahead, on the GPU.

With slots in HBM and several tiles per block, an untraced one-shot call
publishes stage s + 1 (input, slot stores, flag) before it waits for and
reads its peers' stage s.  Its results must be the oracle's bits for every
rank count, vector count per thread, ragged tail and stage count, per-rank
and in one launch of every rank, both parities, in graphs, and when it
alternates with single-stage calls and other forms on one handle.
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


def _check(outs, xs, dtype, what):
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r, o in enumerate(outs):
        assert_bits_equal(to_bits(o), want, dtype, f"{what} rank {r}")


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
@pytest.mark.parametrize("launch", ["rank", "fused"])
@pytest.mark.parametrize("R,dtype,n,cap", [
    (2, "f16", 256 * 9 * 8 + 3, 4),           # 10 tiles of one vector per thread over 4 blocks
    (2, "bf16", 1 << 21, 0),                  # 4 MiB per rank: two vectors per thread, several stages
    (3, "bf16", 256 * 8 * 7 - 1, 3),
    (4, "f16", (1 << 19) + 77, 5),
    (8, "bf16", 256 * 8 * 5 + 9, 2),
])
def test_multi_stage_one_shot_matches_oracle(slots, launch, R, dtype, n, cap):
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, TORCH[dtype], n, slots)
    h.set_algo("oneshot")
    h.set_tactics(max_blocks=cap, cluster_max_bytes=0)
    p = h.plan("allreduce_fused" if launch == "fused" else "allreduce", n)
    assert p.tiles > p.blocks                 # several stages for block 0
    streams = rank_streams(R)
    side = torch.cuda.Stream()
    for c in range(2):                        # both slot parities
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 7 * c + R)
        ins = [to_dev(x, dtype) for x in xs]
        outs = [torch.full_like(t, float("nan")) for t in ins]
        if launch == "rank":
            enqueue(h, "allreduce", ins, outs, streams)
        else:
            side.wait_stream(torch.cuda.current_stream())
            h.allreduce_fused(ins, outs, side)
            torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        h.check()
        _check(outs, xs, dtype, f"{slots} {launch} R={R} n={n} cap={cap} call {c}")
    h.destroy()


def test_ahead_and_single_stage_calls_alternate_in_a_graph():
    """Multi-stage one-shot calls (published ahead), single-stage ones and
    two-shot ones in one graph on one HBM handle, replayed with new inputs."""
    import tensor_decode_all_gb300 as tda
    R, dtype = 2, "bf16"
    big = 256 * 8 * 11 + 5
    h = tda.Handle(R, TORCH[dtype], big, "hbm")
    h.set_tactics(max_blocks=3)
    streams = rank_streams(R)
    ns = [big, 1000, big - 300, 20001, big]
    algos = ["oneshot", "oneshot", "oneshot", "twoshot", "oneshot"]
    ins = [[torch.empty(m, dtype=TORCH[dtype], device="cuda") for _ in range(R)] for m in ns]
    outs = [[torch.empty_like(t) for t in row] for row in ins]
    g = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream()
    cap_stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(g, stream=cap_stream):
            cur = torch.cuda.current_stream()
            for s in streams:
                s.wait_stream(cur)
            for c, m in enumerate(ns):
                h.set_algo(algos[c])
                for r in range(R):
                    h.allreduce(r, ins[c][r], outs[c][r], streams[r])
            for s in streams:
                cur.wait_stream(s)
    torch.cuda.current_stream().wait_stream(cap_stream)
    for rep in range(2):
        xs = [inputs.allreduce_inputs(5, R, m, dtype, "normal", 500 * rep + c) for c, m in enumerate(ns)]
        for c in range(len(ns)):
            for r in range(R):
                ins[c][r].copy_(to_dev(xs[c][r], dtype))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(len(ns)):
            _check(outs[c], xs[c], dtype, f"replay {rep} call {c} ({algos[c]}, n={ns[c]})")
    del g
    h.destroy()
