"""The two-shot form's kernels on the GPU: merged flag rounds and prefetch.

With slots in HBM and several tiles per block, an untraced two-shot call runs
the kernel in which each rank's reduced sub-tile rides on the next tile's
flag round and the next tile's input is copied into shared memory while the
flags are awaited.  Every other two-shot call (host-memory slots, one tile
per block, traced) runs the kernel of two rounds per tile.  Both must give
the oracle's bits for every rank count, sub-tile size and ragged tail, for
blocks of different stage counts in one call, per-rank and in one launch of
every rank, both slot parities, graph replay, and when calls of the two
kernels (and other forms) alternate on one handle.
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


def _run(h, R, n, dtype, launch, calls, what, seed0=0):
    streams = rank_streams(R)
    side = torch.cuda.Stream()
    for c in range(calls):
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", seed0 + c)
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
        _check(outs, xs, dtype, f"{what} call {c}")


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
@pytest.mark.parametrize("launch", ["rank", "fused"])
@pytest.mark.parametrize("sub", [64, 128, 256])
@pytest.mark.parametrize("R,dtype", [(3, "bf16"), (4, "f16"), (5, "bf16"), (8, "bf16"), (8, "f16")])
def test_multi_stage_two_shot_matches_oracle(slots, launch, sub, R, dtype):
    """A block cap of 3 spreads 7-11 tiles over 3 blocks, so block 0 runs more
    stages than block 2, and the ragged tail ends inside the last tile."""
    import tensor_decode_all_gb300 as tda
    tile = R * sub * 8                           # elements per tile
    n = 10 * tile + 8 * sub + 5
    h = tda.Handle(R, TORCH[dtype], n, slots)
    h.set_algo("twoshot")
    h.set_tactics(twoshot_sub=sub, max_blocks=3, cluster_max_bytes=0)
    p = h.plan("allreduce_fused" if launch == "fused" else "allreduce", n)
    assert p.subtile_vecs == sub and p.blocks == 3 and p.max_stages == 4
    _run(h, R, n, dtype, launch, 2, f"{slots} {launch} sub={sub} R={R} n={n}")
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
def test_one_and_several_stages_alternate_on_one_handle(slots):
    """Single-stage calls (two rounds), multi-stage calls (merged rounds in
    HBM), one-shot and tagged calls, in one sequence on one handle and then in
    one graph: the stage counters every kernel shares stay consistent."""
    import tensor_decode_all_gb300 as tda
    R, dtype = 8, "bf16"
    big = 8 * 256 * 8 * 12 + 3                # 12 tiles of 256-vector sub-tiles, ragged
    h = tda.Handle(R, TORCH[dtype], big, slots)
    sizes = [(big, "twoshot", 4), (3000, "twoshot", 0), (big, "twoshot", 5), (70001, "oneshot", 0),
             (big - 4099, "twoshot", 3), (2048, "auto", 0), (big, "twoshot", 0)]
    streams = rank_streams(R)
    for i, (n, algo, cap) in enumerate(sizes):
        h.set_algo(algo)
        h.set_tactics(max_blocks=cap)
        xs = inputs.allreduce_inputs(5, R, n, dtype, "normal", 100 + i)
        ins = [to_dev(x, dtype) for x in xs]
        outs = [torch.full_like(t, float("nan")) for t in ins]
        enqueue(h, "allreduce", ins, outs, streams)
        torch.cuda.synchronize()
        h.check()
        _check(outs, xs, dtype, f"{slots} step {i} n={n} {algo} cap={cap}")
    # the same mix captured in one graph (tactics are frozen per call at capture)
    h.set_algo("twoshot")
    h.set_tactics(max_blocks=4)
    C = 6
    ns = [big, 3000, big - 4099, big, 70001, big]
    ins = [[torch.empty(m, dtype=TORCH[dtype], device="cuda") for _ in range(R)] for m in ns]
    outs = [[torch.empty_like(t) for t in row] for row in ins]
    g = capture(h, "allreduce", ins, outs, streams)
    for rep in range(2):
        xs = [inputs.allreduce_inputs(5, R, ns[c], dtype, "uniform", 1000 * rep + c) for c in range(C)]
        for c in range(C):
            for r in range(R):
                ins[c][r].copy_(to_dev(xs[c][r], dtype))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(C):
            _check(outs[c], xs[c], dtype, f"{slots} graph replay {rep} call {c}")
    del g
    h.destroy()


def test_traced_multi_stage_calls_take_the_two_round_kernel_and_match():
    """A traced call never takes the merged kernel; its bits and its trace
    records (one per block, the block's stage count) are right either way."""
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import trace
    R, dtype = 8, "bf16"
    n = 8 * 256 * 8 * 7 - 5                      # 7 tiles, the last vector partial
    h = tda.Handle(R, TORCH[dtype], n, "hbm")
    h.set_algo("twoshot")
    h.set_tactics(max_blocks=2, twoshot_sub=256)
    buf = trace.start(h, 4)
    _run(h, R, n, dtype, "rank", 2, "traced")
    rec = trace.records(buf)
    rec = rec[rec["stages"] > 0]
    assert len(rec) == 2 * R * 2                          # 2 calls x R ranks x 2 blocks
    assert sorted(set(rec["stages"].tolist())) == [3, 4]  # 7 tiles over 2 blocks: 4 and 3 stages
    h.set_trace(None, 0)
    _run(h, R, n, dtype, "rank", 2, "untraced after traced", seed0=50)
    h.destroy()
