"""Pacing of the first stage's slot stores over the host link (the pace_mbs
tactics) on the GPU.

Pacing only delays when each block of a call starts its slot stores, so
every output must stay bit-identical to the CPU oracle whatever the pace:
one-shot and two-shot forms, per-rank launches, one launch of every rank
(cooperative flag form and cluster form), single-stage and multi-stage calls,
ragged tails, both slot parities, graph replay, and paces from the slowest
the tactic accepts to far faster than the link.  The tactics themselves are
checked against the rule the plan reports.
"""
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, capture, enqueue, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}
NEVER = (1 << 64) - 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def test_defaults_rule_and_declines():
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    h = tda.Handle(2, torch.float16, 4 << 20, "pinned")
    t = h.tactics()
    assert (t["pace_mbs"], t["pace_multi_mbs"], t["pace_min_bytes"]) == (356000, 220000, 128 << 10)
    single = h.plan("allreduce", 131072)          # 256 KiB per rank: one 4 KiB tile per block
    assert single.tiles <= single.blocks and single.pace_cycles > 0
    multi = h.plan("allreduce", 2 << 20)          # 4 MiB per rank: several stages per block
    assert multi.tiles > multi.blocks and multi.pace_cycles > 0
    # same tile size, slower pace for multi-stage calls: proportionally longer delay
    ratio = (multi.pace_cycles / multi.tile_bytes) / (single.pace_cycles / single.tile_bytes)
    assert abs(ratio - 356000 / 220000) < 0.02, ratio
    assert h.plan("allreduce", 65536 - 8).pace_cycles == 0          # below 128 KiB per rank
    assert h.plan("allreduce", 65536).pace_cycles > 0               # exactly 128 KiB
    h.set_tactics(pace_min_bytes=0)
    assert h.plan("allreduce", 32768).pace_cycles > 0                # 64 KiB, one-shot
    h.set_tactics(pace_mbs=0)
    assert h.plan("allreduce", 131072).pace_cycles == 0
    assert h.plan("allreduce", 2 << 20).pace_cycles > 0              # multi-stage pace still set
    h.set_tactics(pace_mbs=178000)
    assert abs(h.plan("allreduce", 131072).pace_cycles / single.pace_cycles - 2.0) < 0.02
    for bad in ({"pace_mbs": 999}, {"pace_multi_mbs": 1}, {"pace_mbs": -5}):
        with pytest.raises(ar.ArError):
            h.set_tactics(**bad)
    assert h.tactics()["pace_mbs"] == 178000                         # a refused change leaves the tactics
    h.destroy()
    # two-shot share 1 / 3 (the first stage's stores of W + Rd = 3RS); one-shot share 1 / R
    g = tda.Handle(4, torch.bfloat16, 1 << 20, "pinned")
    g.set_tactics(pace_multi_mbs=356000)           # one pace whether a call takes one stage or several
    p2 = g.plan("allreduce", 1 << 19)              # 1 MiB per rank: two-shot at R = 4 over the host link
    assert p2.subtile_vecs > 0 and p2.pace_cycles > 0
    g.set_algo("oneshot")
    p1 = g.plan("allreduce", 1 << 19)
    per_byte_2 = p2.pace_cycles / p2.tile_bytes
    per_byte_1 = p1.pace_cycles / p1.tile_bytes
    assert abs(per_byte_1 / per_byte_2 - (1 / 3) / (1 / 4)) < 0.03, (per_byte_1, per_byte_2)
    g.destroy()
    # HBM slots are never paced, whatever the tactics say
    k = tda.Handle(2, torch.float16, 1 << 20, "hbm")
    assert k.tactics()["pace_mbs"] == 0 and k.tactics()["pace_multi_mbs"] == 0
    k.set_tactics(pace_mbs=356000, pace_multi_mbs=220000, pace_min_bytes=0)
    assert k.plan("allreduce", 131072).pace_cycles == 0
    k.destroy()


@pytest.mark.parametrize("pace", [0, 2000, 178000, 356000, 4000000])
@pytest.mark.parametrize("R,dtype,n,algo", [
    (2, "f16", 131072, "oneshot"),          # the 256 KiB payload cap, one tile per block
    (2, "bf16", (1 << 20) + 5, "oneshot"),  # several stages per block, ragged tail
    (4, "bf16", 262144 + 3, "twoshot"),
    (8, "f16", 131072, "twoshot"),
    (3, "bf16", 65536 + 11, "oneshot"),
])
def test_paced_per_rank_calls_match_oracle(pace, R, dtype, n, algo):
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, TORCH[dtype], n, "pinned")
    h.set_algo(algo)
    h.set_tactics(pace_mbs=pace, pace_multi_mbs=pace, pace_min_bytes=0)
    assert (h.plan("allreduce", n).pace_cycles > 0) == (pace > 0)
    streams = rank_streams(R)
    for call in range(2):                      # both slot parities
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 10 * call + R)
        ins = [to_dev(x, dtype) for x in xs]
        outs = [torch.full_like(t, float("nan")) for t in ins]
        enqueue(h, "allreduce", ins, outs, streams)
        torch.cuda.synchronize()
        h.check()
        want = oracle.allreduce(xs, dtype, ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[r]), want, dtype, f"pace={pace} R={R} n={n} {algo} call {call} rank {r}")
    h.destroy()


@pytest.mark.parametrize("form", ["cluster", "flags"])
@pytest.mark.parametrize("R,n", [(2, 131072), (2, 524288 + 1), (4, 131072 + 7), (8, 65536)])
def test_paced_launches_of_every_rank_match_oracle(form, R, n):
    """One launch of every rank: the cluster form (paced while one wave of
    clusters holds the call) and the cooperative flag form."""
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, torch.bfloat16, n, "pinned")
    if form == "cluster":
        if h.info().cluster_form < 1:
            pytest.skip("cluster launches unavailable")
        h.set_algo("cluster")
    else:
        h.set_tactics(cluster_max_bytes=0)
    h.set_tactics(pace_min_bytes=0)
    p = h.plan("allreduce_fused", n)
    assert p.algo == (3 if form == "cluster" else p.algo)
    if form == "flags" or p.blocks <= h.info().cluster_form:
        assert p.pace_cycles > 0
    s = torch.cuda.Stream()
    for call in range(2):
        xs = inputs.allreduce_inputs(5, R, n, "bf16", "normal4", call)
        ins = [to_dev(x, "bf16") for x in xs]
        outs = [torch.full_like(t, float("nan")) for t in ins]
        s.wait_stream(torch.cuda.current_stream())
        h.allreduce_fused(ins, outs, s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        h.check()
        want = oracle.allreduce(xs, "bf16", ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[r]), want, "bf16", f"{form} R={R} n={n} call {call} rank {r}")
    h.destroy()


def test_paced_headline_calls_replay_in_a_graph():
    """The 256 KiB payload cap at its default pace, 20 calls per graph with
    fresh inputs in each, replayed with new inputs: every call of every
    replay equals the oracle."""
    import tensor_decode_all_gb300 as tda
    R, n, C = 2, 131072, 20
    h = tda.Handle(R, torch.float16, n, "pinned")
    assert h.plan("allreduce", n).pace_cycles > 0
    ins = [[torch.empty(n, dtype=torch.float16, device="cuda") for _ in range(R)] for _ in range(C)]
    outs = [[torch.empty_like(t) for t in row] for row in ins]
    g = capture(h, "allreduce", ins, outs, rank_streams(R))
    for rep in range(2):
        xs = [inputs.allreduce_inputs(2, R, n, "f16", "normal4", 1000 * rep + c) for c in range(C)]
        for c in range(C):
            for r in range(R):
                ins[c][r].copy_(to_dev(xs[c][r], "f16"))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(C):
            want = oracle.allreduce(xs[c], "f16", ranks=[0])[0]
            for r in range(R):
                assert_bits_equal(to_bits(outs[c][r]), want, "f16", f"replay {rep} call {c} rank {r}")
    del g
    h.destroy()


@pytest.mark.parametrize("pace", [0, 2000, 220000, 4000000])
@pytest.mark.parametrize("R,n", [(3, 1000 * 37 + 5), (4, 1000 * 500)])
def test_paced_allgather_matches_oracle(pace, R, n):
    """The allgather over the host link, paced as the one-shot form (the same
    link bytes): byte-exact against the oracle's concatenation, per-rank and
    in one launch of every rank, at paces from 2 GB/s to far faster than the
    link and none; several stages per block at the config-4 shard size."""
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, torch.complex64, n, "pinned")
    h.set_tactics(pace_mbs=pace, pace_multi_mbs=pace, pace_min_bytes=0)
    assert (h.plan("allgather", n).pace_cycles > 0) == (pace > 0)
    streams = rank_streams(R)
    for call, launch in enumerate(("rank", "fused")):
        zs = inputs.allgather_inputs(4, R, n, 20 + call)
        ins = [to_dev(z, "c64") for z in zs]
        outs = [torch.empty(R * n, dtype=torch.complex64, device="cuda") for _ in range(R)]
        if launch == "rank":
            enqueue(h, "allgather", ins, outs, streams)
        else:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            h.allgather_fused(ins, outs, s)
            torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        h.check()
        want = oracle.allgather(zs, ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[r]), want, "c64", f"pace={pace} R={R} {launch} rank {r}")
    h.destroy()
