"""The scope at which the ranks of a pinned-host handle synchronise (the
gpu_scope tactic) on the GPU.

With slots in host memory the ranks synchronise either at system scope, the
flags in mapped host memory (two GPUs sharing only the host buffer need
that), or at GPU scope, the flags in HBM and the tagged words and push flags
read and written at GPU scope (every rank is a kernel of this GPU).  The slot
data crosses the host link either way, so every form -- one-shot, two-shot
with one and several stages per block, tagged words, push, the allgather,
per-rank launches and one cooperative launch of every rank -- must give the
oracle's bits with both scopes, when calls switch scope on one handle
(eagerly and in graphs captured under each), and a missing peer must still
time out and record itself.
"""
import time

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


def _allreduce(h, R, n, dtype, seed, launch="rank"):
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", seed)
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.full_like(t, float("nan")) for t in ins]
    if launch == "rank":
        enqueue(h, "allreduce", ins, outs, rank_streams(R))
    else:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        h.allreduce_fused(ins, outs, s)
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    h.check()
    return xs, outs


def _check(xs, outs, dtype, what):
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r, o in enumerate(outs):
        assert_bits_equal(to_bits(o), want, dtype, f"{what} rank {r}")


def test_tactic_defaults_and_refusals():
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    h = tda.Handle(2, torch.float16, 4096, "pinned")
    assert h.tactics()["gpu_scope"] == 1             # the default
    for v in (0, 1):
        h.set_tactics(gpu_scope=v)
        assert h.tactics()["gpu_scope"] == v
    with pytest.raises(ar.ArError):
        h.set_tactics(gpu_scope=2)
    assert h.tactics()["gpu_scope"] == 1
    h.destroy()
    k = tda.Handle(2, torch.float16, 4096, "hbm")
    assert k.tactics()["gpu_scope"] == 1          # HBM handles: always GPU scope
    k.set_tactics(gpu_scope=1)
    with pytest.raises(ar.ArError):
        k.set_tactics(gpu_scope=0)
    k.destroy()


@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("launch", ["rank", "fused"])
@pytest.mark.parametrize("R,dtype,n,algo,cap", [
    (2, "f16", 131072, "oneshot", 0),            # the 256 KiB payload cap: one tile per block, paced
    (2, "bf16", (1 << 20) + 5, "oneshot", 0),    # several stages per block, ragged tail
    (3, "f16", 70001, "oneshot", 0),
    (4, "bf16", 262144 + 3, "twoshot", 0),       # two rounds per tile
    (8, "f16", 8 * 256 * 8 * 5 + 77, "twoshot", 2),  # several tiles per block of 2
    (2, "f16", 4096, "tagged", 0),               # one decode token: tagged words, no flag
    (8, "bf16", 20000 + 3, "tagged", 0),
    (2, "bf16", 65536 + 9, "push", 0),
    (4, "f16", 30000 + 1, "push", 0),
])
def test_allreduce_matches_oracle_with_either_scope(flags, launch, R, dtype, n, algo, cap):
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, TORCH[dtype], n, "pinned")
    h.set_algo(algo)
    h.set_tactics(gpu_scope=flags, max_blocks=cap, cluster_max_bytes=0)
    from tensor_decode_all_gb300 import ar
    assert h.plan("allreduce_fused" if launch == "fused" else "allreduce", n).algo == ar.ALGOS[algo]
    for call in range(2):                        # both slot parities
        xs, outs = _allreduce(h, R, n, dtype, 10 * call + R + flags, launch)
        _check(xs, outs, dtype, f"flags={flags} {launch} R={R} n={n} {algo} call {call}")
    h.destroy()


@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("R,n", [(3, 1000 * 37 + 5), (4, 1000 * 500)])
def test_allgather_matches_oracle_with_either_scope(flags, R, n):
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, torch.complex64, n, "pinned")
    h.set_tactics(gpu_scope=flags)
    streams = rank_streams(R)
    for call, launch in enumerate(("rank", "fused", "rank")):
        zs = inputs.allgather_inputs(4, R, n, 40 + call + flags)
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
            assert_bits_equal(to_bits(outs[r]), want, "c64", f"flags={flags} R={R} {launch} call {call} rank {r}")
    h.destroy()


def test_calls_switch_scope_on_one_handle_eagerly_and_in_graphs():
    """The stage counts go on from the per-block counters, whichever flag
    array a call uses: the array a call switches to holds older (smaller)
    counts, which never pass for the current stage; the tagged words carry
    the stage tag whatever the scope.  Graphs captured under each scope keep
    theirs when replayed in turn."""
    import tensor_decode_all_gb300 as tda
    R, dtype = 4, "bf16"
    n_big = 4 * 256 * 8 * 18 + 13                # 18 tiles of 256-vector sub-tiles, above 131072
    h = tda.Handle(R, TORCH[dtype], n_big, "pinned")
    steps = [(1, n_big, "twoshot"), (0, 3001, "oneshot"), (1, 131072, "oneshot"), (1, 5000, "auto"),
             (0, n_big, "twoshot"), (0, 131072, "oneshot"), (1, n_big - 999, "twoshot"), (0, 77, "oneshot"),
             (0, 4096, "tagged"), (1, 4096, "tagged"), (0, 6000, "push"), (1, 6000, "push"), (0, 4096, "tagged")]
    for i, (flags, n, algo) in enumerate(steps):
        h.set_algo(algo)
        h.set_tactics(gpu_scope=flags, max_blocks=3 if algo == "twoshot" else 0)
        xs, outs = _allreduce(h, R, n, dtype, 300 + i)
        _check(xs, outs, dtype, f"step {i} flags={flags} n={n} {algo}")
    h.set_algo("auto")
    h.set_tactics(max_blocks=0)
    streams = rank_streams(R)
    graphs = []
    ns = [131072, n_big, 2048]
    for flags in (1, 0):
        h.set_tactics(gpu_scope=flags)
        ins = [[torch.empty(m, dtype=TORCH[dtype], device="cuda") for _ in range(R)] for m in ns]
        outs = [[torch.empty_like(t) for t in row] for row in ins]
        graphs.append((flags, capture(h, "allreduce", ins, outs, streams), ins, outs))
    h.set_tactics(gpu_scope=1)
    for rep in range(3):
        for flags, g, ins, outs in graphs:
            xs = [inputs.allreduce_inputs(5, R, m, dtype, "normal", 1000 * rep + 10 * flags + c)
                  for c, m in enumerate(ns)]
            for c in range(len(ns)):
                for r in range(R):
                    ins[c][r].copy_(to_dev(xs[c][r], dtype))
            g.replay()
            torch.cuda.synchronize()
            h.check()
            for c in range(len(ns)):
                _check(xs[c], outs[c], dtype, f"replay {rep} graph of flags={flags} call {c}")
        # an eager call between replays, with the scope the handle has now
        xs, outs = _allreduce(h, R, 131072, dtype, 5000 + rep)
        _check(xs, outs, dtype, f"eager after replay {rep}")
    graphs.clear()
    h.destroy()


@pytest.mark.parametrize("flags", [0, 1])
def test_missing_peer_times_out_with_either_scope(flags):
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    R, n = 2, 131072
    h = tda.Handle(R, torch.float16, n, "pinned")
    h.set_algo("oneshot")
    h.set_tactics(gpu_scope=flags)
    h.set_timeout(50_000_000)                    # 50 ms
    streams = rank_streams(R)
    xs = inputs.allreduce_inputs(2, R, n, "f16", "normal4", 7)
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    h.allreduce(0, ins[0], outs[0], streams[0])   # rank 1 never called
    streams[0].synchronize()
    dt = time.perf_counter() - t0
    st = h.status()
    assert st.code == ar.AR_ETIMEOUT and st.rank == 0 and st.peer == 1
    assert st.want >= 1 and st.seen == 0
    assert 0.04 < dt < 5.0, dt
    h.reset()
    xs, outs = _allreduce(h, R, n, "f16", 8)
    _check(xs, outs, "f16", f"flags={flags} after reset")
    h.destroy()
