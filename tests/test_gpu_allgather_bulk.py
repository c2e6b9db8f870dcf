"""The allgather's bulk-gather kernel on the GPU (slots in HBM, R >= 5,
16-byte vectors): each block's thread 0 moves its peers' tiles with bulk
asynchronous copies through shared memory.  Byte-exact against the oracle's
concatenation for R = 5..8, one and several stages per block, a last tile
cut short, per-rank launches and one launch of every rank, both slot
parities, graph replay, mixed with sizes that take the per-thread kernel on
one handle; and a rank that never launches still ends in a recorded timeout.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, capture, enqueue, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _gather(h, R, n, launch, seed):
    zs = inputs.allgather_inputs(4, R, n, seed)
    ins = [to_dev(z, "c64") for z in zs]
    outs = [torch.full((R * n,), float("nan"), dtype=torch.complex64, device="cuda") for _ in range(R)]
    if launch == "rank":
        enqueue(h, "allgather", ins, outs, rank_streams(R))
    else:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        h.allgather_fused(ins, outs, s)
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    h.check()
    return zs, outs


def _check(zs, outs, what):
    want = oracle.allgather(zs, ranks=[0])[0]
    for r, o in enumerate(outs):
        assert_bits_equal(to_bits(o), want, "c64", f"{what} rank {r}")


@pytest.mark.parametrize("launch", ["rank", "fused"])
@pytest.mark.parametrize("R,n,cap", [
    (5, 2 * 1000 + 2, 0),               # even count: 16-byte vectors, one stage, a short last tile
    (6, 256 * 2 * 9 + 64, 2),           # several stages per block, short last tile
    (7, 256 * 2 * 4, 0),                # whole tiles only
    (8, 1000 * 500, 0),                 # the config-4 shard: several stages per block
    (8, 256 * 2 * 13 + 2, 3),           # several stages on 3 blocks, blocks of different stage counts
])
def test_bulk_gather_matches_oracle(launch, R, n, cap):
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, torch.complex64, n, "hbm")
    h.set_tactics(max_blocks=cap)
    for call in range(2):                            # both slot parities
        zs, outs = _gather(h, R, n, launch, 40 + call)
        _check(zs, outs, f"bulk {launch} R={R} n={n} cap={cap} call {call}")
    h.destroy()


def test_bulk_and_per_thread_kernels_alternate_on_one_handle_and_in_a_graph():
    """An odd element count takes 8-byte vectors (the per-thread kernel), an
    even one the bulk kernel; calls of both, eagerly and in one graph."""
    import tensor_decode_all_gb300 as tda
    R, nmax = 8, 256 * 2 * 20 + 3
    h = tda.Handle(R, torch.complex64, nmax, "hbm")
    for i, n in enumerate([nmax - 1, nmax, 1001, 4096, nmax - 3, 2]):
        zs, outs = _gather(h, R, n, "rank", 70 + i)
        _check(zs, outs, f"eager step {i} n={n}")
    ns = [nmax - 1, 999, 4096]
    ins = [[torch.empty(m, dtype=torch.complex64, device="cuda") for _ in range(R)] for m in ns]
    outs = [[torch.empty(R * m, dtype=torch.complex64, device="cuda") for _ in range(R)] for m in ns]
    g = capture(h, "allgather", ins, outs, rank_streams(R))
    for rep in range(3):
        zs = [inputs.allgather_inputs(4, R, m, 500 + 10 * rep + c) for c, m in enumerate(ns)]
        for c in range(len(ns)):
            for r in range(R):
                ins[c][r].copy_(to_dev(zs[c][r], "c64"))
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(len(ns)):
            _check(zs[c], outs[c], f"graph replay {rep} call {c}")
    del g
    h.destroy()


def test_bulk_gather_missing_rank_times_out_and_reset_restores():
    """Ranks 0..6 of 8 launched, rank 7 never: the flag waits run out, the
    bulk kernel leaves after its own copies have completed, the handle
    records the timeout, and after a reset a full call is byte-exact."""
    import tensor_decode_all_gb300 as tda
    from tensor_decode_all_gb300 import ar
    R, n = 8, 256 * 2 * 6
    h = tda.Handle(R, torch.complex64, n, "hbm")
    h.set_timeout(50_000_000)                         # 50 ms
    streams = rank_streams(R)
    zs = inputs.allgather_inputs(4, R, n, 9)
    ins = [to_dev(z, "c64") for z in zs]
    outs = [torch.empty(R * n, dtype=torch.complex64, device="cuda") for _ in range(R)]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for r in range(R - 1):
        h.allgather(r, ins[r], outs[r], streams[r])
    for s in streams[:-1]:
        s.synchronize()
    dt = time.perf_counter() - t0
    st = h.status()
    assert st.code == ar.AR_ETIMEOUT and st.peer == R - 1, (st.code, st.peer)
    assert 0.04 < dt < 5.0, dt
    h.reset()
    zs, outs = _gather(h, R, n, "rank", 10)
    _check(zs, outs, "after reset")
    h.destroy()
