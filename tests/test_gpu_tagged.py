"""GPU parity of the tagged-word all-reduce form (AR_ALGO_TAGGED).

Each 8-byte word of the exchange buffer carries 4 payload bytes and a 4-byte
tag naming the stage; readers poll their peers' words until the tags match.
The arithmetic is the same rank-order fp32 sum with one rounding, so every
output must equal the CPU oracle bit for bit, as for the flag forms.
"""
import time

import numpy as np
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


def _handle(R, dtype, n, slots, algo="tagged"):
    import tensor_decode_all_gb300 as tda
    h = tda.Handle(R, TORCH[dtype], n, slots)
    if algo:
        h.set_algo(algo)
    return h


def _check(outs, xs, dtype, what):
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r, o in enumerate(outs):
        assert_bits_equal(to_bits(o), want, dtype, f"{what} rank {r}")


@pytest.mark.parametrize("slots", ["pinned", "hbm"])
@pytest.mark.parametrize("R,dtype,n", [
    (2, "f16", 4096),          # one decode token, hidden 4096
    (2, "f16", 4099),          # ragged tail
    (2, "f16", 131072),        # 256 KiB
    (8, "bf16", 393216 // 4),  # 192 KiB per rank
    (8, "bf16", 8191),
    (4, "bf16", 262144),       # 512 KiB per rank: 128 blocks of one tile
    (3, "f16", 1000),
    (1, "bf16", 77),
    (2, "f16", 1),
])
def test_tagged_matches_oracle(R, dtype, n, slots):
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 9)
    h = _handle(R, dtype, n, slots)
    assert h.plan("allreduce", n).algo == 2
    ins = [to_dev(x, dtype) for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    streams = rank_streams(R)
    for call in range(3):      # both buffer parities, then the first again
        enqueue(h, "allreduce", ins, outs, streams)
        torch.cuda.synchronize()
        h.check()
        _check(outs, xs, dtype, f"tagged R={R} {dtype} n={n} {slots} call {call}")
    h.destroy()


def test_tagged_beyond_capacity_takes_the_oneshot_form():
    h = _handle(2, "f16", 1 << 20, "hbm")
    info = h.info()
    cap = info.tagged_capacity_bytes
    # one 4 KiB tile per block of one rank's launch
    assert cap % 4096 == 0 and cap // 4096 <= info.max_blocks and cap >= 512 << 10
    assert h.plan("allreduce", cap // 2).algo == 2
    assert h.plan("allreduce", cap // 2 + 8).algo == 0
    xs = inputs.allreduce_inputs(5, 2, cap // 2 + 8, "f16", "uniform", 4)
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    enqueue(h, "allreduce", ins, outs, rank_streams(2))
    torch.cuda.synchronize()
    h.check()
    _check(outs, xs, "f16", "beyond capacity")
    h.destroy()


@pytest.mark.parametrize("slots", ["pinned", "hbm"])
def test_tagged_graph_replay_fresh_inputs(slots):
    """Workload 1's shape in a graph of C calls per rank, inputs refilled
    between replays: tags and parities stay right across replays."""
    R, n, C = 2, 4096, 10
    h = _handle(R, "f16", n, slots)
    streams = rank_streams(R)
    ins = [[torch.empty(n, dtype=torch.float16, device="cuda") for _ in range(R)] for _ in range(C)]
    outs = [[torch.empty(n, dtype=torch.float16, device="cuda") for _ in range(R)] for _ in range(C)]
    g = capture(h, "allreduce", ins, outs, streams)
    for rep in range(4):
        xs_all = []
        for c in range(C):
            xs = inputs.allreduce_inputs(1, R, n, "f16", "uniform", rep * C + c)
            for r in range(R):
                ins[c][r].copy_(to_dev(xs[r], "f16"))
            xs_all.append(xs)
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(C):
            _check(outs[c], xs_all[c], "f16", f"rep {rep} call {c}")
    del g
    h.destroy()


def test_tagged_interleaves_with_the_flag_forms():
    """Tagged, one-shot and two-shot calls alternate on one handle."""
    R, n, dtype = 8, 65536, "bf16"
    h = _handle(R, dtype, n, "hbm", algo=None)
    streams = rank_streams(R)
    for call, algo in enumerate(["tagged", "oneshot", "tagged", "twoshot", "twoshot", "tagged", "oneshot"]):
        h.set_algo(algo)
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 50 + call)
        ins = [to_dev(x, dtype) for x in xs]
        outs = [torch.empty_like(t) for t in ins]
        enqueue(h, "allreduce", ins, outs, streams)
        torch.cuda.synchronize()
        h.check()
        _check(outs, xs, dtype, f"call {call} ({algo})")
    h.destroy()


def test_tagged_fused_launch():
    R, n, dtype = 8, 4096, "bf16"
    h = _handle(R, dtype, n, "hbm")
    s = torch.cuda.Stream()
    for call in range(3):
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 70 + call)
        ins = [to_dev(x, dtype) for x in xs]
        outs = [torch.empty_like(t) for t in ins]
        s.wait_stream(torch.cuda.current_stream())
        h.allreduce_fused(ins, outs, s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        h.check()
        _check(outs, xs, dtype, f"fused tagged call {call}")
    h.destroy()


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tagged_special_values(dtype):
    """Payload words pass through the tagged buffer untouched: signed zeros,
    infinities, NaN, subnormals, overflow to infinity."""
    R, n = 2, 64
    if dtype == "f16":
        specials = np.array([0x0000, 0x8000, 0x7C00, 0xFC00, 0x7E00, 0x0001, 0x8001, 0x7BFF], np.uint16)
    else:
        specials = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001, 0x7F7F], np.uint16)
    a = np.resize(specials, n)
    b = np.resize(specials[::-1], n)
    h = _handle(R, dtype, n, "pinned")
    ins = [to_dev(a, dtype), to_dev(b, dtype)]
    outs = [torch.empty_like(t) for t in ins]
    enqueue(h, "allreduce", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    h.check()
    _check(outs, [a, b], dtype, "specials")
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
def test_tagged_missing_peer_times_out_and_reset_restores(slots):
    """Only rank 0 of two is launched: its threads poll words nothing writes,
    give up after the limit, record AR_ETIMEOUT and return."""
    import tensor_decode_all_gb300 as tda
    ar = tda.ar
    R, n = 2, 8192
    h = _handle(R, "f16", n, slots)
    h.set_timeout(50_000_000)
    streams = rank_streams(R)
    xs = inputs.allreduce_inputs(5, R, n, "f16", "uniform", 12)
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty_like(t) for t in ins]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    h.allreduce(0, ins[0], outs[0], streams[0])
    streams[0].synchronize()
    dt = time.perf_counter() - t0
    st = h.status()
    assert st.code == ar.AR_ETIMEOUT and st.rank == 0 and st.peer == 1 and st.want >= 1
    assert 0.04 < dt < 5.0, dt
    h.reset()
    enqueue(h, "allreduce", ins, outs, streams)
    torch.cuda.synchronize()
    h.check()
    _check(outs, xs, "f16", "after reset")
    h.destroy()


def test_tagged_with_changing_grids_stays_exact():
    """Calls whose grid changes between calls (a block cap, one launch of all
    ranks) on one handle.  The tagged form runs one tile per block and keeps
    each buffer position to one block index, so a word left by another block
    of an earlier call can never pass for this call's; a call that would need
    a second stage per block takes the one-shot form instead."""
    R, dtype = 2, "f16"
    h = _handle(R, dtype, 8192, "hbm")
    streams = rank_streams(R)
    fs = torch.cuda.Stream()
    # (elements, block cap, fused): 1 tile / 1 block, 4 tiles / 3 blocks,
    # 4 tiles / 2 blocks -- the grid sequence that lets a stale word carry an
    # expected tag when the buffer is indexed by payload vector -- then more.
    seq = [(2048, 1, False), (8192, 3, False), (8192, 2, False), (8192, 0, True), (2048, 1, True),
           (8192, 0, False), (6144, 2, False), (8192, 4, True), (8192, 0, False)] * 3
    for call, (n, cap, fused) in enumerate(seq):
        h.set_tactics(max_blocks=cap)
        tiles = -(-n // 2048)
        assert h.plan("allreduce", n).algo == (2 if (cap == 0 or tiles <= cap) else 0)
        xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 300 + call)
        ins = [to_dev(x, dtype) for x in xs]
        outs = [torch.empty_like(t) for t in ins]
        if fused:
            fs.wait_stream(torch.cuda.current_stream())
            h.allreduce_fused(ins, outs, fs)
            torch.cuda.current_stream().wait_stream(fs)
        else:
            enqueue(h, "allreduce", ins, outs, streams)
        torch.cuda.synchronize()
        h.check()
        _check(outs, xs, dtype, f"call {call} n={n} cap={cap} fused={fused}")
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
@pytest.mark.parametrize("algo", ["tagged", "oneshot", "twoshot"])
def test_stage_counts_across_the_32_bit_wrap(slots, algo):
    """Stage counts seeded just below 2^32 - 1 (the tag period) and 2^32 (where
    the low 32 bits of a count are 0): the tagged words' tags wrap from
    2^32 - 1 to 1 and never take the value 0 of the zeroed buffer, and the flag
    forms' 64-bit counts run on; every call stays exact."""
    R, n, dtype = 2, 8192, "f16"
    for seed in ((1 << 32) - 4, (1 << 32) - 1, (1 << 32) + 3):
        h = _handle(R, dtype, n, slots, algo=algo)
        h.debug_seed_stages(seed)
        streams = rank_streams(R)
        for call in range(8):
            xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 400 + call)
            ins = [to_dev(x, dtype) for x in xs]
            outs = [torch.empty_like(t) for t in ins]
            enqueue(h, "allreduce", ins, outs, streams)
            torch.cuda.synchronize()
            h.check()
            _check(outs, xs, dtype, f"{algo} {slots} seed {seed:#x} call {call}")
        h.destroy()
