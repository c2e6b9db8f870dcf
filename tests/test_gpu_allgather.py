"""GPU parity of the allgather against the CPU oracle (byte-exact)."""
import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, assert_device_equal, capture, enqueue, rank_streams, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _handle(R, n, slots, dtype=torch.complex64):
    import tensor_decode_all_gb300 as tda
    return tda.Handle(R, dtype, n, slots)


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
@pytest.mark.parametrize("R", [4, 8])
def test_config4_c64_1000x500_graph_1000_calls(R, slots):
    """Workload 4: complex64 1000x500 shards, a graph of 100 calls replayed 10
    times with fresh shards each replay (each rank's base shard rotated per
    call): 1000 calls, every call of every replay compared byte for byte with
    the oracle's concatenation on every rank.  The outputs (R x R x 4 MB per
    call) are compared on the device against the oracle's result uploaded."""
    n, C, REPLAYS = 1000 * 500, 100, 10
    h = _handle(R, n, slots)
    streams = rank_streams(R)
    ins = torch.empty((C, R, n), dtype=torch.complex64, device="cuda")
    outs = torch.empty((C, R, R * n), dtype=torch.complex64, device="cuda")
    g = capture(h, "allgather", [[ins[c, r] for r in range(R)] for c in range(C)],
                [[outs[c, r] for r in range(R)] for c in range(C)], streams)
    checked = 0
    for rep in range(REPLAYS):
        zs_all = [inputs.allgather_inputs_rotated(4, R, n, rep * C + c) for c in range(C)]
        for c in range(C):
            ins[c].copy_(torch.from_numpy(np.stack(zs_all[c])), non_blocking=False)
        outs.view(torch.int32).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        h.check()
        for c in range(C):
            want = torch.from_numpy(oracle.allgather(zs_all[c], ranks=[0])[0]).cuda()
            for r in range(R):
                assert_device_equal(outs[c, r], want, f"R={R} {slots} replay {rep} call {c} rank {r}")
                checked += 1
    assert checked == C * REPLAYS * R
    del g
    h.destroy()


@pytest.mark.parametrize("R", [1, 2, 3, 8])
@pytest.mark.parametrize("n", [1, 2, 3, 17, 4096 + 1, 250001])
def test_odd_sizes(R, n):
    """Odd element counts make shard p start at an 8-byte (not 16-byte) offset."""
    zs = inputs.allgather_inputs(4, R, n, 5)
    h = _handle(R, n, "hbm")
    ins = [to_dev(z, "c64") for z in zs]
    outs = [torch.empty(R * n, dtype=torch.complex64, device="cuda") for _ in range(R)]
    enqueue(h, "allgather", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    h.check()
    want = oracle.allgather(zs, ranks=[0])[0]
    for r in range(R):
        assert_bits_equal(to_bits(outs[r]), want, "c64", f"rank {r}")
    h.destroy()


@pytest.mark.parametrize("n", [1, 3, 5, 1001])
def test_fp16_allgather_narrow_vectors(n):
    """A 2-byte dtype with odd numel takes the 2-byte vector path."""
    R = 3
    rng = np.random.default_rng(n)
    xs = [rng.integers(0, 65536, n, dtype=np.uint32).astype(np.uint16) for _ in range(R)]
    h = _handle(R, n, "pinned", torch.float16)
    ins = [to_dev(x, "f16") for x in xs]
    outs = [torch.empty(R * n, dtype=torch.float16, device="cuda") for _ in range(R)]
    enqueue(h, "allgather", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    want = oracle.allgather(xs, ranks=[0])[0].view(np.uint16)
    for r in range(R):
        assert np.array_equal(to_bits(outs[r]), want)
    h.destroy()


@pytest.mark.parametrize("slots", ["hbm", "pinned"])
@pytest.mark.parametrize("launch", ["rank", "fused"])
@pytest.mark.parametrize("R,n", [(2, 256 * 2 * 7 + 1), (3, 256 * 2 * 9), (5, 4099), (8, 256 * 4 * 5 + 3)])
def test_several_stages_per_block(slots, launch, R, n):
    """A block cap of 2 gives each block several stages: in HBM the kernel that
    publishes one stage ahead (16-byte vectors for an even element count,
    8-byte ones for an odd count), over the host link the plain one; both
    byte-exact, per-rank and in one launch of every rank, both parities."""
    h = _handle(R, n, slots)
    h.set_tactics(max_blocks=2)
    p = h.plan("allgather", n)
    assert p.blocks == 2 and p.tiles > 2
    streams = rank_streams(R)
    side = torch.cuda.Stream()
    for c in range(2):
        zs = inputs.allgather_inputs(4, R, n, 30 + c)
        ins = [to_dev(z, "c64") for z in zs]
        outs = [torch.empty(R * n, dtype=torch.complex64, device="cuda") for _ in range(R)]
        if launch == "rank":
            enqueue(h, "allgather", ins, outs, streams)
        else:
            side.wait_stream(torch.cuda.current_stream())
            h.allgather_fused(ins, outs, side)
            torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        h.check()
        want = oracle.allgather(zs, ranks=[0])[0]
        for r in range(R):
            assert_bits_equal(to_bits(outs[r]), want, "c64", f"{slots} {launch} R={R} n={n} call {c} rank {r}")
    h.destroy()
