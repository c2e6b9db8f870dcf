"""Inputs and outputs in pinned host memory (zero copy through ar_allreduce).

Mapped pinned host memory is device-accessible, so a caller may hand the
library host tensors directly: each rank's kernel then reads its input from
and writes its output to host memory.  Every form must still give the
oracle's bits.
"""
import numpy as np
import pytest
import torch

import oracle
from tensor_decode_all_gb300 import inputs
from tests.gpu_helpers import assert_bits_equal, enqueue, rank_streams

pytestmark = pytest.mark.gpu

TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _host(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TORCH[dtype]).pin_memory()


@pytest.mark.parametrize("R,dtype,n,slots,algo,fused", [
    (2, "f16", 131072, "pinned", None, False),
    (2, "f16", 4096, "pinned", None, False),        # tagged words
    (4, "bf16", 300001, "hbm", None, False),
    (8, "bf16", 393216, "hbm", None, False),        # two-shot
    (8, "bf16", 393216, "hbm", None, True),
    (3, "bf16", 65536, "pinned", "oneshot", True),
])
def test_host_buffers_directly(R, dtype, n, slots, algo, fused):
    import tensor_decode_all_gb300 as tda
    xs = inputs.allreduce_inputs(5, R, n, dtype, "uniform", 21)
    h = tda.Handle(R, TORCH[dtype], n, slots)
    if algo:
        h.set_algo(algo)
    ins = [_host(x, dtype) for x in xs]
    outs = [torch.empty(n, dtype=TORCH[dtype]).pin_memory() for _ in range(R)]
    if fused:
        s = torch.cuda.Stream()
        h.allreduce_fused(ins, outs, s)
        s.synchronize()
    else:
        enqueue(h, "allreduce", ins, outs, rank_streams(R))
    torch.cuda.synchronize()
    h.check()
    want = oracle.allreduce(xs, dtype, ranks=[0])[0]
    for r in range(R):
        got = outs[r].view(torch.int16).numpy().view(np.uint16)
        assert_bits_equal(got, want, dtype, f"zero copy R={R} {dtype} n={n} {slots} rank {r}")
    h.destroy()
