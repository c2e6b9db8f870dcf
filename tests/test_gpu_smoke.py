"""The entry point's smoke run on the GPU: one fused all-reduce and one fused
allgather of every rank, each checked against the oracle inside smoke()."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_runs_clean():
    import __graft_entry__
    __graft_entry__.smoke()
