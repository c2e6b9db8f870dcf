"""bench.py's replica mode on CPU: two gloo ranks, max-over-ranks timing and
rank-0-only reference arm.  (The all-reduce's ranks are logical ranks on one
GPU; across GPUs the bench only runs independent replicas.)"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist(world)
    try:
        assert d.pg is not None and d.pg.get_backend() == "gloo"
        d.barrier()
        slowest = d.max(1.0 + rank)          # rank 1 is the slow one
        args = type("A", (), {"warmup": 0, "steps": 1})()
        ref = bench.run_reference(args, d) if rank != 0 else "skipped"
        q.put((rank, slowest, ref))
    finally:
        d.close()


def test_two_gloo_ranks_take_the_max_and_only_rank0_reports():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [g[1] for g in got] == [2.0, 2.0]
    assert got[1][2] is None  # rank 1 prints nothing on the reference arm


def test_max_over_ranks_helper():
    import bench
    assert bench.max_over_ranks([1.0, 3.5, 2.0]) == 3.5


def test_reference_arm_line_on_one_rank():
    """The reference arm's JSON line: the oracle timed on the host cores, on
    the same metric, unit and headline config as the kernels' arm."""
    import json
    import subprocess
    import sys
    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                         cwd=root, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == bench.UNIT
    assert line["higher_is_better"] is True and line["value"] > 0 and line["steps"] == 1
    cfg = dict(line["config"])
    assert cfg.pop("executor").startswith("the CPU oracle")
    assert cfg == bench.headline_config(1)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_profiled_traffic_follows_each_kernel_family(tmp_path, monkeypatch):
    """Counters stay attached to their kernel family: a comment edit keeps
    them, a code edit to one family's source voids that family's counters
    only, and a code edit to a shared header voids all of them."""
    import json
    import shutil
    import bench
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    files = sorted({f for fs in bench.FORM_SOURCES.values() for f in fs})
    for f in files:
        (tmp_path / f).parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(root, f), tmp_path / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    t = {"workloads": {form: {"dram_bytes_per_call": i + 1, "form": form, "source_sha256": bench.source_sha256(form)}
                       for i, form in enumerate(bench.FORM_SOURCES)}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(t))

    def valid():
        return {form for form in bench.FORM_SOURCES if bench.profiled_traffic(form) is not None}

    assert valid() == set(bench.FORM_SOURCES)
    ag = tmp_path / "tensor_decode_all_gb300/csrc/ar_allgather.cu"
    ag.write_text(ag.read_text() + "\n// a comment\n/* another */\n")
    assert valid() == set(bench.FORM_SOURCES)
    ag.write_text(ag.read_text() + "\nnamespace { int unused_edit = 1; }\n")
    assert valid() == set(bench.FORM_SOURCES) - {"allgather"}
    cl = tmp_path / "tensor_decode_all_gb300/csrc/ar_allreduce_cluster.cuh"
    cl.write_text(cl.read_text() + "\n#define EDIT 0\n")
    assert valid() == set(bench.FORM_SOURCES) - {"allgather", "cluster"}
    # the tagged-word header is included by every all-reduce translation unit
    tagged = tmp_path / "tensor_decode_all_gb300/csrc/ar_allreduce_tagged.cuh"
    tagged.write_text(tagged.read_text() + "\n#define EDIT 1\n")
    assert valid() == set()
    hdr = tmp_path / "include/ar.h"
    hdr.write_text(hdr.read_text() + "\n#define EDIT 2\n")
    assert valid() == set()
    assert bench.profiled_traffic("no such workload") is None


def test_algorithmic_bytes_of_each_form():
    """The byte counts behind every roofline fraction: pinned-host one-shot
    W = RS, Rd = R(R-1)S; two-shot, in the flag and the cluster form, W = (R+1)S,
    Rd = (2R-1)S; push R(R-1)S each way; HBM 4RS; allgather 3RS + R^2 S."""
    import bench
    R, S = 8, 1 << 20
    one = {"link_write": R * S, "link_read": R * (R - 1) * S}
    two = {"link_write": (R + 1) * S, "link_read": (2 * R - 1) * S}
    assert bench.algo_bytes("allreduce", R, S, "pinned", "oneshot") == one
    assert bench.algo_bytes("allreduce", R, S, "pinned", "cluster") == one
    assert bench.algo_bytes("allreduce", R, S, "pinned", "tagged") == one
    assert bench.algo_bytes("allreduce", R, S, "pinned", "twoshot") == two
    assert bench.algo_bytes("allreduce", R, S, "pinned", "cluster/sub64") == two
    assert bench.algo_bytes("allreduce", R, S, "pinned", "push") == {"link_write": R * (R - 1) * S,
                                                                   "link_read": R * (R - 1) * S}
    assert bench.algo_bytes("allreduce", R, S, "hbm", "cluster/sub64") == {"dram": 4 * R * S}
    assert bench.algo_bytes("allgather", R, S, "hbm") == {"dram": 3 * R * S + R * R * S}
    assert bench.algo_bytes("allgather", R, S, "pinned") == one
