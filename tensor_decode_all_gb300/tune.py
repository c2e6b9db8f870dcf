"""Measure a handle's all-reduce tactics on this GPU, and keep them.

The library's built-in table (ar_choose_algo) puts the one-shot / two-shot
crossover, the sizes up to which the tagged-word form beats the flag
protocol, and the sizes up to which the cluster form beats the flag forms
when every rank launches at once, and the pace of the first stage's slot
stores over the host link, where they were measured on one GB300.  A caller on another GPU, or
with another clock or memory configuration, can measure them again: ``tune``
times the forms at power-of-two sizes, each in a CUDA graph of several calls
of every rank (the way decode replays them), picks the smallest measured size
from which two-shot is faster at that size and at every larger one, and the
largest size up to which tagged words are faster at every smaller one,
and, for slots in host memory, the fastest pace for a call of one stage per
block and for one of several, and sets them on the handle.  ``save`` / ``load`` keep the result in a JSON file
keyed by the GPU and the handle's shape, so a later process applies it
without measuring ("[SM120] Add optional FlashInfer PCIe-IPC all-reduce for
switch-free hosts", section "Modifications": a tuned, per-size choice of
kernel, with declines for what it does not support).

Timing only: the results of these calls are not checked here (the tests
check both forms against the oracle).
"""
from __future__ import annotations

import json
import os

NEVER = (1 << 64) - 1
DTYPE_NAMES = {1: "f16", 2: "bf16", 3: "c64"}
SLOT_NAMES = {0: "pinned", 1: "hbm"}


def key_for(device_name: str, sm_count: int, R: int, dtype: int, slot_kind: int) -> str:
    """The file key of a tactic: GPU model and SM count, ranks, dtype, slot kind."""
    return f"{device_name}|sm{sm_count}|R{R}|{DTYPE_NAMES.get(dtype, dtype)}|{SLOT_NAMES.get(slot_kind, slot_kind)}"


def handle_key(handle) -> str:
    import torch
    info = handle.info()
    return key_for(torch.cuda.get_device_name(info.device), info.sm_count, info.R, info.dtype, info.slot_kind)


def crossover(times: dict) -> int:
    """times: {bytes: {"oneshot": us, "twoshot": us}}.  The smallest size from
    which two-shot is faster at that size and every larger measured size, or
    NEVER if two-shot is not faster at the largest one."""
    threshold = NEVER
    for size in sorted(times, reverse=True):
        t = times[size]
        if t["twoshot"] < t["oneshot"]:
            threshold = size
        else:
            break
    return threshold


def tagged_limit(times: dict) -> int:
    """times: {bytes: {"tagged": us, "oneshot": us}}.  The largest size up to
    which the tagged-word form is faster at every measured size, or 0 (never)
    if it loses at the smallest one."""
    limit = 0
    for size in sorted(times):
        t = times[size]
        if t["tagged"] < t["oneshot"]:
            limit = size
        else:
            break
    return limit


def cluster_tactics(times: dict):
    """times: {bytes: {"cluster_oneshot": us, "cluster_twoshot": us, "flags": us}},
    measured for launches of every rank at once.  Returns (two-shot size of the
    cluster form, largest size for the cluster form): the crossover rule between
    the cluster form's two variants, then the largest size up to which the
    cluster form (with that crossover) beats the flag forms at every measured
    size (0: never)."""
    tw = crossover({b: {"oneshot": t["cluster_oneshot"], "twoshot": t["cluster_twoshot"]} for b, t in times.items()})
    best = {b: {"tagged": t["cluster_twoshot"] if b >= tw else t["cluster_oneshot"], "oneshot": t["flags"]}
            for b, t in times.items()}
    return tw, tagged_limit(best)


def _time_form(handle, algo: str, nbytes: int, calls: int, replays: int, fused: bool = False) -> float:
    """µs per call of one form at one size: graph of `calls` calls of every
    rank (per-rank launches on forked streams, or one launch of every rank)."""
    import torch
    R = handle.R
    dt = {1: torch.float16, 2: torch.bfloat16}[handle.dtype]
    numel = nbytes // 2
    handle.set_algo(algo)
    streams = [torch.cuda.Stream() for _ in range(R)]
    ins = [[torch.rand(numel, device="cuda").to(dt) for _ in range(R)] for _ in range(calls)]
    outs = [[torch.empty(numel, dtype=dt, device="cuda") for _ in range(R)] for _ in range(calls)]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            cap = torch.cuda.current_stream()
            for s in streams:
                s.wait_stream(cap)
            for c in range(calls):
                if fused:
                    handle.allreduce_fused(ins[c], outs[c], cap)
                    continue
                for r in range(R):
                    handle.allreduce(r, ins[c][r], outs[c][r], streams[r])
            for s in streams:
                cap.wait_stream(s)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(cur)
    for _ in range(replays):
        g.replay()
    b.record(cur)
    torch.cuda.synchronize()
    handle.check()
    del g
    return a.elapsed_time(b) * 1e3 / (replays * calls)


def measure(handle, sizes=None, replays: int = 5, forms=("oneshot", "twoshot")) -> dict:
    """{bytes: {form: us}} at the given sizes; by default the one-shot and
    two-shot forms at powers of two from 64 KiB to min(8 MiB, the handle's
    max payload)."""
    max_bytes = handle.max_numel * 2
    if sizes is None:
        sizes = [1 << k for k in range(16, 24) if (1 << k) <= max_bytes]
    saved = handle.info().algo
    times = {}
    try:
        for nbytes in sizes:
            if nbytes > max_bytes or nbytes % 16:
                raise ValueError(f"size {nbytes} not a multiple of 16 bytes within the handle's max payload")
            calls = max(4, min(20, (256 << 20) // (handle.R * nbytes * 2)))
            times[nbytes] = {algo: _time_form(handle, algo, nbytes, calls, replays) for algo in forms}
    finally:
        handle.set_algo(saved)
    return times


def measure_cluster(handle, sizes=None, replays: int = 5) -> dict:
    """{bytes: {"cluster_oneshot", "cluster_twoshot", "flags": us}} for launches
    of every rank at once: the cluster form forced one-shot and two-shot, and
    the flag forms the handle's per-rank tactics pick (cluster form off).  By
    default powers of two from 2 KiB to min(8 MiB, the handle's max payload).
    The handle's form and tactics are restored afterwards."""
    max_bytes = handle.max_numel * 2
    if sizes is None:
        sizes = [1 << k for k in range(11, 24) if (1 << k) <= max_bytes]
    saved_algo, saved = handle.info().algo, handle.tactics()
    variants = (("cluster_oneshot", "cluster", {"cluster_twoshot_min_bytes": NEVER}),
                ("cluster_twoshot", "cluster", {"cluster_twoshot_min_bytes": 0}),
                ("flags", "auto", {"cluster_max_bytes": 0}))
    times = {}
    try:
        for nbytes in sizes:
            calls = max(4, min(20, (256 << 20) // (handle.R * nbytes * 2)))
            times[nbytes] = {}
            for name, algo, tactics in variants:
                handle.set_tactics(**tactics)
                times[nbytes][name] = _time_form(handle, algo, nbytes, calls, replays, fused=True)
                handle.set_tactics(**saved)
    finally:
        handle.set_algo(saved_algo)
        handle.set_tactics(**saved)
    return times


PACES = (0, 220000, 280000, 356000, 440000)


def best_pace(times: dict) -> int:
    """times: {pace: us}.  The fastest pace (0 = unpaced); ties go to the
    smaller pace, the gentler on the link."""
    return min(sorted(times), key=lambda p: times[p])


def pace_sizes(handle):
    """(single, multi): a payload whose call takes one stage per block (the
    largest power of two up to 1 MiB that does, at least the handle's smallest
    paced size) and one that takes several (the smallest larger power of two
    that does); None where the handle's max payload has none."""
    max_bytes = handle.max_numel * 2
    min_bytes = max(handle.tactics()["pace_min_bytes"], 1 << 12)
    single = multi = None
    for k in range(12, 27):
        nbytes = 1 << k
        if nbytes > max_bytes:
            break
        p = handle.plan("allreduce", nbytes // 2)
        if p.tiles <= p.blocks:
            if nbytes >= min_bytes and nbytes <= (1 << 20):
                single = nbytes
        elif multi is None:
            multi = nbytes
    return single, multi


def measure_pace(handle, paces=PACES, replays: int = 5) -> dict:
    """{"single": {pace: us}, "multi": {pace: us}}: per-rank launches in the
    handle's AUTO form at the two sizes of pace_sizes, each pace set for both
    kinds of call.  The handle's tactics are restored afterwards."""
    saved_algo, saved = handle.info().algo, handle.tactics()
    single, multi = pace_sizes(handle)
    out = {}
    try:
        handle.set_algo("auto")
        for name, nbytes in (("single", single), ("multi", multi)):
            if nbytes is None:
                continue
            calls = max(4, min(20, (256 << 20) // (handle.R * nbytes * 2)))
            out[name] = {"bytes": nbytes, "us": {}}
            for pace in paces:
                handle.set_tactics(pace_mbs=pace, pace_multi_mbs=pace)
                out[name]["us"][pace] = _time_form(handle, "auto", nbytes, calls, replays)
            handle.set_tactics(**saved)
    finally:
        handle.set_algo(saved_algo)
        handle.set_tactics(**saved)
    return out


def tune(handle, sizes=None, tagged_sizes=None, cluster_sizes=None, replays: int = 5) -> dict:
    """Measure the crossovers -- one-shot / two-shot (sizes), tagged words /
    one-shot (tagged_sizes: by default powers of two from 2 KiB to the smaller
    of 512 KiB and the tagged form's capacity) and, where the GPU runs the
    cluster form, its two-shot size and its limit against the flag forms for
    launches of every rank (cluster_sizes) -- set them on the handle, and
    return the tactics and the measured times."""
    if handle.dtype not in (1, 2):
        raise ValueError("tactics apply to fp16/bf16 all-reduce handles")
    times = measure(handle, sizes, replays)
    if tagged_sizes is None:
        cap = min(handle.info().tagged_capacity_bytes, 512 << 10, handle.max_numel * 2)
        tagged_sizes = [1 << k for k in range(11, 20) if (1 << k) <= cap]
    tagged_times = measure(handle, tagged_sizes, replays, forms=("tagged", "oneshot")) if tagged_sizes else {}
    handle.set_tactics(twoshot_min_bytes=crossover(times), tagged_max_bytes=tagged_limit(tagged_times))
    cluster_times = {}
    if handle.info().cluster_form > 0 and (cluster_sizes is None or cluster_sizes):
        cluster_times = measure_cluster(handle, cluster_sizes, replays)
        tw, limit = cluster_tactics(cluster_times)
        handle.set_tactics(cluster_twoshot_min_bytes=tw, cluster_max_bytes=limit)
    pace_times = {}
    if handle.info().slot_kind == 0:
        pace_times = measure_pace(handle, replays=replays)
        changes = {}
        if "single" in pace_times:
            changes["pace_mbs"] = best_pace(pace_times["single"]["us"])
        if "multi" in pace_times:
            changes["pace_multi_mbs"] = best_pace(pace_times["multi"]["us"])
        if changes:
            handle.set_tactics(**changes)
    return {"tactics": handle.tactics(), "times_us": {str(k): v for k, v in times.items()},
            "tagged_times_us": {str(k): v for k, v in tagged_times.items()},
            "cluster_times_us": {str(k): v for k, v in cluster_times.items()},
            "pace_times_us": {k: {"bytes": v["bytes"], "us": {str(p): t for p, t in v["us"].items()}}
                              for k, v in pace_times.items()}}


def save(path: str, key: str, tactics: dict) -> None:
    """Store one key's tactics in the JSON file at path (other keys kept)."""
    data = {}
    if os.path.exists(path):
        with open(path) as f:
            data = json.load(f)
    data[key] = {k: int(v) for k, v in tactics.items()}
    tmp = path + ".tmp"
    with open(tmp, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
    os.replace(tmp, path)


def lookup(path: str, key: str):
    """The stored tactics of a key, or None."""
    if not os.path.exists(path):
        return None
    with open(path) as f:
        return json.load(f).get(key)


def load(path: str, handle) -> bool:
    """Apply the stored tactics for this handle's key; False if there are none."""
    t = lookup(path, handle_key(handle))
    if t is None:
        return False
    handle.set_tactics(**t)
    return True
