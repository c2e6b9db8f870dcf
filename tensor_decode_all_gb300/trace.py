"""Per-block trace of the rank kernels (ar_set_trace), decoded on the host.

With tracing on, thread 0 of every block of every rank writes one record per
call: %globaltimer at the start and end of its work (one clock for all SMs,
so records of different ranks compare) and, in SM clock cycles after the
start, when the block's first stage was published and when it had seen every
peer's data of that stage.  From those records this module checks that the R
rank kernels of each call ran at the same time and splits a call's time into
its phases -- the evidence a timeline profiler would give, without one.
"""
from __future__ import annotations

import ctypes

import numpy as np

RECORD_DTYPE = np.dtype([("rank", "<i4"), ("block", "<i4"), ("call", "<u4"), ("stages", "<u4"),
                         ("t_start_ns", "<u8"), ("t_end_ns", "<u8"), ("cyc_published", "<u4"),
                         ("cyc_peers", "<u4"), ("cyc_end", "<u4"), ("algo", "<u4")])
ALGO_NAMES = {0: "oneshot", 1: "twoshot", 2: "tagged", 3: "cluster", 4: "push"}


class TraceRecord(ctypes.Structure):
    _fields_ = [(name, {"<i4": ctypes.c_int32, "<u4": ctypes.c_uint32, "<u8": ctypes.c_uint64}[fmt.str])
                for name, (fmt, _) in RECORD_DTYPE.fields.items()]


def start(handle, depth: int):
    """Allocate a zeroed device buffer for `depth` calls of every (rank, block)
    and turn tracing on for calls enqueued or captured from now on."""
    import torch
    info = handle.info()
    n = depth * info.R * info.max_blocks
    buf = torch.zeros(n * RECORD_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    handle.set_trace(buf, n)
    return buf


def records(buf) -> np.ndarray:
    """The written records of a trace buffer (device or host bytes)."""
    raw = buf.detach().cpu().numpy() if hasattr(buf, "detach") else np.asarray(buf)
    rec = np.frombuffer(raw.tobytes(), dtype=RECORD_DTYPE)
    return rec[rec["t_end_ns"] != 0]


def overlap_violations(rec: np.ndarray) -> list:
    """(call, block) pairs whose R rank blocks did not all run at one instant
    (the latest start is after the earliest end).  Empty when every block of
    every call overlapped with its peers, which the exchange requires."""
    bad = []
    for (call, block) in sorted({(int(c), int(b)) for c, b in zip(rec["call"], rec["block"])}):
        g = rec[(rec["call"] == call) & (rec["block"] == block)]
        if g["t_start_ns"].max() > g["t_end_ns"].min():
            bad.append((call, block))
    return bad


def summarize(rec: np.ndarray, sm_clock_mhz: float) -> dict:
    """Median phases over blocks (µs), the spread of rank start times per call,
    and per call the time from its first block's start to its last block's end
    and from there to the next call's first start (negative: they overlap)."""
    if len(rec) == 0:
        return {"records": 0}
    us = 1.0 / sm_clock_mhz
    pub = rec["cyc_published"].astype(np.float64) * us
    peers = rec["cyc_peers"].astype(np.float64) * us
    end = rec["cyc_end"].astype(np.float64) * us
    span = (rec["t_end_ns"] - rec["t_start_ns"]).astype(np.float64) / 1e3
    skew = []
    first, last = [], []
    for call in np.unique(rec["call"]):
        g = rec[rec["call"] == call]
        starts = [g[g["rank"] == r]["t_start_ns"].min() for r in np.unique(g["rank"])]
        skew.append((max(starts) - min(starts)) / 1e3)
        first.append(int(g["t_start_ns"].min()))
        last.append(int(g["t_end_ns"].max()))
    # per call: its first block's start to its last block's end, and that end to
    # the next call's first start (calls in order of their call count)
    call_span = [(b - a) / 1e3 for a, b in zip(first, last)]
    call_gap = [(first[i + 1] - last[i]) / 1e3 for i in range(len(first) - 1)]
    return {
        "records": int(len(rec)),
        "calls": int(len(np.unique(rec["call"]))),
        "ranks": int(len(np.unique(rec["rank"]))),
        "blocks_per_rank": int(len(np.unique(rec["block"]))),
        "algo": sorted({ALGO_NAMES.get(int(a), str(int(a))) for a in rec["algo"]}),
        "median_us": {"start_to_published": round(float(np.median(pub)), 3),
                      "published_to_peers_seen": round(float(np.median(peers - pub)), 3),
                      "peers_seen_to_end": round(float(np.median(end - peers)), 3),
                      "block_span": round(float(np.median(span)), 3)},
        "rank_start_skew_us": {"median": round(float(np.median(skew)), 3), "max": round(float(np.max(skew)), 3)},
        "call_us": {"span_median": round(float(np.median(call_span)), 3),
                    "gap_median": round(float(np.median(call_gap)), 3) if call_gap else None},
        "overlap_violations": len(overlap_violations(rec)),
    }
