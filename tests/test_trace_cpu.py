"""Host side of the trace: record layout, overlap check and phase summary."""
import numpy as np

from tensor_decode_all_gb300 import trace


def _rec(rows):
    a = np.zeros(len(rows), dtype=trace.RECORD_DTYPE)
    for i, (rank, block, call, t0, t1, pub, peers, end) in enumerate(rows):
        a[i] = (rank, block, call, 1, t0, t1, pub, peers, end, 0)
    return a


def test_record_is_48_bytes_and_unwritten_records_are_dropped():
    assert trace.RECORD_DTYPE.itemsize == 48
    a = _rec([(0, 0, 0, 100, 200, 10, 20, 30), (1, 0, 0, 150, 250, 10, 20, 30)])
    raw = np.concatenate([a.view(np.uint8), np.zeros(48 * 3, np.uint8)])
    got = trace.records(raw)
    assert len(got) == 2 and list(got["rank"]) == [0, 1]


def test_overlap_violation_found_only_where_a_peer_started_after_another_ended():
    ok = _rec([(0, 0, 0, 100, 300, 1, 2, 3), (1, 0, 0, 250, 400, 1, 2, 3),
               (0, 1, 0, 100, 300, 1, 2, 3), (1, 1, 0, 200, 300, 1, 2, 3)])
    assert trace.overlap_violations(ok) == []
    bad = _rec([(0, 0, 0, 100, 200, 1, 2, 3), (1, 0, 0, 250, 400, 1, 2, 3),
                (0, 0, 1, 500, 600, 1, 2, 3), (1, 0, 1, 550, 650, 1, 2, 3)])
    assert trace.overlap_violations(bad) == [(0, 0)]


def test_summary_phases_and_start_skew():
    # SM clock 1000 MHz: 1000 cycles = 1 us
    rows = [(0, 0, 0, 1_000, 9_000, 2_000, 5_000, 8_000), (1, 0, 0, 3_000, 9_500, 2_000, 5_000, 8_000),
            (0, 0, 1, 20_000, 28_000, 2_000, 5_000, 8_000), (1, 0, 1, 20_500, 28_000, 2_000, 5_000, 8_000)]
    s = trace.summarize(_rec(rows), sm_clock_mhz=1000.0)
    assert s["records"] == 4 and s["calls"] == 2 and s["ranks"] == 2
    assert s["median_us"] == {"start_to_published": 2.0, "published_to_peers_seen": 3.0,
                              "peers_seen_to_end": 3.0, "block_span": 7.75}
    assert s["rank_start_skew_us"] == {"median": 1.25, "max": 2.0}
    assert s["overlap_violations"] == 0
    # call 0 runs 1.0 .. 9.5 us, call 1 20.0 .. 28.0 us
    assert s["call_us"] == {"span_median": 8.25, "gap_median": 10.5}
