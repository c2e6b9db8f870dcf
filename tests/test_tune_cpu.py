"""Host logic of the tactic tuner: the crossover rule and the tactic file."""
import json

from tensor_decode_all_gb300 import tune


def test_crossover_smallest_size_from_which_twoshot_always_wins():
    t = {65536: {"oneshot": 5.0, "twoshot": 6.0},
         262144: {"oneshot": 8.0, "twoshot": 7.0},
         1048576: {"oneshot": 20.0, "twoshot": 12.0}}
    assert tune.crossover(t) == 262144


def test_crossover_ignores_an_isolated_win_below_a_loss():
    # two-shot wins at 64 KiB by noise, loses at 256 KiB, wins from 1 MiB
    t = {65536: {"oneshot": 5.0, "twoshot": 4.9},
         262144: {"oneshot": 8.0, "twoshot": 8.5},
         1048576: {"oneshot": 20.0, "twoshot": 12.0}}
    assert tune.crossover(t) == 1048576


def test_crossover_never_when_the_largest_size_prefers_oneshot():
    t = {65536: {"oneshot": 5.0, "twoshot": 4.0}, 1048576: {"oneshot": 10.0, "twoshot": 11.0}}
    assert tune.crossover(t) == tune.NEVER
    assert tune.crossover({}) == tune.NEVER


def test_key_names_gpu_ranks_dtype_and_slots():
    assert tune.key_for("GB300", 152, 8, 2, 1) == "GB300|sm152|R8|bf16|hbm"
    assert tune.key_for("GB300", 152, 2, 1, 0) == "GB300|sm152|R2|f16|pinned"


def test_save_and_lookup_keep_other_keys(tmp_path):
    path = str(tmp_path / "tactics.json")
    a = {"twoshot_min_bytes": 524288, "twoshot_sub": 0, "max_blocks": 0}
    b = {"twoshot_min_bytes": tune.NEVER, "twoshot_sub": 128, "max_blocks": 12}
    tune.save(path, "k1", a)
    tune.save(path, "k2", b)
    assert tune.lookup(path, "k1") == a
    assert tune.lookup(path, "k2") == b
    assert tune.lookup(path, "k3") is None
    assert tune.lookup(str(tmp_path / "missing.json"), "k1") is None
    with open(path) as f:
        assert sorted(json.load(f)) == ["k1", "k2"]


def test_tagged_limit_largest_size_up_to_which_tagged_always_wins():
    t = {2048: {"tagged": 3.0, "oneshot": 3.5}, 8192: {"tagged": 3.2, "oneshot": 3.6},
         32768: {"tagged": 4.8, "oneshot": 4.6}, 131072: {"tagged": 5.0, "oneshot": 6.0}}
    assert tune.tagged_limit(t) == 8192          # the win at 128 KiB after a loss does not count
    assert tune.tagged_limit({2048: {"tagged": 4.0, "oneshot": 3.5}}) == 0
    assert tune.tagged_limit({}) == 0


def test_cluster_tactics_crossover_then_limit_against_the_flag_forms():
    t = {2048: {"cluster_oneshot": 2.9, "cluster_twoshot": 4.1, "flags": 3.7},
         65536: {"cluster_oneshot": 3.4, "cluster_twoshot": 4.6, "flags": 4.2},
         524288: {"cluster_oneshot": 7.4, "cluster_twoshot": 6.8, "flags": 7.9},
         1048576: {"cluster_oneshot": 12.1, "cluster_twoshot": 12.0, "flags": 9.8},
         4194304: {"cluster_oneshot": 37.6, "cluster_twoshot": 36.0, "flags": 27.7}}
    tw, limit = tune.cluster_tactics(t)
    assert tw == 524288                 # two-shot faster from 512 KiB on
    assert limit == 524288              # the cluster form loses to the flags from 1 MiB
    # one-shot throughout, and a cluster form that loses at the smallest size: never
    t2 = {2048: {"cluster_oneshot": 4.0, "cluster_twoshot": 5.0, "flags": 3.5},
          8192: {"cluster_oneshot": 3.0, "cluster_twoshot": 5.0, "flags": 3.5}}
    assert tune.cluster_tactics(t2) == (tune.NEVER, 0)
    assert tune.cluster_tactics({}) == (tune.NEVER, 0)


def test_best_pace_is_the_fastest_and_ties_go_to_the_gentler_pace():
    assert tune.best_pace({0: 7.9, 220000: 8.2, 356000: 7.1, 440000: 7.2}) == 356000
    assert tune.best_pace({0: 5.0, 356000: 5.0}) == 0
    assert tune.best_pace({220000: 63.5, 356000: 72.5, 0: 77.0}) == 220000


class _FakePlan:
    def __init__(self, tiles, blocks):
        self.tiles, self.blocks = tiles, blocks


class _FakeHandle:
    """A pinned R=2 handle's plans: one 4 KiB tile per block up to 380 blocks."""
    def __init__(self, max_numel, pace_min=128 << 10):
        self.max_numel, self.pace_min = max_numel, pace_min

    def tactics(self):
        return {"pace_min_bytes": self.pace_min}

    def plan(self, op, numel):
        tiles = -(-numel * 2 // 4096)
        return _FakePlan(tiles, min(tiles, 380))


def test_pace_sizes_pick_a_single_stage_and_a_multi_stage_payload():
    assert tune.pace_sizes(_FakeHandle(4 << 20)) == (1 << 20, 2 << 20)
    assert tune.pace_sizes(_FakeHandle(128 << 10)) == (256 << 10, None)     # 256 KiB max payload
    assert tune.pace_sizes(_FakeHandle(32 << 10)) == (None, None)           # below the smallest paced size
