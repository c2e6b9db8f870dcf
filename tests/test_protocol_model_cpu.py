"""Counter-level models of the exchange protocol's two reuse hazards, on CPU.

These are models of the design, not of the arithmetic: they replay the
per-block counters a sequence of calls leaves behind (grids that change from
call to call, as block caps, traced kernels and single-launch calls make them)
and look for a reader that could take a stale value for the one it waits for.
Each model first finds the hazard in the layout the design rejected, so that a
model that could not see it would fail here, then finds none in the layout the
kernels use.

1. Tagged words.  A reader accepts a word when its tag equals the tag of the
   stage it waits for.  Indexed by payload vector, a word can be left by
   another block index of an earlier call, whose own stage count passed
   through the expected value.  Indexed by (stage, block) with one stage per
   block, every word is written by one block index only, whose tags only
   grow, and the tag x mod (2^32 - 1) + 1 is never 0 (the zeroed buffer).
2. Slot parity.  Slots are double-buffered by a block's call count, so a
   region written in call k + 1 must use the other half than in call k (a slow
   peer may still read call k's half).  If blocks that a smaller grid leaves
   idle keep their old count, a region can land on a block of the same parity;
   with every idle block's count advanced to the launched blocks' count, the
   halves alternate for every region.
"""
import itertools
import random

TAG_PERIOD = (1 << 32) - 1


def stage_tag(x: int) -> int:
    """The tag of stage count x: x mod (2^32 - 1), plus one (1 .. 2^32 - 1)."""
    return x % TAG_PERIOD + 1


def stale_tag_hit(calls, layout, bmax=8, seed=0):
    """Replay (tiles, blocks) calls; return the first read that an earlier
    call's word with the expected tag would satisfy, or None.

    Every block index b keeps a stage count (the same on every rank, which run
    the same grid) and a call count (its parity picks the buffer half).  Reads
    are checked before the call's own writes land: the worst case."""
    seq = [seed] * bmax
    ncalls = [0] * bmax
    mem = {}
    for k, (tiles, blocks) in enumerate(calls):
        B = min(blocks, tiles, bmax)
        stages = {b: (tiles - b + B - 1) // B for b in range(B)}
        where = []
        for b in range(B):
            for s in range(stages[b]):
                pos = b + s * B if layout == "vector" else s * bmax + b
                where.append((b, s, (ncalls[b] & 1, pos), stage_tag(seq[b] + s + 1)))
        for b, s, key, tag in where:
            old = mem.get(key)
            if old is not None and old[0] == tag:
                return k, b, s, old
        for b, s, key, tag in where:
            mem[key] = (tag, b, k)
        for b in range(B):
            seq[b] += stages[b]
            ncalls[b] += 1
    return None


def test_stage_tag_is_never_zero_and_steps_by_one():
    for x in list(range(0, 4)) + list(range(TAG_PERIOD - 3, TAG_PERIOD + 4)) + [(1 << 32) + 7, (1 << 64) - 1]:
        assert 1 <= stage_tag(x) <= TAG_PERIOD
        nxt = stage_tag(x + 1)
        assert nxt == stage_tag(x) + 1 or (stage_tag(x) == TAG_PERIOD and nxt == 1)
    assert stage_tag(TAG_PERIOD - 1) == TAG_PERIOD and stage_tag(TAG_PERIOD) == 1
    assert stage_tag(1 << 32) == 2     # where the count's low 32 bits are 0


def test_vector_indexed_tagged_buffer_admits_a_stale_word():
    """The model sees the hazard: some sequence of three calls with changing
    grids lets a reader take another block's old word."""
    options = [(t, b) for t in range(1, 7) for b in range(1, 5)]
    hit = None
    for n in (2, 3):
        for seq in itertools.product(options, repeat=n):
            if stale_tag_hit(list(seq), "vector"):
                hit = seq
                break
        if hit:
            break
    assert hit is not None and len(hit) <= 3, hit


def test_block_stage_indexed_single_stage_calls_admit_none():
    """The kernels' layout, one stage per block (tiles <= blocks): no stale
    word passes, over every sequence of up to four calls from a small set of
    grids, random longer ones, and stage counts seeded just below the tag
    period and 2^32."""
    options = [(t, b) for t in range(1, 6) for b in range(1, 6) if t <= b]
    for n in (1, 2, 3, 4):
        for seq in itertools.product(options, repeat=n):
            assert stale_tag_hit(list(seq), "block-stage") is None, seq
    rng = random.Random(7)
    for seed in (0, TAG_PERIOD - 5, (1 << 32) - 5):
        for _ in range(2000):
            seq = []
            for _ in range(rng.randint(2, 12)):
                b = rng.randint(1, 8)
                seq.append((rng.randint(1, b), b))
            assert stale_tag_hit(seq, "block-stage", seed=seed) is None, (seed, seq)


def test_block_stage_indexed_multi_stage_calls_also_admit_none_in_the_model():
    """Within the model the (stage, block) layout holds for several stages per
    block too; the kernels still run one stage per block because the buffer
    holds one 4 KiB tile per block and parity."""
    rng = random.Random(11)
    for _ in range(5000):
        seq = [(rng.randint(1, 12), rng.randint(1, 8)) for _ in range(rng.randint(2, 8))]
        assert stale_tag_hit(seq, "block-stage") is None, seq


def parity_reuse_hit(calls, advance_idle, bmax=4):
    """Replay (regions, regions per tile) calls; return the first region whose
    buffer half in call k + 1 equals its half in call k, or None."""
    ncalls = [0] * bmax
    last = {}
    for k, (units, per_tile) in enumerate(calls):
        tiles = -(-units // per_tile)
        B = min(tiles, bmax)
        now = {}
        for t in range(tiles):
            b = t % B
            for u in range(t * per_tile, min(units, (t + 1) * per_tile)):
                now[u] = (ncalls[b] & 1, b)
        for u, (half, b) in now.items():
            if u in last and last[u][2] == k - 1 and last[u][0] == half:
                return k, u, last[u], (half, b)
        for u, (half, b) in now.items():
            last[u] = (half, b, k)
        launched = ncalls[0] + 1
        for b in range(bmax):
            if b < B:
                ncalls[b] += 1
            elif advance_idle:
                ncalls[b] = launched
    return None


def test_slot_parity_needs_the_idle_blocks_advanced():
    options = [(u, t) for u in range(1, 9) for t in (1, 2)]
    without = None
    for n in (2, 3, 4):
        for seq in itertools.product(options, repeat=n):
            if parity_reuse_hit(list(seq), advance_idle=False):
                without = seq
                break
        if without:
            break
    assert without is not None and len(without) == 2, "the model must see the hazard without the advance"
    # a two-shot call of one 512-vector tile (two 256-vector regions, one
    # block), then a one-shot call of the same bytes on two blocks
    assert parity_reuse_hit([(2, 2), (2, 1)], advance_idle=False) is not None
    assert parity_reuse_hit([(2, 2), (2, 1)], advance_idle=True) is None
    for n in (2, 3):
        for seq in itertools.product(options, repeat=n):
            assert parity_reuse_hit(list(seq), advance_idle=True) is None, seq
    rng = random.Random(3)
    for _ in range(3000):
        seq = [(rng.randint(1, 16), rng.choice((1, 2))) for _ in range(rng.randint(2, 10))]
        assert parity_reuse_hit(seq, advance_idle=True, bmax=6) is None, seq
