"""CPU model of the one-pass HiCache filter's chained scan (decoupled look-back).

`filter_onepass_kernel` (decode_context_mla_gb300/csrc/relayout.cu) gives each block a tile in
the order the blocks start (a ticket), publishes the tile's count as an aggregate, then reads the
status words of the 32 tiles before it at a time (lane l: tile - 1 - l), waits until all 32 are
published, sums the counts from the nearest tile back to the nearest one that already holds its
inclusive prefix (that tile's inclusive value included), moves 32 tiles further back if none
does, and publishes its own inclusive prefix.  Here blocks are generators run by a seeded random
scheduler that keeps at most `resident` blocks running and starts them in ticket order; a run
fails on a hang or on a prefix that differs from the exclusive sum of the counts.  Two planted
mistakes (stopping at the farthest inclusive tile of a window, and leaving the inclusive tile's
own value out) must be caught.
"""
import random

import pytest

AGG, INC = 1, 2


def run(counts, seed, resident=6, window=32, mistake=None):
    rng = random.Random(seed)
    n = len(counts)
    status = [(0, 0)] * n                      # (flag, value)
    prefix = [None] * n

    def block(t):
        if t == 0:
            status[0] = (INC, counts[0])
            prefix[0] = 0
            return
        status[t] = (AGG, counts[t])
        yield
        acc, j = 0, t - 1
        while True:
            slots = [j - l for l in range(window)]
            while not all(s < 0 or status[s][0] != 0 for s in slots):
                yield                            # spin: a predecessor has not published yet
            seen = [(INC, 0) if s < 0 else status[s] for s in slots]
            incs = [l for l, (f, _) in enumerate(seen) if f == INC]
            if incs:
                first = incs[-1] if mistake == "farthest" else incs[0]
                upto = first if mistake == "drop_inclusive" else first + 1
                acc += sum(v for _, v in seen[:upto])
                break
            acc += sum(v for _, v in seen)
            j -= window
            yield
        prefix[t] = acc
        status[t] = (INC, acc + counts[t])

    running, next_tile = [], 0
    steps = 0
    while next_tile < n or running:
        steps += 1
        assert steps < 10 ** 6, "model did not finish"
        if next_tile < n and len(running) < resident and (not running or rng.random() < 0.5):
            g = block(next_tile)
            running.append(g)
            next_tile += 1
            continue
        g = rng.choice(running)
        try:
            next(g)
        except StopIteration:
            running.remove(g)
    want, run_sum = [], 0
    for c in counts:
        want.append(run_sum)
        run_sum += c
    return prefix == want


@pytest.mark.parametrize("n,resident", [(1, 4), (5, 2), (40, 6), (150, 20), (400, 64)])
def test_lookback_prefixes_match_the_exclusive_sums(n, resident):
    for seed in range(10):
        rng = random.Random(1000 + seed)
        counts = [rng.randint(0, 4096) for _ in range(n)]
        assert run(counts, seed, resident=resident)


@pytest.mark.parametrize("mistake", ["farthest", "drop_inclusive"])
def test_model_catches_a_wrong_look_back(mistake):
    caught = False
    for seed in range(20):
        rng = random.Random(seed)
        counts = [rng.randint(1, 4096) for _ in range(120)]
        if not run(counts, seed, resident=24, mistake=mistake):
            caught = True
            break
    assert caught
