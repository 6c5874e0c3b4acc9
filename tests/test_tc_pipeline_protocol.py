"""CPU model of the barrier protocol of the persistent 128-row decode kernel (both CTAs of a pair).

`decode_tc_bf16_persist_kernel` (decode_context_mla_gb300/csrc/decode_tc.cu) runs six roles per CTA
that meet only through mbarriers: a TMA producer, a QK issuer, a PV issuer, a relay and two softmax
warpgroups.  A mistake in who arrives where, or when, shows on the GPU as a hang or a fault, so the
protocol is checked here, on the CPU, before any change to it runs:

* each role is a generator that yields the barrier phase it waits for and arrives on barriers as
  the kernel does (arrival counts, transaction bytes, waits by phase parity);
* MMA commits complete in issue order, TMA and st.async bytes land in any order, and a seeded
  random scheduler interleaves everything;
* a run fails on a hang (every role blocked), an arrival into a phase that has none left
  (over-arrival), or a score write into an exchange buffer that still holds a unit's O.

Shares are cut from item tile counts the way the kernel cuts them (contiguous balanced shares of
the tile sequence, units of 1 tile upwards, runs of items with the same query rows), and two
planted mistakes must be caught.
"""
import random

import pytest


class Bar:
    """An mbarrier: an arrival count per phase, a transaction-byte count, a phase counter."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.tx, self.phase = name, count, count, 0, 0

    def arrive(self, n=1, tx=0):
        self.tx += tx
        self.pending -= n
        if self.pending < 0:
            raise AssertionError(f"over-arrival on {self.name} in phase {self.phase}")
        self._check()

    def complete_tx(self, nbytes):
        self.tx -= nbytes
        self._check()

    def _check(self):
        if self.pending == 0 and self.tx == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        """try_wait.parity: the phase with this parity has completed."""
        return (self.phase & 1) != parity


def run_pair(units, seed, same_q_waits_last_qk=True, hold_buffers=True):
    """Runs both CTAs over one share: units = [(tiles, query-rows id), ...]."""
    rng = random.Random(seed)
    n_tiles = sum(n for n, _ in units)
    C = []
    for c in range(2):
        B = {}
        for s in range(3):
            for name, cnt in (("kv_full", 1), ("kv_empty", 1), ("s_full", 1), ("p_full", 128)):
                B[f"{name}{s}"] = Bar(f"c{c}.{name}{s}", cnt)
        for s in range(2):
            for name, cnt in (("o_par", 1), ("mref", 128), ("x_full", 1), ("x_empty", 1), ("x_read", 128)):
                B[f"{name}{s}"] = Bar(f"c{c}.{name}{s}", cnt)
        for name, cnt in (("q_full", 129), ("o_full", 1), ("o_free", 256), ("l", 256), ("stg", 256)):
            B[name] = Bar(f"c{c}.{name}", cnt)
        C.append(B)
    landing = []                     # TMA / st.async bytes in flight
    mma = [[], []]                   # commits in issue order
    staging = [[False, False], [False, False]]
    errors = []

    def wait(c, name, parity):
        bar = C[c][name]
        return lambda: bar.done(parity)

    def producer(c):
        for t in range(n_tiles):
            if t >= 3:
                yield wait(c, f"kv_empty{t % 3}", ((t // 3) - 1) & 1)
            landing.append(lambda c=c, s=t % 3: C[c][f"kv_full{s}"].arrive(1))

    def qk_issuer(c):
        t = 0
        for u, (n, _) in enumerate(units):
            yield wait(c, "q_full", u & 1)
            for _ in range(n):
                yield wait(c, f"kv_full{t % 3}", (t // 3) & 1)
                mma[c].append(f"s_full{t % 3}")
                t += 1

    def pv_issuer(c):
        t = 0
        for u, (n, _) in enumerate(units):
            for i in range(n):
                yield wait(c, f"p_full{t % 3}", (t // 3) & 1)
                if i == 0 and u > 0:
                    yield wait(c, "o_free", (u - 1) & 1)
                mma[c] += [f"kv_empty{t % 3}", f"o_par{t & 1}"] + (["o_full"] if i == n - 1 else [])
                t += 1

    def relay(c):
        # buffers start empty: virtual tiles -2 and -1; -1 waits for unit 0's O if unit 0 has one tile
        C[1 - c]["x_empty0"].arrive(1)
        if hold_buffers and units[0][0] == 1:
            yield wait(c, "stg", 0)
        C[1 - c]["x_empty1"].arrive(1)
        t = 0
        for u, (n, _) in enumerate(units):
            n_next = units[u + 1][0] if u + 1 < len(units) else 0
            for i in range(n):
                yield wait(c, f"x_read{t & 1}", (t >> 1) & 1)
                if hold_buffers:
                    hold = u + 1 if (i == n - 1 and n_next == 1) else (u if i >= n - 2 else -1)
                    if hold >= 0:
                        yield wait(c, "stg", hold & 1)
                C[1 - c][f"x_empty{t & 1}"].arrive(1)
                t += 1

    def softmax(c, g):
        B = C[c]
        gi = 0
        for u, (n, q) in enumerate(units):
            if u == 0 and g == 0:                 # the first unit's Q: TMA part + TMEM part
                B["q_full"].arrive(1, tx=40960)
                landing.append(lambda B=B: B["q_full"].complete_tx(40960))
                B["q_full"].arrive(128)
            gs = gi
            for i in range((g - gs) & 1, n, 2):
                gt = gs + i
                yield wait(c, f"s_full{gt % 3}", (gt // 3) & 1)
                yield wait(c, f"x_empty{g}", (gt >> 1) & 1)
                if staging[1 - c][g]:
                    errors.append(f"c{c} tile {gt}: scores sent into a buffer holding the peer's O")
                landing.append(lambda c=c, g=g: C[1 - c][f"x_full{g}"].complete_tx(32768))
                B[f"x_full{g}"].arrive(1, tx=32768)
                yield wait(c, f"x_full{g}", (gt >> 1) & 1)
                B[f"x_read{g}"].arrive(128)
                if i >= 1:
                    yield wait(c, f"mref{g ^ 1}", ((gt - 1) >> 1) & 1)
                    if rng.random() < 0.3:         # a row moved the reference max: rescale O
                        yield wait(c, f"o_par{(gt - 1) & 1}", ((gt - 1) >> 1) & 1)
                B[f"mref{g}"].arrive(128)
                B[f"p_full{gt % 3}"].arrive(128)
            gi = gs + n
            if ((gi - 1) & 1) != g and u + 1 < len(units):
                # the warpgroup without the last tile readies the next unit's Q
                if units[u + 1][1] != q or same_q_waits_last_qk:
                    yield wait(c, f"s_full{(gi - 1) % 3}", ((gi - 1) // 3) & 1)
                if units[u + 1][1] == q:
                    B["q_full"].arrive(128)
                    B["q_full"].arrive(1)
                else:
                    B["q_full"].arrive(1, tx=40960)
                    landing.append(lambda B=B: B["q_full"].complete_tx(40960))
                    B["q_full"].arrive(128)
            yield wait(c, "o_full", u & 1)
            B["l"].arrive(128)
            yield wait(c, "l", u & 1)
            staging[c][g] = True                  # O through this warpgroup's exchange buffer
            yield lambda: True
            B["o_free"].arrive(128)
            yield lambda: True
            staging[c][g] = False
            B["stg"].arrive(128)

    roles = {}
    for c in range(2):
        roles.update({f"c{c}.producer": producer(c), f"c{c}.qk": qk_issuer(c), f"c{c}.pv": pv_issuer(c),
                      f"c{c}.relay": relay(c), f"c{c}.wg0": softmax(c, 0), f"c{c}.wg1": softmax(c, 1)})
    pending = {k: next(r, None) for k, r in roles.items()}
    while True:
        moves = [("role", k) for k in roles if pending[k] is not None and pending[k]()]
        moves += [("land", None)] if landing else []
        moves += [("mma", c) for c in range(2) if mma[c]]
        if not moves:
            break
        kind, k = rng.choice(moves)
        if kind == "role":
            pending[k] = next(roles[k], None)
        elif kind == "land":
            landing.pop(rng.randrange(len(landing)))()
        else:
            C[k][mma[k].pop(0)].arrive(1)
    stuck = sorted(k for k in roles if pending[k] is not None)
    return stuck, errors


def shares(tiles_per_item, qid, n_clusters):
    """The units of each cluster's contiguous balanced share, as (tiles, query-rows id)."""
    pre = [0]
    for n in tiles_per_item:
        pre.append(pre[-1] + n)
    total = pre[-1]
    out = []
    for k in range(n_clusters):
        lo, hi = total * k // n_clusters, total * (k + 1) // n_clusters
        units = [(min(pre[i + 1], hi) - max(pre[i], lo), qid[i]) for i in range(len(tiles_per_item))
                 if min(pre[i + 1], hi) > max(pre[i], lo)]
        if units:
            out.append(units)
    return out


def _random_layouts(n, seed):
    rng = random.Random(seed)
    for _ in range(n):
        q, units = 0, []
        for u in range(rng.randint(1, 6)):
            if u and rng.random() < 0.5:
                q += 1
            units.append((rng.randint(1, 5), q))
        yield units, rng.randrange(1 << 30)


@pytest.mark.parametrize("n_clusters", [76, 20, 7])
def test_dsv3_shaped_shares_run_to_completion(n_clusters):
    # 3 requests x 8 shards, 4 tiles per item, shards innermost (same query rows per request)
    for units in shares([4] * 24, [i // 8 for i in range(24)], n_clusters):
        for seed in range(12):
            stuck, errors = run_pair(units, seed)
            assert not stuck and not errors, (units, seed, stuck, errors[:2])


def test_random_unit_layouts_run_to_completion():
    for units, seed in _random_layouts(300, 7):
        stuck, errors = run_pair(units, seed)
        assert not stuck and not errors, (units, seed, stuck, errors[:2])


def test_model_catches_unordered_same_q_arrivals():
    # arriving for the next unit's Q without waiting for the last QK: over-arrival or a phase alias
    caught = 0
    for units, seed in _random_layouts(300, 8):
        try:
            stuck, errors = run_pair(units, seed, same_q_waits_last_qk=False)
        except AssertionError:
            caught += 1
            continue
        caught += bool(stuck or errors)
    assert caught > 0


def test_model_catches_buffers_released_during_staging():
    caught = sum(bool(run_pair(units, seed, hold_buffers=False)[1]) for units, seed in _random_layouts(300, 9))
    assert caught > 0
