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

A second, finer model (run_pair_abort: softmax warps one by one, transaction bytes per copy, the
teardown) covers aborts: any wait may run out its limit, and the copies and MMAs left in flight
must all be waited for before TMEM is freed and the CTA exits; the earlier teardown, which
missed some of them, must be caught.
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


# ---------------------------------------------------------------------------------------------
# Aborts.  Every wait of the kernel gives up after a limit (the kernel parameter wait_cycles):
# the waiting thread sets the CTA's abort flag and leaves its loop, and every other wait of that
# CTA then returns at once unless its phase has already completed.  The peer CTA learns nothing
# of it: its own waits on the aborted CTA run out in turn.  The model below follows the kernel's
# code paths after a failed wait (which arrivals still happen, which copies and MMAs are left in
# flight) down to the teardown, and checks that
#   * no MMA is in flight when TMEM is freed,
#   * no TMA copy lands in a CTA after it has exited (st.async writes into the peer are ordered
#     before the issuing CTA's release arrival at the final cluster barrier),
#   * no barrier receives more arrivals than a phase holds.
# Drain waits (the ones that let copies and MMAs already issued finish) have a limit far above
# any copy's or MMA's latency: in the model they give up only when nothing is left in flight.
# ---------------------------------------------------------------------------------------------
class W:
    """A wait: bounded (gives up at the kernel's limit), a drain (gives up only when nothing is
    in flight), or hard (the cluster barrier: never gives up)."""

    def __init__(self, bar, parity, drain=False, hard=False):
        self.bar, self.parity, self.drain, self.hard = bar, parity, drain, hard

    def done(self):
        return self.bar.done(self.parity)


class Flag:
    """A barrier stand-in whose wait completes once `value` is set."""

    def __init__(self, value=False):
        self.value = value

    def done(self, parity):
        return self.value


def run_pair_abort(units, seed, abort_after=(None, None), teardown_drain=True):
    """Both CTAs over one share; CTA c's waits may start to run out after abort_after[c] steps
    (None: never).  teardown_drain=True is the kernel's teardown (copies drained after every
    role has finished); False is the earlier one, where a role drained only the copies it saw
    in flight when it left its loop."""
    rng = random.Random(seed)
    C = []
    for c in range(2):
        B = {}
        for s in range(3):
            for name, cnt in (("kv_full", 1), ("kv_empty", 1), ("s_full", 1), ("p_full", 128)):
                B[f"{name}{s}"] = Bar(f"c{c}.{name}{s}", cnt)
        for s in range(2):
            for name, cnt in (("o_par", 1), ("mref", 128), ("x_full", 1), ("x_empty", 1), ("x_read", 128)):
                B[f"{name}{s}"] = Bar(f"c{c}.{name}{s}", cnt)
        for name, cnt in (("q_full", 129), ("o_full", 1), ("o_free", 256), ("l", 256), ("stg", 256),
                          ("drain_qk", 1), ("drain_pv", 1)):
            B[name] = Bar(f"c{c}.{name}", cnt)
        C.append(B)
    landing = []                       # (source CTA, target CTA, kind, apply)
    mma = [[], []]                     # (issuer, barrier) commits in issue order
    abort = [False, False]
    issued = [0, 0]                    # stage loads issued
    q_last = [-1, -1]                  # unit of the last Q copy issued
    arrived = [False, False]
    cluster = Flag()
    errors = []
    steps = [0]

    def land(src, dst, kind, fn):
        landing.append((src, dst, kind, fn))

    def issue_q(c, u):
        C[c]["q_full"].arrive(1, tx=40960)
        land(c, c, "tma", lambda B=C[c]: B["q_full"].complete_tx(40960))
        q_last[c] = max(q_last[c], u)

    def producer(c):
        B, gi, ok = C[c], 0, True
        for n, _ in units:
            if not ok:
                break
            for _ in range(n):
                st = gi % 3
                if gi >= 3:
                    if not (yield W(B[f"kv_empty{st}"], ((gi // 3) - 1) & 1)):
                        ok = False
                        break
                B[f"kv_full{st}"].arrive(1, tx=1)
                land(c, c, "tma", lambda b=B[f"kv_full{st}"]: b.complete_tx(1))
                issued[c] = gi + 1
                gi += 1
        if not teardown_drain and abort[c]:
            for i in range(max(0, issued[c] - 3), issued[c]):
                yield W(B[f"kv_full{i % 3}"], (i // 3) & 1, drain=True)

    def qk_issuer(c):
        B, gi, ok = C[c], 0, True
        for ui, (n, _) in enumerate(units):
            if not ok or not (yield W(B["q_full"], ui & 1)):
                break
            for _ in range(n):
                st = gi % 3
                if not (yield W(B[f"kv_full{st}"], (gi // 3) & 1)):
                    ok = False
                    break
                mma[c].append(("qk", f"s_full{st}"))
                gi += 1
        mma[c].append(("qk", "drain_qk"))
        yield W(B["drain_qk"], 0, drain=True)

    def pv_issuer(c):
        B, gi, ok = C[c], 0, True
        for ui, (n, _) in enumerate(units):
            if not ok:
                break
            for i in range(n):
                st = gi % 3
                good = yield W(B[f"p_full{st}"], (gi // 3) & 1)
                if good and i == 0 and ui > 0:
                    good = yield W(B["o_free"], (ui - 1) & 1)
                if not good:
                    ok = False
                    break
                mma[c] += [("pv", f"kv_empty{st}"), ("pv", f"o_par{gi & 1}")]
                if i == n - 1:
                    mma[c].append(("pv", "o_full"))
                gi += 1
        mma[c].append(("pv", "drain_pv"))
        yield W(B["drain_pv"], 0, drain=True)

    def relay(c):
        B, P = C[c], C[1 - c]
        P["x_empty0"].arrive(1)
        okr = True
        if units[0][0] == 1:
            okr = yield W(B["stg"], 0)
        if okr:
            P["x_empty1"].arrive(1)
        gi = 0
        for ui, (n, _) in enumerate(units):
            if not okr:
                break
            n_next = units[ui + 1][0] if ui + 1 < len(units) else 0
            for i in range(n):
                if not (yield W(B[f"x_read{gi & 1}"], (gi >> 1) & 1)):
                    okr = False
                    break
                hold = ui + 1 if (i == n - 1 and n_next == 1) else (ui if i >= n - 2 else -1)
                if hold >= 0 and not (yield W(B["stg"], hold & 1)):
                    okr = False
                    break
                P[f"x_empty{gi & 1}"].arrive(1)
                gi += 1

    def softmax_warp(c, w):
        # warps 2..9: warpgroup g = (w - 2) >> 2; row 0 (which arms x_full) in warp 4 + 4g;
        # the Q copies are issued by warp 2 + 4g; every thread arrives, 32 per warp
        B = C[c]
        g = (w - 2) >> 2
        row0 = w == 4 + 4 * g
        tma_thread = w == 2 + 4 * g
        gi, ok, my_q = 0, True, -1
        for ui, (n, q) in enumerate(units):
            if not ok:
                break
            if ui == 0 and g == 0:
                if tma_thread:
                    issue_q(c, 0)
                    my_q = 0
                B["q_full"].arrive(32)
            gs = gi
            i = (g - gs) & 1
            while ok and i < n:
                gt = gs + i
                st = gt % 3
                ok = yield W(B[f"s_full{st}"], (gt // 3) & 1)
                if ok:
                    ok = yield W(B[f"x_empty{g}"], (gt >> 1) & 1)
                if not ok:
                    break
                land(c, 1 - c, "st.async", lambda P=C[1 - c], g=g: P[f"x_full{g}"].complete_tx(8192))
                if row0:
                    B[f"x_full{g}"].arrive(1, tx=32768)
                ok = yield W(B[f"x_full{g}"], (gt >> 1) & 1)
                if not ok:
                    break
                B[f"x_read{g}"].arrive(32)
                if i >= 1:
                    ok = yield W(B[f"mref{g ^ 1}"], ((gt - 1) >> 1) & 1)
                    if not ok:
                        break
                    if rng.random() < 0.3:     # a row of this warp moved the reference: rescale O
                        ok = yield W(B[f"o_par{(gt - 1) & 1}"], ((gt - 1) >> 1) & 1)
                        if not ok:
                            break
                B[f"mref{g}"].arrive(32)
                B[f"p_full{st}"].arrive(32)
                i += 2
            gi = gs + n
            if ok and ((gi - 1) & 1) != g and ui + 1 < len(units):
                gl = gi - 1
                ok = yield W(B[f"s_full{gl % 3}"], (gl // 3) & 1)
                if ok:
                    if units[ui + 1][1] == q:
                        B["q_full"].arrive(32)
                        if tma_thread:
                            B["q_full"].arrive(1)
                    else:
                        if tma_thread:
                            issue_q(c, ui + 1)
                            my_q = ui + 1
                        B["q_full"].arrive(32)
            # the unit's epilogue (also after a failed wait: its output is written empty)
            if ok:
                ok = yield W(B["o_full"], ui & 1)
            B["l"].arrive(32)
            okl = yield W(B["l"], ui & 1)
            ok = okl and ok
            yield W(Flag(True), 0)             # O is staged through exchange buffer g
            B["o_free"].arrive(32)
            B["stg"].arrive(32)
        if not teardown_drain and my_q >= 0 and abort[c]:
            yield W(B["q_full"], my_q & 1, drain=True)

    def teardown(c):
        B = C[c]
        if teardown_drain and abort[c]:
            for i in range(max(0, issued[c] - 3), issued[c]):
                yield W(B[f"kv_full{i % 3}"], (i // 3) & 1, drain=True)
            if q_last[c] >= 0:
                yield W(B["q_full"], q_last[c] & 1, drain=True)
        if mma[c]:
            errors.append(f"c{c}: TMEM freed with {len(mma[c])} MMA commit(s) in flight")
        # release arrival at the cluster barrier: this CTA's st.async writes are performed first
        for x in [x for x in landing if x[0] == c and x[2] == "st.async"]:
            landing.remove(x)
            x[3]()
        arrived[c] = True
        if all(arrived):
            cluster.value = True
        yield W(cluster, 0, hard=True)
        if any(x[1] == c for x in landing):
            errors.append(f"c{c}: a copy lands after the CTA exited: "
                          + ", ".join(f"{x[2]} from c{x[0]}" for x in landing if x[1] == c))

    roles = {}
    for c in range(2):
        roles.update({f"c{c}.producer": producer(c), f"c{c}.qk": qk_issuer(c), f"c{c}.pv": pv_issuer(c),
                      f"c{c}.relay": relay(c)})
        for w in range(2, 10):
            roles[f"c{c}.sm{w}"] = softmax_warp(c, w)
    pending = {}
    try:
        for k, r in roles.items():
            pending[k] = next(r, None)
        started = [False, False]
        while True:
            steps[0] += 1
            for c in range(2):
                if not started[c] and all(pending[k] is None for k in roles if k.startswith(f"c{c}.")):
                    started[c] = True
                    roles[f"c{c}.teardown"] = teardown(c)
                    pending[f"c{c}.teardown"] = next(roles[f"c{c}.teardown"], None)
            moves = []
            for k, wt in pending.items():
                if wt is None:
                    continue
                c = int(k[1])
                if wt.done():
                    moves.append(("go", k, True))
                elif wt.hard:
                    pass
                elif wt.drain:
                    if not landing and not mma[c]:
                        moves.append(("go", k, False))            # nothing left to wait for
                elif abort[c]:
                    moves.append(("go", k, False))
                elif abort_after[c] is not None and steps[0] >= abort_after[c]:
                    moves.append(("timeout", k, False))
            if landing:
                moves.append(("land", None, None))
            for c in range(2):
                if mma[c]:
                    moves.append(("mma", c, None))
            if not moves:
                # nothing can move: every wait still blocked runs out its limit in the end
                moves = [("timeout", k, False) for k, wt in pending.items()
                         if wt is not None and not wt.drain and not wt.hard]
            if not moves:
                break
            kind, k, val = rng.choice(moves)
            if kind in ("go", "timeout"):
                if kind == "timeout":
                    abort[int(k[1])] = True
                try:
                    pending[k] = roles[k].send(val)
                except StopIteration:
                    pending[k] = None
            elif kind == "land":
                x = landing.pop(rng.randrange(len(landing)))
                x[3]()
            else:
                C[k][mma[k].pop(0)[1]].arrive(1)
    except AssertionError as e:
        errors.append(str(e))
    stuck = sorted(k for k in pending if pending[k] is not None)
    return stuck, errors, abort


def _abort_cases(n, seed):
    rng = random.Random(seed)
    for units, s in _random_layouts(n, seed):
        total = sum(t for t, _ in units)
        # when each CTA's waits may start to run out: early, mid-share or never
        pick = lambda: rng.choice([None, rng.randint(0, 40 * total + 40)])
        yield units, s, (pick(), pick())


def test_aborts_at_any_wait_drain_everything():
    n_abort = 0
    for units, seed, after in _abort_cases(400, 11):
        stuck, errors, aborted = run_pair_abort(units, seed, after)
        assert not stuck and not errors, (units, seed, after, stuck, errors[:2])
        n_abort += any(aborted)
    assert n_abort > 200          # most cases do abort somewhere


def test_aborts_with_an_immediate_limit_drain_everything():
    # a wait limit of zero: every wait that is not already satisfied gives up at once
    layouts = list(_random_layouts(200, 12)) + [(u, s) for u in ([(1, 0)], [(2, 0)], [(3, 0)], [(2, 0), (1, 1)])
                                                for s in range(50)]
    for units, seed in layouts:
        stuck, errors, aborted = run_pair_abort(units, seed, (0, 0))
        assert not stuck and not errors, (units, seed, stuck, errors[:2])
        assert all(aborted)


def test_abort_model_without_aborts_matches_the_protocol():
    for units, seed in _random_layouts(200, 13):
        stuck, errors, aborted = run_pair_abort(units, seed)
        assert not stuck and not errors and not any(aborted), (units, seed, stuck, errors[:2])


def test_abort_model_catches_copies_drained_only_by_their_role():
    # the earlier teardown: a producer that had issued a short share's loads and left its loop
    # before another role aborted did not wait for them, and they could land after the CTA exited
    caught = 0
    for units in ([(2, 0)], [(3, 0)], [(2, 0), (1, 1)]):
        for seed in range(100):
            stuck, errors, _ = run_pair_abort(units, seed, (0, 0), teardown_drain=False)
            caught += bool(errors)
    assert caught > 0


# ---------------------------------------------------------------------------------------------
# One exchange buffer for both softmax warpgroups.  The non-persistent 128-row kernel had a
# four-stage variant (measured, not kept) in which the two warpgroups, taking alternate tiles,
# shared one exchange buffer; it faulted the GPU twice and its source was not kept.  This
# model rebuilds its exchange protocol from that description (one item per CTA pair: one unit
# of n tiles, tiles alternating between the warpgroups, the peer's partial of tile t in the
# single buffer, tile t + 1 sent once tile t has been read) and checks the buffer's contents
# at every read.  With one set of exchange barriers for both warpgroups, the two warpgroups'
# row-0 threads arm the same x_full phase (an over-arrival), parity waits alias across tiles,
# and roles hang: on the GPU a hang ran into the bounded waits, whose abort path then let
# loads still in flight land after the CTA exited (the teardown gap the abort model above
# catches).  With the barriers indexed by tile parity (each warpgroup arms and waits only its
# own) every read sees its own tile's partial.  The kept kernels give each warpgroup its own
# buffer and barriers (run_pair above).
# ---------------------------------------------------------------------------------------------
def run_pair_one_buffer(n, seed, stages=4, per_parity_barriers=True):
    rng = random.Random(seed)
    C = []
    for c in range(2):
        B = {}
        for s in range(stages):
            for name, cnt in (("kv_full", 1), ("kv_empty", 1), ("s_full", 1), ("p_full", 128)):
                B[f"{name}{s}"] = Bar(f"c{c}.{name}{s}", cnt)
        for s in range(2):
            for name, cnt in (("mref", 128), ("x_full", 1), ("x_empty", 1), ("x_read", 128)):
                B[f"{name}{s}"] = Bar(f"c{c}.{name}{s}", cnt)
        C.append(B)
    landing, mma, errors = [], [[], []], []
    buf = [None, None]                 # the tile whose partial CTA c's buffer holds
    writing = [None, None]             # a partial landing in CTA c's buffer

    def xb(t):                         # exchange barrier index of tile t
        return t & 1 if per_parity_barriers else 0

    def xpar(t):                       # parity of tile t's phase on its exchange barrier
        return (t >> 1) & 1 if per_parity_barriers else t & 1

    def wait(c, name, parity):
        bar = C[c][name]
        return lambda: bar.done(parity)

    def producer(c):
        for t in range(n):
            if t >= stages:
                yield wait(c, f"kv_empty{t % stages}", ((t // stages) - 1) & 1)
            landing.append(lambda c=c, s=t % stages: C[c][f"kv_full{s}"].arrive(1))

    def qk_issuer(c):
        for t in range(n):
            yield wait(c, f"kv_full{t % stages}", (t // stages) & 1)
            mma[c].append(f"s_full{t % stages}")

    def pv_issuer(c):
        for t in range(n):
            yield wait(c, f"p_full{t % stages}", (t // stages) & 1)
            mma[c].append(f"kv_empty{t % stages}")

    def relay(c):
        # the buffer starts empty (tile 0 may be sent); once tile t's partial has been read,
        # tile t + 1 may be sent (on the barrier of t + 1's parity)
        C[1 - c]["x_empty0"].arrive(1)
        for t in range(n):
            yield wait(c, f"x_read{xb(t)}", xpar(t))
            C[1 - c][f"x_empty{xb(t + 1)}"].arrive(1)

    def softmax(c, g):
        B, P = C[c], C[1 - c]
        for t in range(g, n, 2):
            yield wait(c, f"s_full{t % stages}", (t // stages) & 1)
            yield wait(c, f"x_empty{xb(t)}", xpar(t))

            def land_partial(c=c, t=t):
                if writing[1 - c] is not None and writing[1 - c] != t:
                    errors.append(f"c{1 - c}: partials of tiles {writing[1 - c]} and {t} in the buffer at once")
                buf[1 - c] = t
                writing[1 - c] = None
                C[1 - c][f"x_full{xb(t)}"].complete_tx(32768)

            writing[1 - c] = t if writing[1 - c] is None else writing[1 - c]
            landing.append(land_partial)
            B[f"x_full{xb(t)}"].arrive(1, tx=32768)
            yield wait(c, f"x_full{xb(t)}", xpar(t))
            if buf[c] != t:
                errors.append(f"c{c} tile {t}: read the partial of tile {buf[c]}")
            B[f"x_read{xb(t)}"].arrive(128)
            if t >= 1:
                yield wait(c, f"mref{g ^ 1}", ((t - 1) >> 1) & 1)
            B[f"mref{g}"].arrive(128)
            B[f"p_full{t % stages}"].arrive(128)

    roles = {}
    for c in range(2):
        roles.update({f"c{c}.producer": producer(c), f"c{c}.qk": qk_issuer(c), f"c{c}.pv": pv_issuer(c),
                      f"c{c}.relay": relay(c), f"c{c}.wg0": softmax(c, 0), f"c{c}.wg1": softmax(c, 1)})
    try:
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
    except AssertionError as e:
        errors.append(str(e))
    stuck = sorted(k for k in pending if pending[k] is not None)
    return stuck, errors


def test_one_buffer_with_barriers_per_tile_parity_runs_clean():
    for n in (1, 2, 3, 5, 8, 13):
        for seed in range(60):
            stuck, errors = run_pair_one_buffer(n, seed, per_parity_barriers=True)
            assert not stuck and not errors, (n, seed, stuck, errors[:2])


def test_one_buffer_with_one_barrier_set_is_caught():
    caught = 0
    for n in (2, 3, 5, 8):
        for seed in range(60):
            stuck, errors = run_pair_one_buffer(n, seed, per_parity_barriers=False)
            caught += bool(stuck or errors)
    assert caught > 100
