"""CPU model of the barrier protocol of the few-head decode kernel (one CTA).

`decode_fh_bf16_kernel` (decode_context_mla_gb300/csrc/decode_fewhead.cu) runs four roles that
meet only through mbarriers: a TMA producer (a Q buffer per unit, KV tiles into a 2-stage ring),
a QK issuer, a PV issuer and the softmax warpgroups (one actor here).  Besides hangs, the model
checks the buffer reuse the kernel relies on without a wait of its own:

* the softmax writes P^T of tile i into buffer i % 2 without waiting for that buffer's release:
  its last reader, PV(i - 2), must have completed before S(i) exists (PV(i - 2) committed the
  stage's empty barrier, which the load of tile i waited for, and QK(i) waited for that load);
* a stage is reloaded only after the PV that read it completed; QK(i) overwrites score buffer
  i % 2 only after the softmax loaded S(i - 2); the first PV of a unit overwrites its O buffer
  only after the epilogue two units back read it; a unit's Q buffer is reloaded only after the
  last QK that read it completed.

Each role is a generator that yields the barrier phase it waits for and arrives as the kernel
does; each MMA issuer's commits complete in its own issue order (the two issuers' in any
interleaving), TMA bytes land in any order, and a seeded random scheduler interleaves
everything.  A planted mistake (the PV issuer releasing the stage before its MMAs) must be
caught by the buffer checks.
"""
import random

import pytest


class Bar:
    """An mbarrier: arrivals per phase and a phase counter (transaction bytes folded into one
    arrival when a copy lands)."""

    def __init__(self, name, count):
        self.name, self.count, self.pending, self.phase = name, count, count, 0

    def arrive(self, n=1):
        self.pending -= n
        if self.pending < 0:
            raise AssertionError(f"over-arrival on {self.name} in phase {self.phase}")
        if self.pending == 0:
            self.phase += 1
            self.pending = self.count

    def done(self, parity):
        """try_wait.parity: the phase with this parity has completed."""
        return (self.phase & 1) != parity


def run(units, seed, release_after_pv=True):
    """One CTA over one share: units = tile counts of its units, in order."""
    rng = random.Random(seed)
    n_tiles = sum(units)
    B = {}
    for s in range(2):
        for name, cnt in (("kv_full", 1), ("kv_empty", 1), ("q_full", 1), ("q_free", 1),
                          ("s_full", 1), ("s_free", 1), ("p_full", 1), ("p_free", 1),
                          ("o_free", 1), ("o_full", 1)):
            B[f"{name}{s}"] = Bar(f"{name}{s}", cnt)
    B["o"] = Bar("o", 1)
    landing = []                  # copies in flight: (callback)
    mma = {"qk": [], "pv": []}    # per issuer, in issue order: ("mma", what) or ("commit", barrier)
    state = {"pv_done": set(), "s_loaded": set(), "stage_tile": {}, "epi_done": set(),
             "qk_done_units": set()}
    errors = []

    def wait(name, parity):
        bar = B[name]
        return lambda: bar.done(parity)

    def producer():
        t = 0
        for u, n in enumerate(units):
            if u >= 2:
                yield wait(f"q_free{u & 1}", ((u >> 1) - 1) & 1)
            if u >= 2 and u - 2 not in state["qk_done_units"]:
                errors.append(f"Q buffer {u & 1} reloaded for unit {u} before unit {u - 2}'s QK completed")
            landing.append(lambda u=u: B[f"q_full{u & 1}"].arrive())
            for _ in range(n):
                st = t & 1
                if t >= 2:
                    yield wait(f"kv_empty{st}", ((t >> 1) - 1) & 1)
                if t >= 2 and t - 2 not in state["pv_done"]:
                    errors.append(f"stage {st} reloaded for tile {t} before PV({t - 2}) completed")

                def land(t=t, st=st):
                    state["stage_tile"][st] = t
                    B[f"kv_full{st}"].arrive()
                landing.append(land)
                t += 1

    def qk_issuer():
        t = 0
        for u, n in enumerate(units):
            yield wait(f"q_full{u & 1}", (u >> 1) & 1)
            for _ in range(n):
                sb = t & 1
                if t >= 2:
                    yield wait(f"s_free{sb}", ((t >> 1) - 1) & 1)
                    if t - 2 not in state["s_loaded"]:
                        errors.append(f"QK({t}) overwrote S buffer {sb} before S({t - 2}) was loaded")
                yield wait(f"kv_full{sb}", (t >> 1) & 1)
                mma["qk"] += [("mma", ("qk", t)), ("commit", f"s_full{sb}")]
                t += 1
            mma["qk"].append(("qdone", u))
            mma["qk"].append(("commit", f"q_free{u & 1}"))

    def pv_issuer():
        t = 0
        for u, n in enumerate(units):
            for i in range(n):
                sb = t & 1
                yield wait(f"p_full{sb}", (t >> 1) & 1)
                if i == 0 and u >= 2:
                    yield wait(f"o_free{u & 1}", ((u >> 1) - 1) & 1)
                    if u - 2 not in state["epi_done"]:
                        errors.append(f"PV of unit {u} overwrote O buffer {u & 1} before unit {u - 2}'s epilogue")
                ops = [("mma", ("pv", t)), ("commit", f"kv_empty{sb}")]
                if not release_after_pv:          # the planted mistake: release, then the MMAs
                    ops.reverse()
                mma["pv"] += ops + [("commit", f"p_free{sb}"), ("commit", "o")]
                if i == n - 1:
                    mma["pv"].append(("commit", f"o_full{u & 1}"))
                t += 1

    def softmax():
        t = 0
        for u, n in enumerate(units):
            for i in range(n):
                sb = t & 1
                yield wait(f"s_full{sb}", (t >> 1) & 1)
                if state["stage_tile"].get(sb) != t:
                    errors.append(f"S({t}) computed from the wrong tile in stage {sb}")
                state["s_loaded"].add(t)
                B[f"s_free{sb}"].arrive()
                # a rescale of O (when a row's reference max moves) waits for PV(t - 2), then PV(t - 1)
                if rng.random() < 0.2 and t >= 1:
                    if t >= 2:
                        yield wait(f"p_free{sb}", ((t >> 1) - 1) & 1)
                    yield wait("o", (t - 1) & 1)
                # P^T of tile t into buffer sb, with no wait: PV(t - 2) must be complete
                if t >= 2 and t - 2 not in state["pv_done"]:
                    errors.append(f"P({t}) written into buffer {sb} before PV({t - 2}) completed")
                B[f"p_full{sb}"].arrive()
                t += 1
            # the unit's epilogue reads O once the unit's last PV completed
            yield wait(f"o_full{u & 1}", (u >> 1) & 1)
            state["epi_done"].add(u)
            B[f"o_free{u & 1}"].arrive()

    roles = [producer(), qk_issuer(), pv_issuer(), softmax()]
    waits = [None] * len(roles)
    live = list(range(len(roles)))

    def advance(k):
        try:
            waits[k] = next(roles[k])
        except StopIteration:
            live.remove(k)

    for k in list(live):
        advance(k)
    steps = 0
    while live or landing or mma["qk"] or mma["pv"]:
        steps += 1
        assert steps < 200000, "model did not finish"
        choices = [("role", k) for k in live if waits[k]()]
        if landing:
            choices.append(("land", None))
        for q in ("qk", "pv"):
            if mma[q]:
                choices.append(("mma", q))
        if not choices:
            blocked = {k: waits[k] for k in live}
            raise AssertionError(f"hang: roles {sorted(blocked)} blocked")
        kind, arg = rng.choice(choices)
        if kind == "role":
            advance(arg)
        elif kind == "land":
            landing.pop(rng.randrange(len(landing)))()
        else:
            op, what = mma[arg].pop(0)
            if op == "commit":
                B[what].arrive()
            elif op == "qdone":
                state["qk_done_units"].add(what)
            elif what[0] == "pv":
                state["pv_done"].add(what[1])
    return errors


UNIT_SETS = [
    [1],
    [5],
    [1, 1, 1, 1, 1],
    [3, 1, 2, 1, 4],
    [2, 2, 2],
    [1, 7, 1, 1, 3, 2],
    [12, 1, 1],
]


@pytest.mark.parametrize("units", UNIT_SETS)
def test_few_head_protocol_runs_and_reuses_buffers_safely(units):
    for seed in range(40):
        errs = run(units, seed)
        assert not errs, (units, seed, errs[:3])


def test_model_catches_a_stage_released_before_its_pv():
    """Planted mistake: the PV issuer commits the stage's empty barrier before its MMAs, so a
    reload (and the next P write into the same buffer) can overtake the PV still reading."""
    kinds = set()
    for seed in range(200):
        for e in run([4, 3, 5], seed, release_after_pv=False):
            kinds.add("P" if e.startswith("P(") else e.split(" ")[0])
    assert {"stage", "P"} <= kinds, kinds
