"""Model check of the bulk kernel's stage protocol, on the CPU.

The kernel's producer lane fills a ring of shared-memory stages; consumer
groups take the emitted units round-robin; every stage has a "full" and an
"empty" mbarrier whose waits only see phase parity.  This model replays the
protocol under random interleavings, with copies landing out of order, and
checks that every group reads exactly the unit it expects and that every
position's accumulator slot is finalised exactly once with the right sum.

mbarrier model: the barrier counts completed phases ``ph``; a parity probe
``try_wait(P)`` is true iff ``P != ph % 2`` (it asks about the current phase
or the one before it, nothing older).

It also shows the model is not vacuous: dropping the consumer's wait for the
release of the stage's previous fill makes a group read the wrong unit, and
allowing more groups than stages makes groups read wrong units or stall.

A second model injects a wait that runs out in one lane of one group: the
warp must leave as a whole (the kernel decides with a warp-wide vote), and
every other wait must then end through its own bound, with the status set
and no position written with a wrong value.
"""

import random

import pytest


class Bar:
    def __init__(self, count):
        self.count, self.ph, self.pend, self.tx = count, 0, count, 0

    def arrive(self, tx=0):
        self.pend -= 1
        self.tx += tx
        self._check()

    def land(self, n):
        self.tx -= n
        self._check()

    def _check(self):
        if self.pend == 0 and self.tx == 0:
            self.ph += 1
            self.pend = self.count

    def try_wait(self, parity):
        return parity != (self.ph & 1)


class WrongUnit(AssertionError):
    pass


def simulate(seed, stages, group_warps, units, ring_slots, release_wait=True):
    """units: list of (position, value).  Returns {position: sum}."""
    rnd = random.Random(seed)
    NS, G = stages, group_warps
    groups = 8 // G
    full = [Bar(1) for _ in range(NS)]
    empty = [Bar(G) for _ in range(NS)]
    stage, meta = [None] * NS, [None] * NS
    inflight = []
    acc, cnt = [0] * ring_slots, [0] * ring_slots
    done = {}

    def finalize(slot, pos):
        assert pos not in done, f"position {pos} finalised twice"
        done[pos] = acc[slot]

    prod = dict(i=0, it=0, seq=0, pos=None, n=0, slot=None, dones=0, state="emit")
    warps = [dict(it=w // G, phase="release", live=True, m=None) for w in range(8)]

    def close_position():
        if prod["n"]:
            sl = prod["slot"]
            cnt[sl] -= G * prod["n"]
            if cnt[sl] == 0:
                finalize(sl, prod["pos"])
        prod["n"] = 0

    for _ in range(500000):
        actors = ([] if prod["state"] == "end" else ["P"]) + \
                 [w for w in range(8) if warps[w]["live"]] + (["L"] if inflight else [])
        if not actors:
            return done
        a = rnd.choice(actors)
        if a == "L":                      # a bulk copy lands
            s, u = inflight.pop(rnd.randrange(len(inflight)))
            stage[s] = u
            full[s].land(1)
        elif a == "P":
            s, f = prod["it"] % NS, prod["it"] // NS
            if prod["state"] == "emit":
                if prod["i"] == len(units):
                    close_position()
                    prod["state"] = "dones"
                    continue
                pos, _ = units[prod["i"]]
                if prod["pos"] is not None and pos != prod["pos"]:
                    close_position()
                prod["pos"] = pos
                if not empty[s].try_wait((f & 1) ^ 1):
                    continue
                if prod["n"] == 0:
                    sl = prod["seq"] % ring_slots
                    prod["seq"] += 1
                    acc[sl], cnt[sl], prod["slot"] = 0, 0, sl
                meta[s] = (prod["it"], pos, prod["slot"], units[prod["i"]][1])
                stage[s] = None
                full[s].arrive(tx=1)
                inflight.append((s, prod["it"]))
                prod["it"] += 1
                prod["n"] += 1
                prod["i"] += 1
            else:                         # one end marker per group
                if prod["dones"] == groups:
                    prod["state"] = "end"
                    continue
                if not empty[s].try_wait((f & 1) ^ 1):
                    continue
                meta[s] = (prod["it"], -1, None, 0)
                full[s].arrive()
                prod["it"] += 1
                prod["dones"] += 1
        else:
            w = warps[a]
            s, f = w["it"] % NS, w["it"] // NS
            if w["phase"] == "release":
                if release_wait and f > 0 and not empty[s].try_wait((f - 1) & 1):
                    continue
                w["phase"] = "full"
            elif w["phase"] == "full":
                if not full[s].try_wait(f & 1):
                    continue
                m = meta[s]
                if m[0] != w["it"]:
                    raise WrongUnit(f"group expected unit {w['it']}, stage holds {m[0]}")
                if m[1] < 0:
                    w["live"] = False
                    continue
                if stage[s] != w["it"]:
                    raise WrongUnit(f"unit {w['it']}: data not landed")
                w["m"], w["phase"] = m, "work"
            else:
                _, pos, sl, val = w["m"]
                if a % G == 0:
                    acc[sl] += val
                cnt[sl] += 1
                if cnt[sl] == 0:
                    finalize(sl, pos)
                empty[s].arrive()
                w["it"] += groups
                w["phase"] = "release"
    raise AssertionError("no progress")


def group_warps_for(stages):
    gw = 1
    while gw < 8 and 8 // gw > stages:
        gw *= 2
    return gw


def random_units(rnd):
    units, expect = [], {}
    for pos in range(rnd.randint(1, 12)):
        for _ in range(rnd.choice([0, 1, 1, 2, 3, 5, 9])):
            v = rnd.randint(1, 100)
            units.append((pos, v))
            expect[pos] = expect.get(pos, 0) + v
    return units, expect


@pytest.mark.parametrize("block", range(4))
def test_protocol_delivers_every_unit_once(block):
    for trial in range(block * 400, (block + 1) * 400):
        rnd = random.Random(trial)
        NS = rnd.choice([1, 2, 3, 4, 6, 7, 8, 14, 16, 32])
        units, expect = random_units(rnd)
        got = simulate(trial, NS, group_warps_for(NS), units, NS + 2)
        assert got == expect, (trial, NS)


def _fails(release_wait, force_gw=None):
    for trial in range(2000):
        rnd = random.Random(trial)
        NS = rnd.choice([1, 2, 3, 4, 6, 7])
        units, expect = random_units(rnd)
        try:
            got = simulate(trial, NS, force_gw or group_warps_for(NS), units, NS + 2,
                           release_wait=release_wait)
        except AssertionError:       # wrong unit, double finalise or deadlock
            return True
        if got != expect:
            return True
    return False


def test_model_catches_missing_release_wait():
    assert _fails(release_wait=False)


def test_model_catches_more_groups_than_stages():
    assert _fails(release_wait=True, force_gw=1)


# ---------------------------------------------------------------------------
# A wait that runs out in one group
# ---------------------------------------------------------------------------

class ExitedLanesInCollective(AssertionError):
    pass


def simulate_timeout(seed, stages, group_warps, units, ring_slots, fault_warp, fault_unit,
                     uniform=True):
    """As ``simulate``, with bounded waits and one injected time-out: when
    warp ``fault_warp`` waits for its unit ``fault_unit`` to land, one of its
    lanes gives up while the other 31 see what the barrier says.  Waits give
    up for real only when nothing anywhere can progress (time passes with
    no arrival).  ``uniform`` is the kernel's rule: a warp whose lanes
    disagree leaves as a whole; without it the lanes that saw the data go on
    to the warp's full-mask reduction while the others have left.

    Returns (finalised {position: sum}, status set)."""
    rnd = random.Random(seed)
    NS, G = stages, group_warps
    groups = 8 // G
    full = [Bar(1) for _ in range(NS)]
    empty = [Bar(G) for _ in range(NS)]
    stage, meta = [None] * NS, [None] * NS
    inflight = []
    acc, cnt = [0] * ring_slots, [0] * ring_slots
    done = {}
    status = False

    def finalize(slot, pos):
        assert pos not in done, f"position {pos} finalised twice"
        done[pos] = acc[slot]

    prod = dict(i=0, it=0, seq=0, pos=None, n=0, slot=None, dones=0, state="emit")
    warps = [dict(it=w // G, phase="release", live=True, m=None) for w in range(8)]

    def close_position():
        if prod["n"]:
            sl = prod["slot"]
            cnt[sl] -= G * prod["n"]
            if cnt[sl] == 0:
                finalize(sl, prod["pos"])
        prod["n"] = 0

    idle = 0
    for _ in range(500000):
        actors = ([] if prod["state"] == "end" else ["P"]) + \
                 [w for w in range(8) if warps[w]["live"]] + (["L"] if inflight else [])
        if not actors:
            return done, status
        if idle > 50 * len(actors) and not inflight:
            # nothing can move: every bounded wait runs out
            status = True
            prod["state"] = "end"
            for w in warps:
                w["live"] = False
            continue
        a = rnd.choice(actors)
        moved = True
        if a == "L":
            s, u = inflight.pop(rnd.randrange(len(inflight)))
            stage[s] = u
            full[s].land(1)
        elif a == "P":
            s, f = prod["it"] % NS, prod["it"] // NS
            if prod["state"] == "emit":
                if prod["i"] == len(units):
                    close_position()
                    prod["state"] = "dones"
                    continue
                pos, _ = units[prod["i"]]
                if prod["pos"] is not None and pos != prod["pos"]:
                    close_position()
                prod["pos"] = pos
                if not empty[s].try_wait((f & 1) ^ 1):
                    moved = False
                else:
                    if prod["n"] == 0:
                        sl = prod["seq"] % ring_slots
                        prod["seq"] += 1
                        acc[sl], cnt[sl], prod["slot"] = 0, 0, sl
                    meta[s] = (prod["it"], pos, prod["slot"], units[prod["i"]][1])
                    stage[s] = None
                    full[s].arrive(tx=1)
                    inflight.append((s, prod["it"]))
                    prod["it"] += 1
                    prod["n"] += 1
                    prod["i"] += 1
            else:
                if prod["dones"] == groups:
                    prod["state"] = "end"
                    continue
                if not empty[s].try_wait((f & 1) ^ 1):
                    moved = False
                else:
                    meta[s] = (prod["it"], -1, None, 0)
                    full[s].arrive()
                    prod["it"] += 1
                    prod["dones"] += 1
        else:
            w = warps[a]
            s, f = w["it"] % NS, w["it"] // NS
            if w["phase"] == "release":
                if f > 0 and not empty[s].try_wait((f - 1) & 1):
                    moved = False
                else:
                    w["phase"] = "full"
            elif w["phase"] == "full":
                seen = full[s].try_wait(f & 1)
                lanes = [seen] * 32
                if a == fault_warp and w["it"] == fault_unit:
                    lanes[rnd.randrange(32)] = False
                if all(lanes):
                    m = meta[s]
                    if m[0] != w["it"]:
                        raise WrongUnit(f"group expected unit {w['it']}, stage holds {m[0]}")
                    if m[1] < 0:
                        w["live"] = False
                        continue
                    w["m"], w["phase"] = m, "work"
                elif not any(lanes):
                    moved = False            # still waiting
                elif uniform:
                    status = True            # the warp leaves as a whole
                    w["live"] = False
                else:
                    raise ExitedLanesInCollective(
                        f"warp {a}: {lanes.count(True)} lanes reach the reduction, "
                        f"{lanes.count(False)} have left")
            else:
                _, pos, sl, val = w["m"]
                if a % G == 0:
                    acc[sl] += val
                cnt[sl] += 1
                if cnt[sl] == 0:
                    finalize(sl, pos)
                empty[s].arrive()
                w["it"] += groups
                w["phase"] = "release"
        idle = 0 if moved else idle + 1
    raise AssertionError("no progress")


def _timeout_trials(uniform, n=600):
    for trial in range(n):
        rnd = random.Random(10_000 + trial)
        NS = rnd.choice([1, 2, 3, 4, 6, 7, 8, 16])
        units, expect = random_units(rnd)
        gw = group_warps_for(NS)
        fault_warp = rnd.randrange(8)
        # one of the units this warp's group takes
        first = fault_warp // gw
        fault_unit = first + (8 // gw) * rnd.randrange(max(1, len(units) // (8 // gw) + 1))
        yield trial, NS, gw, units, expect, fault_warp, fault_unit


def test_timeout_in_one_group_ends_every_wait():
    """One lane of one warp gives up: the warp leaves as a whole, the rest of
    the kernel ends through its own bounded waits, the status is set, and
    no position is written with a wrong or repeated value."""
    faulted = 0
    for trial, NS, gw, units, expect, fw, fu in _timeout_trials(uniform=True):
        got, status = simulate_timeout(trial, NS, gw, units, NS + 2, fw, fu)
        for pos, v in got.items():
            assert v == expect[pos], (trial, pos)
        if status:
            faulted += 1
            assert len(got) <= len(expect)
        else:
            assert got == expect, trial      # the fault never hit a wait
    assert faulted > 100


def test_model_catches_lanes_leaving_one_by_one():
    """Without the warp-wide decision, a lane that gave up leaves while the
    others go on to the full-mask reduction."""
    with pytest.raises(ExitedLanesInCollective):
        for trial, NS, gw, units, _, fw, fu in _timeout_trials(uniform=False):
            simulate_timeout(trial, NS, gw, units, NS + 2, fw, fu, uniform=False)
