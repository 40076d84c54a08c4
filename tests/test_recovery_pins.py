"""Pins of the recovery planner of the oracle (``oracle/akv_recovery.py``).

Each pin ties the planner to something other than itself: hand-worked plans
of the Figure 10 program (``tests/golden/recovery_fig10.json``), the keys
the main oracle's replay really gives each query, brute force over every
subset of the missing tokens on tiny programs (the smallest closed set), and
the defining invariants.  Planted mistakes (one level of dependencies only,
dependencies taken from the final active set, every missing token seeded)
must each make a pin fail.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle.akv_recovery as R
from oracle.akv_oracle import OracleCache

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _gold():
    with open(os.path.join(GOLDEN, "recovery_fig10.json")) as f:
        return json.load(f)


def _program(ops):
    out = []
    for op in ops:
        if op[0] == "append":
            out.append(("append", op[1]))
        elif op[0] == "drop":
            out.append(("drop", [tuple(r) for r in op[1]]))
        else:
            out.append(("repos",))
    return out


def _random_program(rng, n_ops):
    prog, n = [], 0
    for _ in range(n_ops):
        u = rng.random()
        if u < 0.55 or n == 0:
            k = int(rng.integers(1, 4))
            prog.append(("append", k))
            n += k
        elif u < 0.85:
            b = int(rng.integers(0, n))
            prog.append(("drop", [(b, int(min(n, b + rng.integers(1, 3))))]))
        else:
            prog.append(("repos",))
    return prog, n


def pin_fig10_hand_worked():
    g = _gold()
    prog = _program(g["ops"])
    n, read, active = R.replay_visibility(prog)
    assert n == 6
    assert [sorted(r) for r in read] == [[], [0], [0, 1], [0, 2], [0, 2], [0, 2, 4]]
    assert active == {0, 2, 4, 5}
    for case in g["cases"]:
        tokens, segs = R.plan_recovery(prog, case["missing"], case["need"])
        assert tokens == case["tokens"], case["why"]
        assert [list(s) for s in segs] == case["segments"], case["why"]


def pin_reads_match_replay():
    """read[t] plus t is the set of keys active when t is appended, as the
    main oracle's sequence state holds it (logical indices of alive slots)."""
    rng = np.random.default_rng(7)
    for _ in range(40):
        prog, n = _random_program(rng, int(rng.integers(1, 12)))
        _, read, active = R.replay_visibility(prog)
        c = OracleCache(2, 1, 4, 1e4, "fp32", layers=[], page_size=4)
        sid = c.create()
        t = 0
        for op in prog:
            if op[0] == "append":
                for _ in range(op[1]):
                    c.append(sid, np.zeros((0, 1, 1, 4)), np.zeros((0, 1, 1, 4)))
                    s = c.seqs[sid]
                    assert set(s.logical[s.alive].tolist()) == read[t] | {t}
                    t += 1
            elif op[0] == "drop":
                c.drop(sid, op[1])
            else:
                c.reposition(sid)
        s = c.seqs[sid]
        assert set(s.logical[s.alive].tolist()) == active


def _closed(read, missing, plan):
    return all((read[t] & missing) <= plan for t in plan)


def pin_minimal_by_brute_force():
    """The plan is the smallest set of missing tokens that holds the needed
    missing tokens and is closed under 'a recomputed token's query read it'
    (every such set, by enumeration on tiny programs)."""
    rng = np.random.default_rng(11)
    for _ in range(60):
        prog, n = _random_program(rng, int(rng.integers(2, 10)))
        if n == 0:
            continue
        _, read, active = R.replay_visibility(prog)
        missing = {t for t in range(n) if rng.random() < 0.5}
        need = None if rng.random() < 0.5 else {t for t in range(n) if rng.random() < 0.4}
        seed = (active if need is None else need) & missing
        closed = []
        ms = sorted(missing)
        for k in range(len(ms) + 1):
            for sub in itertools.combinations(ms, k):
                s = set(sub)
                if seed <= s and _closed(read, missing, s):
                    closed.append(s)
        smallest = min(closed, key=len)
        assert all(smallest <= s for s in closed)      # unique least closed set
        tokens, segs = R.plan_recovery(prog, missing, need)
        assert set(tokens) == smallest
        assert [t for b, e in segs for t in range(b, e)] == tokens


def pin_invariants():
    rng = np.random.default_rng(13)
    for _ in range(40):
        prog, n = _random_program(rng, int(rng.integers(2, 16)))
        if n == 0:
            continue
        _, read, active = R.replay_visibility(prog)
        missing = {t for t in range(n) if rng.random() < 0.4}
        tokens, _ = R.plan_recovery(prog, missing)
        plan = set(tokens)
        assert plan <= missing                       # resident tokens are never recomputed
        assert (active & missing) <= plan
        assert _closed(read, missing, plan)
        assert R.plan_recovery(prog, set())[0] == []  # nothing missing, nothing to do
    # every token missing and all of them needed: everything is recomputed
    prog, n = [("append", 3), ("drop", [(0, 1)]), ("append", 2)], 5
    assert R.plan_recovery(prog, set(range(n)), set(range(n)))[0] == list(range(n))


PINS = [pin_fig10_hand_worked, pin_reads_match_replay, pin_minimal_by_brute_force, pin_invariants]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

def _plan_one_level(program, missing, need=None):
    n, read, active = R.replay_visibility(program)
    missing = set(missing)
    need = active if need is None else set(need)
    plan = need & missing
    for t in list(plan):
        plan |= read[t] & missing
    tokens = sorted(plan)
    return tokens, _segments(tokens)


def _plan_final_active(program, missing, need=None):
    n, read, active = R.replay_visibility(program)
    missing = set(missing)
    need = active if need is None else set(need)
    plan = need & missing
    work = list(plan)
    while work:
        t = work.pop()
        for u in active:                   # what is active now, not what t read
            if u < t and u in missing and u not in plan:
                plan.add(u)
                work.append(u)
    tokens = sorted(plan)
    return tokens, _segments(tokens)


def _plan_all_missing(program, missing, need=None):
    tokens = sorted(set(missing))
    return tokens, _segments(tokens)


def _segments(tokens):
    segs = []
    for t in tokens:
        if segs and segs[-1][1] == t:
            segs[-1][1] = t + 1
        else:
            segs.append([t, t + 1])
    return [tuple(s) for s in segs]


MISTAKES = [_plan_one_level, _plan_final_active, _plan_all_missing]


@pytest.mark.parametrize("mistake", MISTAKES, ids=[m.__name__ for m in MISTAKES])
def test_planted_mistake_is_caught(mistake, monkeypatch):
    monkeypatch.setattr(R, "plan_recovery", mistake)
    failed = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed > 0
