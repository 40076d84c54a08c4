"""Pins of the prefix-sharing / eviction oracle to facts fixed outside it.

* the worked cases of ``tests/golden/prefix_matching.json``, derived by hand
  from the pages' Figure 5 and Figure 11 and the rules of Appendix A.1.2 and
  4.2.2 (each case names what it follows);
* the record state machine against the independent cache oracle
  (``OracleCache`` replays the same programs with its own code);
* a brute-force matcher written here on top of ``OracleCache`` on tiny random
  programs;
* the fork plan against Eq. (5): the entry's stored keys rotated by the
  plan's deltas equal the keys of a cache built directly from the request
  prefix (fp64, 1e-10), and a shared page moves nothing.

``test_prefix_pins_catch_planted_mistakes`` plants plausible mistakes in the
oracle (on the CPU) and checks that some pin fails for each.
"""
import json
import os

import numpy as np
import pytest

import oracle.akv_oracle as O
import oracle.akv_prefix as P

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold():
    with open(os.path.join(GOLD, "prefix_matching.json")) as f:
        return json.load(f)


def _program(named, tokens):
    """Golden path with token names -> (program, token ids); drops name tokens
    by their append order."""
    order, prog, ids = {}, [], []
    for op in named:
        if op[0] == "append":
            order[op[1]] = len(ids)
            ids.append(tokens[op[1]])
            prog.append(("append", 1))
        elif op[0] == "drop":
            prog.append(("drop", [(order[x], order[x] + 1) for x in op[1]]))
        else:
            prog.append(("repos",))
    return prog, ids


def _recs(named, tokens):
    prog, ids = _program(named, tokens)
    return P.records(prog, ids)


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_golden_matches():
    g = _gold()
    for case in g["cases"]:
        entries = {int(k): _recs(v, g["tokens"]) for k, v in case["entries"].items()}
        got = P.match(entries, _recs(case["request"], g["tokens"]), case["page_size"])
        assert got == case["expect"], (case["name"], got)


def pin_golden_eviction():
    g = _gold()
    for case in g["eviction"]:
        entries = {int(k): _recs(v, g["tokens"]) for k, v in case["entries"].items()}
        use = {int(k): v for k, v in case["last_use"].items()}
        assert P.evict_order(entries, use) == case["order"], case["name"]


def _random_program(rng, n_ops, max_append=5):
    prog, n = [], 0
    for _ in range(n_ops):
        u = rng.random()
        if u < 0.55 or n == 0:
            k = int(rng.integers(1, max_append + 1))
            prog.append(("append", k))
            n += k
        elif u < 0.8:
            b = int(rng.integers(0, n))
            prog.append(("drop", [(b, int(min(n, b + rng.integers(1, 4))))]))
        else:
            prog.append(("repos",))
    return prog, n


def _replay_cache(recs, layers=0, k_raw=None, v=None):
    """OracleCache state after a record list (records -> cache operations)."""
    c = O.OracleCache(2, 1, 8, 1e4, "f64", layers=list(range(layers)), page_size=4)
    sid = c.create()
    t = 0
    for r in recs:
        if r[0] == "T":
            if layers:
                c.append(sid, k_raw[:, t:t + 1], v[:, t:t + 1], token_ids=[r[1]])
            else:
                c.append(sid, np.zeros((0, 1, 1, 8)), np.zeros((0, 1, 1, 8)), token_ids=[r[1]])
            t += 1
        elif r[0] == "D":
            c.drop(sid, list(r[1]))
        else:
            c.reposition(sid)
    return c, sid


def pin_state_against_cache_oracle():
    """Active flags, positions and held slots of the record state machine
    equal those of the cache oracle on random programs."""
    rng = np.random.default_rng(5)
    for _ in range(60):
        prog, n = _random_program(rng, int(rng.integers(1, 14)))
        recs = P.records(prog, list(range(1000, 1000 + n)))
        st = P.State(recs)
        c, sid = _replay_cache(recs)
        s = c.seqs[sid]
        held = set(int(x) for x in s.logical)
        assert [t for t in range(n) if st.held[t]] == sorted(held)
        for i, t in enumerate(s.logical):
            assert st.alive[t] == bool(s.alive[i]) and st.pos[t] == int(s.pos[i])
            assert int(s.pos[i]) == i            # positions == slots while held
        assert st.next_pos == s.next_pos
        assert all(not st.alive[t] for t in range(n) if t not in held)


def _stored_by_cache(recs, page_size):
    """Tokens with a stored key per the cache oracle: held, and the page of
    their slot holds an active token."""
    c, sid = _replay_cache(recs)
    s = c.seqs[sid]
    live = {i // page_size for i in range(len(s.logical)) if s.alive[i]}
    return {int(t): i for i, t in enumerate(s.logical) if i // page_size in live}


def _brute_match(entries, req, page_size):
    best_exact, best_valid = None, None
    for eid in sorted(entries):
        e = entries[eid]
        stored = _stored_by_cache(e, page_size)
        m = 0
        while m < min(len(e), len(req)) and e[m] == req[m]:
            m += 1
        for n in range(1, m + 1):
            c, sid = _replay_cache(req[:n])
            s = c.seqs[sid]
            need = {int(t): int(p) for t, a, p in zip(s.logical, s.alive, s.pos) if a}
            if not all(t in stored for t in need):
                continue
            rot = sum(stored[t] != p for t, p in need.items())
            if rot == 0 and (best_exact is None or n > best_exact[0]):
                best_exact = (n, eid)
            if best_valid is None or (n, -rot) > best_valid[:2]:
                best_valid = (n, -rot, eid)
    if best_valid is None:
        return ("none", -1, 0, 0)
    if best_exact is not None and best_exact[0] >= best_valid[0]:
        return ("exact", best_exact[1], best_exact[0], 0)
    return ("retrigger", best_valid[2], best_valid[0], -best_valid[1])


def _family(rng, n_entries, page_size):
    """Entries and a request grown from one random trunk (so that prefixes are
    shared), with branches made of appends, drops and repositions."""
    trunk, n = _random_program(rng, int(rng.integers(2, 8)))
    ids = list(rng.integers(0, 3, size=200))    # few distinct ids: chance coincidences
    progs = []
    for _ in range(n_entries + 1):
        cut = int(rng.integers(1, len(trunk) + 1))
        base = trunk[:cut]
        nb = sum(op[1] for op in base if op[0] == "append")
        tail, m = [], nb
        for _ in range(int(rng.integers(0, 5))):
            u = rng.random()
            if u < 0.5 or m == 0:
                k = int(rng.integers(1, 4))
                tail.append(("append", k))
                m += k
            elif u < 0.8:
                b = int(rng.integers(0, m))
                tail.append(("drop", [(b, int(min(m, b + rng.integers(1, 3))))]))
            else:
                tail.append(("repos",))
        progs.append((base + tail, m))
    recs = [P.records(p, ids[:m]) for p, m in progs]
    return {i: r for i, r in enumerate(recs[:-1])}, recs[-1]


def pin_match_brute_force():
    rng = np.random.default_rng(17)
    kinds = set()
    for it in range(150):
        S = [1, 2, 4][it % 3]
        entries, req = _family(rng, int(rng.integers(1, 4)), S)
        got = P.match(entries, req, S)
        want = _brute_match(entries, req, S)
        assert (got["kind"], got["entry"], got["n_records"], got["n_rotated"]) == want, (it, got, want)
        kinds.add(got["kind"])
    assert kinds == {"none", "exact", "retrigger"}


def pin_fork_plan_rotation():
    """Eq. (5) on the plan: rotating each needed stored key by the plan's
    delta gives the key of a cache built from the request prefix itself."""
    rng = np.random.default_rng(23)
    n_checked = 0
    for it in range(120):
        S = [1, 2, 4][it % 3]
        entries, req = _family(rng, 1, S)
        got = P.match(entries, req, S)
        if got["kind"] == "none":
            continue
        e = entries[got["entry"]]
        n = got["n_records"]
        plan = P.fork_plan(e, req, n, S)
        ntok = max(sum(1 for r in e if r[0] == "T"), sum(1 for r in req if r[0] == "T"))
        k_raw = rng.standard_normal((1, ntok, 1, 8))
        v = rng.standard_normal((1, ntok, 1, 8))
        ce, se = _replay_cache(e, 1, k_raw, v)
        cr, sr = _replay_cache(req[:n], 1, k_raw, v)
        es, rs = ce.seqs[se], cr.seqs[sr]
        eslot = {int(t): i for i, t in enumerate(es.logical)}
        rslot = {int(t): i for i, t in enumerate(rs.logical)}
        freq = ce.freq
        rotated = 0
        for t, (dst, src, delta) in plan["moves"].items():
            assert src == eslot[t] and dst == rslot[t] and delta == dst - src
            k = O.reposition_key(es.K[:, src], src, dst, freq)
            np.testing.assert_allclose(k, rs.K[:, dst], rtol=0, atol=1e-10)
            np.testing.assert_array_equal(es.V[:, src], rs.V[:, dst])
            rotated += delta != 0
        assert rotated == got["n_rotated"]
        assert plan["n_slots"] == rs.next_pos
        for k, kind in enumerate(plan["pages"]):
            act = [i for i in range(len(rs.logical)) if rs.alive[i] and i // S == k]
            if kind == "shared":
                assert all(eslot[int(rs.logical[i])] == i for i in act)
            elif kind == "none":
                assert not act
        n_checked += 1
    assert n_checked > 40


def pin_records_canonical():
    """Records follow the history rules: merged non-empty drop ranges, an
    empty drop is no record, one record per appended token."""
    r = P.records([("append", 3), ("drop", [(2, 3), (0, 1), (1, 2)]), ("drop", []),
                   ("drop", [(1, 1)]), ("repos",)], [7, 8, 9])
    assert r == [("T", 7), ("T", 8), ("T", 9), ("D", ((0, 3),)), ("R",)]


PINS = {name: fn for name, fn in globals().items() if name.startswith("pin_")}


@pytest.mark.parametrize("pin", sorted(PINS))
def test_prefix_pin(pin):
    PINS[pin]()


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------

def _stored_ignores_pages(self, page_size):
    return {t: self.pos[t] for t in range(len(self.alive)) if self.held[t]}


def _stored_alive_only(self, page_size):
    return {t: self.pos[t] for t in range(len(self.alive)) if self.alive[t]}


def _apply_repos_keeps_next(self, r, _orig=P.State.apply):
    nxt = self.next_pos
    _orig(self, r)
    if r[0] == "R":
        self.next_pos = nxt


def _evict_ignores_active(entries, last_use):
    ids = sorted(entries)
    klass = {}
    for a in ids:
        ra = entries[a]
        ext = [b for b in ids if b != a and len(entries[b]) > len(ra) and entries[b][:len(ra)] == ra]
        if not ext:
            klass[a] = 1
        else:
            klass[a] = 0 if any(r[0] == "D" for b in ext for r in entries[b][len(ra):]) else 2
    return sorted(ids, key=lambda e: (klass[e], last_use[e], e))


def _evict_lru_only(entries, last_use):
    return sorted(entries, key=lambda e: (last_use[e], e))


def _match_ties_to_retrigger(entries, req, page_size):
    best_exact, best_valid = None, None
    for eid in sorted(entries):
        recs = entries[eid]
        m = P.common_length(recs, req)
        stored = P.State(recs).stored(page_size)
        for n in range(1, m + 1):
            st = P.State(req[:n])
            need = [t for t in range(len(st.alive)) if st.alive[t]]
            if any(t not in stored for t in need):
                continue
            rot = sum(1 for t in need if stored[t] != st.pos[t])
            if rot == 0 and (best_exact is None or (n, -eid) > best_exact):
                best_exact = (n, -eid)
            if rot and (best_valid is None or (n, -rot, -eid) > best_valid):
                best_valid = (n, -rot, -eid)
    if best_valid is not None and (best_exact is None or best_valid[0] >= best_exact[0]):
        n = best_valid[0]
        return dict(kind="retrigger", entry=-best_valid[2], n_records=n,
                    n_tokens=sum(1 for r in req[:n] if r[0] == "T"), n_rotated=-best_valid[1])
    if best_exact is None:
        return dict(kind="none", entry=-1, n_records=0, n_tokens=0, n_rotated=0)
    n = best_exact[0]
    return dict(kind="exact", entry=-best_exact[1], n_records=n,
                n_tokens=sum(1 for r in req[:n] if r[0] == "T"), n_rotated=0)


def _common_skips_mismatch(a, b):
    """Keeps matching past a differing record (no stop rule)."""
    n = 0
    while n < len(a) and n < len(b) and (a[n] == b[n] or a[n][0] == b[n][0] == "T"):
        n += 1
    return n


def _records_keep_empty_drop(program, token_ids, _orig=P.records):
    out = _orig(program, token_ids)
    if any(op[0] == "drop" and not any(e > b for b, e in op[1]) for op in program):
        out.append(("D", ()))
    return out


MUTANTS = {
    "stored_ignores_released_pages": ("State", "stored", _stored_ignores_pages),
    "stored_alive_only": ("State", "stored", _stored_alive_only),
    "repos_keeps_next_pos": ("State", "apply", _apply_repos_keeps_next),
    "eviction_drop_of_inactive_counts": (None, "evict_order", _evict_ignores_active),
    "eviction_lru_only": (None, "evict_order", _evict_lru_only),
    "tie_goes_to_retrigger": (None, "match", _match_ties_to_retrigger),
    "no_stop_at_first_difference": (None, "common_length", _common_skips_mismatch),
    "empty_drop_recorded": (None, "records", _records_keep_empty_drop),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_prefix_pins_catch_planted_mistakes(name, monkeypatch):
    cls, attr, fn = MUTANTS[name]
    monkeypatch.setattr(getattr(P, cls) if cls else P, attr, fn)
    failed = []
    for pin, f in PINS.items():
        try:
            f()
        except Exception:  # an assertion, or the mutant breaking outright
            failed.append(pin)
    assert failed, f"no pin caught mutant {name}"
