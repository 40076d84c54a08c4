"""The library's host-only prefix index through the C ABI, against the
oracle (``oracle/akv_prefix.py``): the worked cases of the golden file,
random program families with shared prefixes, eviction order, churn.
No GPU: the index does no device work."""
import json
import os

import numpy as np
import pytest

from agent_kv_cache_gb300 import PrefixIndex, abi, build
import oracle.akv_prefix as P
from test_prefix_pins import _family, _program

GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()


def _to_program(recs):
    """Records -> (program, token ids) that expand to exactly those records."""
    prog, ids = [], []
    for r in recs:
        if r[0] == "T":
            if prog and prog[-1][0] == "append":
                prog[-1] = ("append", prog[-1][1] + 1)
            else:
                prog.append(("append", 1))
            ids.append(r[1])
        elif r[0] == "D":
            prog.append(("drop", [list(x) for x in r[1]]))
        else:
            prog.append(("repos",))
    return prog, ids


def _check_coords(prog, m):
    """(op_index, op_tokens) name the covered prefix of the program."""
    if m["kind"] == "none":
        return
    covered = sum(op[1] for op in prog[:m["op_index"]] if op[0] == "append") + m["op_tokens"]
    assert covered == m["n_tokens"]
    if m["op_tokens"]:
        assert prog[m["op_index"]][0] == "append" and m["op_tokens"] <= prog[m["op_index"]][1]


def test_golden_cases_through_the_abi():
    g = json.load(open(os.path.join(GOLD, "prefix_matching.json")))
    for case in g["cases"]:
        idx = PrefixIndex(case["page_size"])
        for k, v in case["entries"].items():
            prog, ids = _program(v, g["tokens"])
            idx.insert(int(k), prog, ids)
        prog, ids = _program(case["request"], g["tokens"])
        got = idx.match(prog, ids)
        want = case["expect"]
        assert {k: got[k] for k in want} == want, (case["name"], got)
        _check_coords(prog, got)
    for case in g["eviction"]:
        idx = PrefixIndex(16)
        for k, v in case["entries"].items():
            prog, ids = _program(v, g["tokens"])
            idx.insert(int(k), prog, ids, use_time=case["last_use"][k])
        assert idx.evict_order() == case["order"], case["name"]


@pytest.mark.parametrize("seed", range(6))
def test_random_families_match_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    for it in range(60):
        S = [1, 2, 4, 16][it % 4]
        entries, req = _family(rng, int(rng.integers(1, 6)), S)
        idx = PrefixIndex(S)
        for eid, recs in entries.items():
            prog, ids = _to_program(recs)
            idx.insert(eid, prog, ids)
        prog, ids = _to_program(req)
        got = idx.match(prog, ids)
        want = P.match(entries, req, S)
        assert {k: got[k] for k in want} == want, (seed, it, got, want)
        _check_coords(prog, got)
        use = {e: int(rng.integers(0, 4)) for e in entries}
        for e, u in use.items():
            idx.touch(e, u)
        assert idx.evict_order() == P.evict_order(entries, use)


def test_churn_insert_remove():
    """Entries removed and re-inserted in random order; every match equals
    the oracle over the entries present."""
    rng = np.random.default_rng(99)
    entries, req = _family(rng, 12, 4)
    idx = PrefixIndex(4)
    present = {}
    for step in range(80):
        e = int(rng.integers(0, len(entries)))
        if e in present:
            idx.remove(e)
            del present[e]
        else:
            prog, ids = _to_program(entries[e])
            idx.insert(e, prog, ids)
            present[e] = entries[e]
        prog, ids = _to_program(req)
        got = idx.match(prog, ids)
        want = P.match(present, req, 4)
        assert {k: got[k] for k in want} == want, (step, got, want)


def test_long_programs_match_oracle():
    """Agent-sized histories (hundreds of tokens, drops of spans, repositions)
    sharing a trunk; matching the request grown from the same trunk."""
    rng = np.random.default_rng(7)
    trunk, n = [], 0
    for _ in range(30):
        k = int(rng.integers(5, 40))
        trunk.append(("append", k))
        n += k
        if rng.random() < 0.4:
            b = int(rng.integers(0, n))
            trunk.append(("drop", [(b, min(n, b + int(rng.integers(1, 30))))]))
        if rng.random() < 0.2:
            trunk.append(("repos",))
    ids = list(rng.integers(0, 50000, size=n + 500))
    entries = {}
    for e in range(8):
        cut = int(rng.integers(1, len(trunk) + 1))
        prog = trunk[:cut]
        m = sum(op[1] for op in prog if op[0] == "append")
        tail = [("append", int(rng.integers(1, 20)))]
        if rng.random() < 0.5:
            tail.append(("drop", [(0, int(rng.integers(1, 10)))]))
        if rng.random() < 0.5:
            tail.append(("repos",))
        m2 = m + tail[0][1]
        entries[e] = P.records(prog + tail, ids[:m2])
    req = P.records(trunk + [("append", 3)], ids[:n + 3])
    for S in (1, 16):
        idx = PrefixIndex(S)
        for e, recs in entries.items():
            prog, tok = _to_program(recs)
            idx.insert(e, prog, tok)
        prog, tok = _to_program(req)
        got = idx.match(prog, tok)
        want = P.match(entries, req, S)
        assert {k: got[k] for k in want} == want, (S, got, want)


def test_index_errors():
    idx = PrefixIndex(16)
    idx.insert(3, [("append", 2)], [1, 2])
    with pytest.raises(abi.AkvError) as e:
        idx.insert(3, [("append", 1)], [1])             # id taken
    assert e.value.code == abi.AKV_EINVAL
    with pytest.raises(abi.AkvError) as e:
        idx.insert(4, [("append", 2)], [1])             # fewer ids than tokens
    assert e.value.code == abi.AKV_EINVAL
    with pytest.raises(abi.AkvError) as e:
        idx.insert(4, [("append", 2), ("drop", [(1, 3)])], [1, 2])
    assert e.value.code == abi.AKV_ERANGE
    with pytest.raises(abi.AkvError) as e:
        idx.remove(77)
    assert e.value.code == abi.AKV_ENOSEQ
    assert idx.match([("append", 1)], [9])["kind"] == "none"
    with pytest.raises(abi.AkvError):
        PrefixIndex(3)
