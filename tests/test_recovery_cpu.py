"""The library's recovery planner (akv_restore_plan_recovery, host code of
libakv, no GPU work) against the oracle's (oracle/akv_recovery.py) on the
Figure 10 program and random programs, and its argument checks."""
import json
import os

import numpy as np
import pytest

from agent_kv_cache_gb300 import abi, build
import oracle.akv_recovery as R

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()


def _flags(n, tokens):
    f = np.zeros(n, np.uint8)
    f[list(tokens)] = 1
    return f


def _random_program(rng, n_ops):
    prog, n = [], 0
    for _ in range(n_ops):
        u = rng.random()
        if u < 0.5 or n == 0:
            k = int(rng.integers(1, 40))
            prog.append(("append", k))
            n += k
        elif u < 0.85:
            ranges = []
            for _ in range(int(rng.integers(1, 4))):
                b = int(rng.integers(0, n))
                ranges.append((b, int(min(n, b + rng.integers(1, 20)))))
            prog.append(("drop", ranges))
        else:
            prog.append(("repos",))
    return prog, n


def test_figure10_cases():
    with open(os.path.join(GOLDEN, "recovery_fig10.json")) as f:
        g = json.load(f)
    prog = [("append", op[1]) if op[0] == "append" else
            ("drop", [tuple(r) for r in op[1]]) if op[0] == "drop" else ("repos",)
            for op in g["ops"]]
    for case in g["cases"]:
        need = None if case["need"] is None else _flags(6, case["need"])
        got = abi.akv_restore_plan_recovery(prog, 6, _flags(6, case["missing"]), need)
        assert got == case["tokens"], case["why"]


@pytest.mark.parametrize("seed", range(6))
def test_random_programs_match_oracle(seed):
    rng = np.random.default_rng(seed)
    for _ in range(30):
        prog, n = _random_program(rng, int(rng.integers(1, 25)))
        p_miss = rng.random()
        missing = {t for t in range(n) if rng.random() < p_miss}
        need = None if rng.random() < 0.5 else {t for t in range(n) if rng.random() < 0.3}
        want, _ = R.plan_recovery(prog, missing, need)
        got = abi.akv_restore_plan_recovery(prog, n, _flags(n, missing),
                                            None if need is None else _flags(n, need))
        assert got == want


def test_argument_checks():
    prog = [("append", 3), ("drop", [(0, 2)])]
    with pytest.raises(abi.AkvError) as e:
        abi.akv_restore_plan_recovery(prog + [("append", 1)], 3, np.zeros(3, np.uint8))
    assert e.value.code == abi.AKV_EINVAL            # appends 4 tokens, not 3
    with pytest.raises(abi.AkvError) as e:
        abi.akv_restore_plan_recovery([("append", 2), ("drop", [(1, 5)])], 2, np.zeros(2, np.uint8))
    assert e.value.code == abi.AKV_ERANGE
    assert abi.akv_restore_plan_recovery(prog, 3, np.zeros(3, np.uint8)) == []
    assert abi.akv_restore_plan_recovery([], 0, np.zeros(0, np.uint8)) == []
