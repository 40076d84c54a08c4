"""CUDA library vs the CPU oracle, element by element, through the C ABI.

Sizes are ones the oracle finishes in seconds while still spanning several
pages/tiles with ragged tails; the full-size workloads are covered by
``test_gpu_fullsize.py``.
"""
import json
import os

import numpy as np
import pytest
import torch

from agent_kv_cache_gb300 import Cache, abi, build
from workloads import synth, traces
from twin import ATTN_TOL, Twin

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    abi.lib()


def test_tiny_workload():
    """1 layer, 8/2 heads, D 64, fp32, 512 tokens, 3 seeded spans dropped,
    reposition, then one decode step."""
    spans = traces.tiny_spans(traces.seed_for(0))
    t = Twin(layers=1, hq=8, hkv=2, head_dim=64, page_size=16, dtype="fp32",
             rope_theta=1e4, max_pages=96, max_seqs=2, max_slots=1024,
             seed=traces.seed_for(0))
    s = t.create()
    t.append([s], [512])
    t.check(s)
    t.drop(s, spans)
    t.check(s)
    t.reposition([s])
    t.check(s)
    t.append([s], [1])
    t.check(s)
    t.decode([s], 0)


def test_fig10_positions_through_library():
    g = json.load(open(os.path.join(GOLD, "fig10_positions.json")))
    t = Twin(page_size=1, max_pages=64, max_slots=64)
    s = t.create()
    name_of = {}
    for op in g["ops"]:
        if op[0] == "append":
            name_of[t.gpu.info(s)["n_logical"]] = op[1]
            t.append([s], [1])
        elif op[0] == "drop":
            idx = {n: i for i, n in name_of.items()}
            t.drop(s, [(idx[n], idx[n] + 1) for n in op[1]])
        elif op[0] == "repos":
            t.reposition([s])
        else:
            keep = t.gpu.keep_mask(s)
            seen = {name_of[int(l)]: int(p) for l, p, a in
                    zip(t.gpu.logical(s), t.gpu.positions(s), keep) if a}
            assert seen == op[2]
            assert t.gpu.info(s)["next_pos"] - 1 == op[2][op[1]]
        t.check(s)
    t.decode([s], 0)


CONFIGS = [
    # dtype, page, G, D
    ("bf16", 16, 4, 128),
    ("bf16", 16, 8, 64),
    ("bf16", 16, 1, 128),
    ("bf16", 1, 4, 64),
    ("bf16", 64, 2, 128),
    ("fp32", 16, 4, 64),
    ("fp32", 4, 16, 128),
]


@pytest.mark.parametrize("dtype,page,G,D", CONFIGS)
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_operation_sequences(dtype, page, G, D, seed):
    rng = np.random.default_rng(1000 * seed + page + G + D)
    hkv = 2
    t = Twin(layers=2, hq=hkv * G, hkv=hkv, head_dim=D, page_size=page, dtype=dtype,
             rope_theta=1e4 if D == 64 else 5e5, max_pages=2048, max_seqs=8,
             max_slots=1024, seed=seed)
    seqs = [t.create()]
    t.append(seqs, [int(rng.integers(1, 200))])
    step = 0
    for _ in range(10):
        g = seqs[int(rng.integers(0, len(seqs)))]
        op = rng.choice(["append", "drop", "drop", "repos", "fork", "decode"])
        n = t.gpu.info(g)["n_logical"]
        if op == "append":
            t.append([g], [int(rng.integers(1, 120))])
        elif op == "drop" and n:
            rs = []
            for _ in range(int(rng.integers(1, 4))):
                b = int(rng.integers(0, n))
                rs.append((b, int(rng.integers(b, min(n, b + 90) + 1))))
            t.drop(g, rs)
        elif op == "repos":
            t.reposition([g])
        elif op == "fork" and len(seqs) < 6:
            seqs.append(t.fork(g))
        elif op == "decode":
            t.append(seqs, [1] * len(seqs))
            t.decode(seqs, step)
            step += 1
        for s in seqs:
            t.check(s)
    t.append(seqs, [1] * len(seqs))
    t.decode(seqs, step)


def test_batched_reposition_and_decode():
    t = Twin(layers=3, hq=16, hkv=4, head_dim=128, page_size=16, dtype="bf16",
             rope_theta=5e5, max_pages=4096, max_seqs=8, max_slots=4096)
    seqs = [t.create() for _ in range(5)]
    t.append(seqs, [700, 1, 16, 333, 1500])
    t.drop(seqs[0], [(0, 100), (300, 500)])
    t.drop(seqs[1], [(0, 1)])
    t.drop(seqs[3], [(5, 6), (40, 41), (100, 332)])
    t.drop(seqs[4], [(1024, 1500)])
    t.reposition(seqs)
    for s in seqs:
        t.check(s)
    t.append(seqs, [1] * 5)
    t.decode(seqs, 0)
    t.drop(seqs[2], [(0, 17)])           # every token of seq 2 dropped
    t.append(seqs[:2] + seqs[3:], [1] * 4)
    for s in seqs:
        t.check(s)
    t.decode(seqs, 1)                    # seq 2 has nothing active: zeros


@pytest.mark.parametrize("dtype,page,G", [("bf16", 16, 4), ("bf16", 16, 8), ("bf16", 4, 4),
                                          ("fp32", 16, 4)])
def test_poisoned_pool_memory_does_not_leak_into_attention(dtype, page, G):
    """Slots that are not active (dropped, or never written) may hold any bit
    pattern; attention must ignore them.  The pools start filled with NaN."""
    t = Twin(layers=2, hq=2 * G, hkv=2, head_dim=128, page_size=page, dtype=dtype,
             rope_theta=5e5, max_pages=512, max_seqs=4, max_slots=2048, seed=5)
    t.gpu.k_pool.fill_(float("nan"))
    t.gpu.v_pool.fill_(float("nan"))
    a, b = t.create(), t.create()
    t.append([a, b], [37, 301])                 # ragged tails: never-written slots
    t.drop(b, [(3, 40), (100, 101)])
    t.append([a, b], [1, 1])
    t.decode([a, b], 0)
    t.reposition([b])
    t.append([a, b], [1, 1])
    for s in (a, b):
        t.check(s)
    t.decode([a, b], 1)


def test_long_splits_wrap_the_stage_ring():
    """Splits of ~50 tiles: every shared-memory stage is refilled many times."""
    t = Twin(layers=1, hq=32, hkv=8, head_dim=128, page_size=16, dtype="bf16",
             rope_theta=5e5, max_pages=6000, max_seqs=4, max_slots=17000, seed=9)
    seqs = [t.create() for _ in range(4)]
    t.append(seqs, [16000, 15000, 16383, 9000])
    t.drop(seqs[0], [(1000, 5000)])
    t.drop(seqs[2], [(0, 16), (300, 301)])
    t.append(seqs, [1, 1, 1, 1])
    t.decode(seqs, 0)
    t.reposition(seqs[:3])
    t.append(seqs, [1, 1, 1, 1])
    for s in seqs:
        t.check(s, kv=False)
    t.decode(seqs, 1)


PARTIAL = [
    # dtype, page, G, D, rope_dim
    ("bf16", 16, 4, 128, 64),
    ("bf16", 16, 8, 64, 32),
    ("bf16", 32, 2, 128, 96),
    ("fp32", 4, 2, 128, 48),
    ("bf16", 1, 16, 64, 16),
]


@pytest.mark.parametrize("dtype,page,G,D,R", PARTIAL)
def test_partial_rope_operation_sequences(dtype, page, G, D, R):
    """Only the first R dims rotate; the rest are copied by append and
    reposition and read as they are by decode."""
    rng = np.random.default_rng(R * 7 + D + page)
    t = Twin(layers=2, hq=2 * G, hkv=2, head_dim=D, page_size=page, dtype=dtype,
             rope_theta=5e5, max_pages=2048, max_seqs=6, max_slots=1024, seed=R, rope_dim=R)
    seqs = [t.create(), t.create()]
    t.append(seqs, [150, 333])
    for step in range(6):
        g = seqs[step % 2]
        n = t.gpu.info(g)["n_logical"]
        b = int(rng.integers(0, n - 1))
        t.drop(g, [(b, min(n, b + int(rng.integers(1, 60))))])
        if step % 2:
            t.reposition(seqs)
        t.append(seqs, [1, 1])
        for s in seqs:
            t.check(s)
        t.decode(seqs, step)


@pytest.mark.parametrize("dtype,page,G,D", [("bf16", 16, 4, 128), ("bf16", 16, 8, 64),
                                            ("fp32", 16, 2, 64), ("bf16", 4, 4, 128)])
def test_sliding_window_over_positions(dtype, page, G, D):
    """Windows count positions: after a drop without a reposition the window
    holds fewer keys; windowed and full layers alternate (two plans)."""
    t = Twin(layers=4, hq=2 * G, hkv=2, head_dim=D, page_size=page, dtype=dtype,
             rope_theta=1e4, max_pages=4096, max_seqs=6, max_slots=8192, seed=3)
    seqs = [t.create() for _ in range(3)]
    t.append(seqs, [2000, 777, 64])
    t.set_window(1, 128)
    t.set_window(3, 40)
    step = 0
    for w1, w3 in [(128, 40), (1, 5000), (16, 300), (700, 1)]:
        t.set_window(1, w1)
        t.set_window(3, w3)
        t.append(seqs, [1, 1, 1])
        t.decode(seqs, step)
        step += 1
    t.drop(seqs[0], [(1900, 1995), (1500, 1510)])   # gaps inside the windows
    t.drop(seqs[2], [(0, 64)])
    t.append(seqs, [1, 1, 1])
    for w1, w3 in [(128, 40), (10, 200), (3000, 2)]:
        t.set_window(1, w1)
        t.set_window(3, w3)
        t.decode(seqs, step)
        step += 1
    t.reposition(seqs)
    t.append(seqs, [1, 1, 1])
    t.decode(seqs, step)
    for s in seqs:
        t.check(s)


def _random_program(rng, n_tokens, n_ops):
    prog, appended = [], 0
    per = max(1, n_tokens // max(1, n_ops // 2))
    while appended < n_tokens:
        kind = rng.choice(["append", "append", "drop", "repos"]) if appended else "append"
        if kind == "append":
            k = int(min(n_tokens - appended, rng.integers(1, per + 1)))
            prog.append(("append", k))
            appended += k
        elif kind == "drop":
            b = int(rng.integers(0, appended))
            prog.append(("drop", [(b, int(min(appended, b + rng.integers(1, 40))))]))
        else:
            prog.append(("repos",))
    return prog


RESTORE = [
    # dtype, page, G, D, rope_dim, window, kernel (1: tensor cores, two query
    # tiles per CTA; 2: tensor cores, one tile per CTA; 0: CUDA cores)
    ("bf16", 16, 4, 128, 0, 0, 1),
    ("bf16", 16, 4, 128, 0, 0, 2),
    ("bf16", 16, 4, 128, 0, 0, 0),
    ("bf16", 16, 8, 64, 0, 0, 1),
    ("bf16", 16, 8, 64, 0, 0, 2),
    ("bf16", 16, 8, 64, 0, 0, 0),
    ("bf16", 16, 1, 128, 0, 0, 1),
    ("bf16", 16, 2, 64, 0, 0, 1),
    ("bf16", 8, 16, 64, 32, 0, 1),
    ("bf16", 8, 16, 64, 32, 0, 2),
    ("fp32", 16, 2, 64, 0, 0, 1),
    ("bf16", 16, 4, 128, 64, 0, 1),
    ("bf16", 16, 4, 128, 64, 0, 0),
    ("bf16", 16, 4, 128, 0, 24, 1),
    ("bf16", 16, 4, 128, 0, 24, 2),
    ("bf16", 16, 2, 128, 0, 100, 1),
    ("fp32", 4, 16, 128, 32, 7, 1),
]


@pytest.mark.parametrize("dtype,page,G,D,R,W,tc", RESTORE)
@pytest.mark.parametrize("seed", [1, 2])
def test_restore_attention_random_programs(dtype, page, G, D, R, W, tc, seed):
    """Every appended token's restore attention equals its attention at the
    time it was appended (oracle replay), keys dropped later included.
    bf16 runs the tensor-core kernel in both forms and the CUDA-core one."""
    rng = np.random.default_rng(seed * 100 + D + G + R + W)
    t = Twin(layers=2, hq=2 * G, hkv=2, head_dim=D, page_size=page, dtype=dtype,
             rope_theta=1e4, max_pages=512, max_seqs=4, max_slots=2048, seed=seed, rope_dim=R)
    t.gpu.set_restore_tensor_cores(tc)
    if W:
        t.set_window(1, W)
    prog = _random_program(rng, int(rng.integers(150, 400)), 16)
    t.restore(prog, layer=0)
    t.restore(prog, layer=1)
    # the cache state is rebuilt by replaying the program through the API
    s = t.create()
    for op in prog:
        if op[0] == "append":
            t.append([s], [op[1]])
        elif op[0] == "drop":
            t.drop(s, op[1])
        else:
            t.reposition([s])
    t.check(s)


@pytest.mark.parametrize("tc", [1, 2, 0])
def test_restore_attention_long_program(tc):
    """A 2000-token program with few repositions: eras of thousands of keys
    (many 64-key tiles per query tile), drops that empty whole tiles, and a
    query tile that straddles an era boundary."""
    rng = np.random.default_rng(77)
    prog, appended = [], 0
    while appended < 2000:
        n = int(rng.integers(1, 300))
        prog.append(("append", n))
        appended += n
        u = rng.random()
        if u < 0.5:
            b = int(rng.integers(0, appended))
            prog.append(("drop", [(b, int(min(appended, b + rng.integers(1, 200))))]))
        elif u < 0.7:
            prog.append(("repos",))
    t = Twin(layers=2, hq=8, hkv=2, head_dim=128, page_size=16, dtype="bf16", rope_theta=5e5,
             max_pages=1024, max_seqs=4, max_slots=8192, seed=5)
    t.gpu.set_restore_tensor_cores(tc)
    t.set_window(1, 700)
    t.restore(prog, layer=0)
    t.restore(prog, layer=1)


@pytest.mark.parametrize("tc", [1, 2, 0])
def test_restore_recovers_only_the_planned_tokens(tc):
    """A restore after some tokens lost their KV: the library's recovery plan
    (which equals the oracle's) picks the tokens to recompute, and restore
    attention over just those tokens gives each its original attention
    (oracle replay of those tokens) and leaves every other output row alone.
    Also: nothing selected, and every token selected."""
    from oracle.akv_recovery import plan_recovery
    rng = np.random.default_rng(31 + tc)
    t = Twin(layers=2, hq=8, hkv=2, head_dim=128, page_size=16, dtype="bf16", rope_theta=5e5,
             max_pages=512, max_seqs=4, max_slots=4096, seed=9)
    t.gpu.set_restore_tensor_cores(tc)
    for trial in range(3):
        prog = _random_program(rng, int(rng.integers(300, 700)), 20)
        n = sum(op[1] for op in prog if op[0] == "append")
        missing = np.zeros(n, np.uint8)
        b = int(rng.integers(0, n // 2))
        missing[b:b + int(rng.integers(20, n // 2))] = 1          # an evicted stretch
        missing[rng.random(n) < 0.1] = 1                          # and scattered pages
        plan = Cache.plan_recovery(prog, n, missing)
        assert plan == plan_recovery(prog, set(np.flatnonzero(missing).tolist()))[0]
        assert 0 < len(plan) < n
        t.restore_tokens(prog, 0, plan)
    prog = _random_program(rng, 200, 10)
    n = sum(op[1] for op in prog if op[0] == "append")
    t.restore_tokens(prog, 1, [])
    t.restore_tokens(prog, 1, list(range(n)))


def test_restore_attention_figure10_program():
    g = json.load(open(os.path.join(GOLD, "fig10_positions.json")))
    names = [op[1] for op in g["ops"] if op[0] == "append"]
    idx = {nm: i for i, nm in enumerate(names)}
    prog = []
    for op in g["ops"]:
        if op[0] == "append":
            prog.append(("append", 1))
        elif op[0] == "drop":
            prog.append(("drop", [(idx[x], idx[x] + 1) for x in op[1]]))
        elif op[0] == "repos":
            prog.append(("repos",))
    t = Twin(layers=1, hq=8, hkv=2, head_dim=64, page_size=16, dtype="bf16", seed=10)
    t.restore(prog)
    t2 = Twin(layers=1, hq=8, hkv=2, head_dim=64, page_size=16, dtype="fp32", seed=10)
    t2.restore(prog)


def test_restore_rejects_bad_programs():
    t = Twin(layers=1, hq=8, hkv=2, head_dim=64, page_size=16, dtype="bf16", max_slots=64)
    z = torch.zeros((10, 8, 64), dtype=torch.bfloat16, device="cuda")
    zk = torch.zeros((10, 2, 64), dtype=torch.bfloat16, device="cuda")
    for prog, code in [([("append", 9)], abi.AKV_EINVAL),
                       ([("append", 11)], abi.AKV_EINVAL),
                       ([("append", 5), ("drop", [(3, 7)]), ("append", 5)], abi.AKV_ERANGE)]:
        with pytest.raises(abi.AkvError) as e:
            t.gpu.restore_attention(prog, 0, z, zk, zk)
        assert e.value.code == code
    t3 = Twin(layers=1, hq=8, hkv=2, head_dim=64, page_size=16, dtype="bf16", max_slots=8)
    with pytest.raises(abi.AkvError) as e:          # positions reach max_slots
        t3.gpu.restore_attention([("append", 10)], 0, z, zk, zk)
    assert e.value.code == abi.AKV_ECAPACITY


def _history(t, ops, toks):
    s = t.create()
    names = {}
    for op in ops:
        if op[0] == "append":
            names[op[1]] = t.gpu.info(s)["n_logical"]
            t.append([s], [1], token_ids=[toks[op[1]]])
        elif op[0] == "drop":
            t.drop(s, [(names[n], names[n] + 1) for n in op[1]])
        else:
            t.reposition([s])
    return s


def test_history_keys_figure5_and_figure11():
    g = json.load(open(os.path.join(GOLD, "fig5_histories.json")))
    t = Twin(page_size=1, max_pages=256, max_seqs=16, max_slots=64)
    seqs = {name: _history(t, ops, g["tokens"]) for name, ops in g["paths"].items()}
    keys = {name: t.gpu.history_key(s) for name, s in seqs.items()}
    assert len(set(keys.values())) == len(keys), keys
    again = _history(t, g["paths"]["fig5_2"], g["tokens"])
    assert t.gpu.history_key(again) == keys["fig5_2"]


def test_history_key_equality_matches_operation_logs():
    rng = np.random.default_rng(7)
    t = Twin(page_size=4, max_pages=4096, max_seqs=64, max_slots=256)
    seqs = []
    for i in range(40):
        s = t.create()
        for _ in range(int(rng.integers(1, 5))):
            op = int(rng.integers(0, 3))
            n = t.gpu.info(s)["n_logical"]
            if op == 0 or n == 0:
                k = int(rng.integers(1, 3))
                t.append([s], [k], token_ids=list(rng.integers(0, 2, size=k)))
            elif op == 1:
                b = int(rng.integers(0, n))
                t.drop(s, [(b, b + 1)])
            else:
                t.reposition([s])
        seqs.append(s)
    for a in seqs:
        for b in seqs:
            same_log = t.orc.history(t.o[a]) == t.orc.history(t.o[b])
            assert t.history_equal(a, b) == same_log
    # appending n tokens at once == n appends of one
    a, b = t.create(), t.create()
    t.append([a], [5], token_ids=[1, 2, 3, 4, 5])
    t.append([b], [2], token_ids=[1, 2])
    t.append([b], [3], token_ids=[3, 4, 5])
    assert t.history_equal(a, b)


def test_copy_on_write_isolation():
    t = Twin(layers=2, hq=8, hkv=2, head_dim=64, page_size=16, dtype="bf16",
             rope_theta=1e4, max_pages=512, max_seqs=8, max_slots=2048)
    base = t.create()
    t.append([base], [203])                     # ragged: tail page partly filled
    pages0, _ = t.gpu.page_table(base)
    snap_k = t.gpu.k_pool[:, torch.from_numpy(pages0.astype(np.int64)).cuda()].clone()
    snap_v = t.gpu.v_pool[:, torch.from_numpy(pages0.astype(np.int64)).cuda()].clone()
    kids = [t.fork(base) for _ in range(3)]
    for p in pages0:
        assert t.gpu.refcount(int(p)) == 4
    t.drop(kids[0], [(40, 90)])
    t.reposition([kids[0]])
    t.append([kids[1]], [30])                   # writes into the shared tail: copy-on-write
    t.drop(kids[2], [(0, 5)])
    t.reposition([kids[2]])
    t.append(kids, [1, 1, 1])
    for s in [base] + kids:
        t.check(s)
    idx = torch.from_numpy(pages0.astype(np.int64)).cuda()
    # bit patterns, so never-written slots (any bits, NaN included) compare too
    assert torch.equal(t.gpu.k_pool[:, idx].view(torch.int16), snap_k.view(torch.int16))
    assert torch.equal(t.gpu.v_pool[:, idx].view(torch.int16), snap_v.view(torch.int16))
    # kept prefix of kids[0] (pages before the first drop) is still shared
    p0, _ = t.gpu.page_table(kids[0])
    assert list(p0[:2]) == list(pages0[:2])
    t.decode([base] + kids, 0)
    for s in kids + [base]:
        t.free(s)
    free, used = t.gpu.pool_stats()
    assert used == 0 and free == 512


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("G,D,n_kids,rope", [(4, 128, 19, 0), (8, 128, 9, 0), (2, 64, 20, 0),
                                              (1, 64, 18, 0), (4, 64, 37, 0), (4, 128, 11, 64),
                                              (8, 64, 7, 32)])
def test_branches_share_pages_in_decode(G, D, n_kids, rope, mode):
    """Branches forked from one prefix hold the same pages: a decode call
    reads them once for all rows that hold them identically (mode 1: the
    tensor-core shared-prefix items of up to 128 query rows; mode 2: shared
    items of the one-row kernel, two rows each).  Every row must still get
    exactly its own attention, including rows whose keep bits on a shared
    page differ (dropped without reposition), rows that repositioned (kept
    leading pages stay shared), rows that copied the tail on append, and the
    partly filled shared tail page; rope > 0: only the first rope dims rotate."""
    hkv = 2
    t = Twin(layers=2, hq=hkv * G, hkv=hkv, head_dim=D, page_size=16, dtype="bf16",
             rope_theta=5e5 if D == 128 else 1e4, max_pages=4096, max_seqs=n_kids + 4,
             max_slots=2048, seed=11, rope_dim=rope)
    root = t.create()
    t.append([root], [1000])                    # 62 full pages and a partly filled tail
    kids = [t.fork(root) for _ in range(n_kids)]
    rng = np.random.default_rng(G * 100 + D)
    for i, k in enumerate(kids):
        kind = i % 5
        if kind == 1:                            # keep bits differ on a few shared pages
            b = int(rng.integers(200, 700))
            t.drop(k, [(b, b + int(rng.integers(1, 60)))])
        elif kind == 2:                          # leading pages stay shared
            b = int(rng.integers(300, 900))
            t.drop(k, [(b, b + int(rng.integers(20, 90)))])
            t.reposition([k])
        elif kind == 3:                          # tail copied on write
            t.append([k], [int(rng.integers(1, 40))])
    rows = [root] + kids + [kids[0]]             # the same sequence twice is allowed
    t.gpu.set_decode_sharing(mode)
    t.decode(rows, 0)
    st = t.gpu.decode_plan_stats()
    assert st["shared_items"] > 0 and st["members"] > 0, st
    # without sharing: against the oracle too, and close to the shared plan
    # (the softmax weights are rounded to bf16 against each split's running
    # maximum, so other split boundaries move the result by bf16 roundings)
    t.gpu.set_decode_sharing(False)
    t.decode(rows, 0)
    assert t.gpu.decode_plan_stats()["shared_items"] == 0
    outs = []
    for share in (mode, 0):
        t.gpu.set_decode_sharing(share)
        q = torch.randn(len(rows), t.hq, D, generator=torch.Generator().manual_seed(5))
        outs.append(t.gpu.decode_attention(1, q.to(torch.bfloat16).cuda(), rows).cpu())
    diff = (outs[0] - outs[1]).abs()
    assert diff.max() <= 1e-2 and diff.mean() <= 1e-3, (diff.max(), diff.mean())
    t.gpu.set_decode_sharing(mode)
    # an output buffer that is only 4-byte aligned gets the same bits
    q = torch.randn(len(rows), t.hq, D, generator=torch.Generator().manual_seed(5))
    q = q.to(torch.bfloat16).cuda()
    flat = torch.empty(len(rows) * t.hq * D + 1, dtype=torch.float32, device="cuda")
    odd = flat[1:].view(len(rows), t.hq, D)
    t.gpu.decode_attention(1, q, rows, odd)
    assert torch.equal(odd.cpu(), outs[0])
    # and a query that is only 2-byte aligned
    qflat = torch.empty(q.numel() + 1, dtype=torch.bfloat16, device="cuda")
    qodd = qflat[1:].view_as(q)
    qodd.copy_(q)
    got = t.gpu.decode_attention(1, qodd, rows)
    assert torch.equal(got.cpu(), outs[0])
    t.append(rows[:-1], [1] * (len(rows) - 1))   # every row copies its tail
    t.gpu.set_decode_sharing(mode)
    t.decode(rows[:-1], 1)
    assert t.gpu.decode_plan_stats()["shared_items"] > 0
    # appends only: the shared part of the plan is reused, the tails grow
    for step in (2, 3):
        t.append(rows[:-1], [1 + step] * (len(rows) - 1))
        t.decode(rows[:-1], step)
    # a drop in one branch changes its layout: the plan is found again
    t.drop(kids[1], [(100, 140)])
    t.append(rows[:-1], [1] * (len(rows) - 1))
    t.decode(rows[:-1], 4)
    assert t.gpu.decode_plan_stats()["shared_items"] > 0
    for s in rows[:-1]:
        t.check(s)


def test_errors_leave_state_unchanged():
    t = Twin(layers=1, hq=4, hkv=2, head_dim=64, page_size=16, dtype="bf16",
             rope_theta=1e4, max_pages=16, max_seqs=2, max_slots=400)
    s = t.create()
    t.append([s], [100])                          # 7 pages, 9 free

    def snapshot():
        return (t.gpu.info(s), t.gpu.keep_mask(s).tolist(), t.gpu.page_table(s)[0].tolist(),
                t.gpu.history_key(s), t.gpu.pool_stats())

    before = snapshot()
    for bad in ([(0, 101)], [(-1, 3)], [(7, 3)]):
        with pytest.raises(abi.AkvError) as e:
            t.gpu.drop(s, bad)
        assert e.value.code == abi.AKV_ERANGE
    with pytest.raises(abi.AkvError) as e:
        t.gpu.drop(12345, [(0, 1)])
    assert e.value.code == abi.AKV_ENOSEQ
    k = torch.zeros((1, 320, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(abi.AkvError) as e:        # 100 + 320 > max_slots
        t.gpu.append([s], [320], k, k)
    assert e.value.code == abi.AKV_ECAPACITY
    k = torch.zeros((1, 200, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(abi.AkvError) as e:        # needs 12 more pages, 9 free
        t.gpu.append([s], [200], k, k)
    assert e.value.code == abi.AKV_ENOPAGES
    t2 = t.create()
    with pytest.raises(abi.AkvError) as e:        # max_seqs == 2
        t.gpu.seq_create()
    assert e.value.code == abi.AKV_ECAPACITY
    t.free(t2)
    with pytest.raises(abi.AkvError) as e:
        t.gpu.reposition([s, s])
    assert e.value.code == abi.AKV_EINVAL
    assert snapshot() == before
    t.check(s)
    # a reposition needing more fresh pages than are free is refused as a whole
    # (the fresh pages are taken before the old ones are released)
    t.drop(s, [(0, 1)])
    before = snapshot()
    other = t.create()
    t.append([other], [96])                       # 6 pages: 3 left free
    with pytest.raises(abi.AkvError) as e:
        t.gpu.reposition([s])                     # needs 7
    assert e.value.code == abi.AKV_ENOPAGES
    assert snapshot()[:4] == before[:4]
    t.check(s)
    t.free(other)
    t.reposition([s])
    t.check(s)
    t.free(s)
    assert t.gpu.pool_stats() == (16, 0)


def test_bounded_waits_time_out_and_recover():
    """A one-poll wait limit makes the tcgen05 restore kernel's mbarrier
    waits run out: it drains its own copies and MMAs, reports AKV_DERR_WAIT
    in the error word and returns (no hang, no fault). The tensor-core
    decode under the same limit either completes or reports the same bit
    (one poll may already see its data land), never anything else. With the
    limit restored both calls match the oracle again."""
    t = Twin(layers=1, hq=8, hkv=2, head_dim=128, page_size=16, dtype="bf16", max_pages=2048,
             max_seqs=8, max_slots=4096, seed=3)
    seqs = [t.create() for _ in range(4)]
    t.append(seqs, [3000] * 4)
    prog = [("append", 120), ("drop", [(10, 40)]), ("repos",), ("append", 30)]
    n = 150
    q = torch.zeros((n, 8, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((n, 2, 128), dtype=torch.bfloat16, device="cuda")
    qd = torch.zeros((4, 8, 128), dtype=torch.bfloat16, device="cuda")
    abi.akv_set_wait_limit(t.gpu.handle, 1)
    t.gpu.decode_attention(0, qd, seqs)
    w_dec = t.gpu.sync_errors()
    t.gpu.restore_attention(prog, 0, q, kv, kv)
    w_res = t.gpu.sync_errors()
    abi.akv_set_wait_limit(t.gpu.handle, 1 << 22)
    assert w_res == abi.AKV_DERR_WAIT, w_res
    assert w_dec in (0, abi.AKV_DERR_WAIT), w_dec
    assert t.gpu.sync_errors() == 0
    t.decode(seqs, step=0)
    t.restore(prog)
    for g in seqs:
        t.check(g)


def test_decode_back_to_back_and_one_at_a_time():
    """The one-row decode kernel splits a call for a quarter of the GPU's
    block slots when decode calls come back to back (the next call's blocks
    start in the rest) and for a whole wave when a call runs on its own; the
    choice is made on the device, per call.  Calls enqueued back to back
    (three rounds over every layer, no wait in between) and the same calls
    one at a time (a synchronisation before each) must all match the oracle,
    and both sets must agree within the attention tolerance."""
    build()
    t = Twin(layers=4, hq=32, hkv=8, head_dim=128, page_size=16, dtype="bf16", rope_theta=5e5,
             max_pages=2048, max_seqs=8, max_slots=4096, seed=21)
    seqs = [t.create() for _ in range(4)]
    t.append(seqs, [3000, 1000, 2500, 400])
    t.drop(seqs[0], [(100, 900)])
    t.drop(seqs[2], [(2000, 2400)])
    t.reposition([seqs[0], seqs[2]])
    t.append(seqs, [1, 1, 1, 1])
    L = t.L
    q = [np.stack([synth.query(t.seed, t.tag[s], l, 0, t.hq, t.d, t.width) for s in seqs])
         for l in range(L)]
    qd = [torch.from_numpy(x).to(torch.bfloat16).cuda() for x in q]
    want = [t.orc.attention(l, q[l], [t.o[s] for s in seqs]) for l in range(L)]
    outs = [torch.empty((len(seqs), t.hq, t.d), dtype=torch.float32, device="cuda")
            for _ in range(3 * L)]
    torch.cuda.synchronize()
    for r in range(3):
        for l in range(L):
            t.gpu.decode_attention(l, qd[l], seqs, out=outs[r * L + l])
    torch.cuda.synchronize()
    alone = []
    for l in range(L):
        torch.cuda.synchronize()
        alone.append(t.gpu.decode_attention(l, qd[l], seqs).clone())
        torch.cuda.synchronize()
    tmax, tmean = ATTN_TOL["bf16"]
    for i, o in enumerate(outs + alone):
        l = i % L
        err = np.abs(o.double().cpu().numpy() - want[l])
        assert err.max() <= tmax and err.mean() <= tmean, (i, err.max(), err.mean())
    for l in range(L):
        d = (outs[l] - alone[l]).abs()
        assert d.max().item() <= tmax and d.mean().item() <= tmean
    assert t.gpu.sync_errors() == 0
