"""History-keyed prefix sharing and drop-aware eviction on the GPU, against
the oracle.

A family of programs shares one trunk; each program is replayed on the GPU
(append with token ids, drop, reposition) and published.  A request is then
matched and materialised with ``akv_prefix_fork``; the match must equal the
oracle's (``oracle/akv_prefix.py``), the child's keep mask, positions,
logical map and page table must equal the oracle's plan bit for bit, its
keys must be within the chained-rounding bound of a cache built directly
from the request prefix (``OracleCache``), V bit-exact, and after the
request's remaining operations the child's decode attention must equal the
oracle's.  K/V of logical token t come from one seeded stream per family,
so equal prefixes have equal inputs.
"""
import numpy as np
import pytest
import torch

from agent_kv_cache_gb300 import Cache, PrefixIndex, abi, build
import oracle.akv_prefix as P
from oracle.akv_oracle import OracleCache
from twin import ATTN_TOL, check_key_step, key_tolerance
from workloads import synth

pytestmark = pytest.mark.gpu


class Family:
    def __init__(self, dtype="bf16", D=64, G=4, S=16, L=2, seed=3, max_pages=8192, theta=1e4):
        build()
        self.L, self.hkv, self.hq, self.D, self.S, self.dtype = L, 2, 2 * G, D, S, dtype
        self.gpu = Cache(L, self.hq, self.hkv, D, S, dtype, max_pages, 48, 4096, theta)
        self.idx = PrefixIndex(S)
        self.theta = theta
        self.seed, self.tag = seed, 1
        self.width = synth.width_for(dtype)
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.entries = {}     # entry id -> records
        self.use = {}         # entry id -> last use (mirrors the index clock)
        self.clock = 0

    def kv(self, t0, n):
        k = synth.kv_tokens(self.seed, self.tag, synth.KIND_K, range(self.L), t0, n, self.hkv,
                            self.D, self.width)
        v = synth.kv_tokens(self.seed, self.tag, synth.KIND_V, range(self.L), t0, n, self.hkv,
                            self.D, self.width)
        return k, v

    def run(self, seq, program, ids, t0=0):
        """Apply a program to a GPU sequence whose first t0 tokens exist."""
        t = t0
        for op in program:
            if op[0] == "append":
                n = op[1]
                k, v = self.kv(t, n)
                dev = lambda x: torch.from_numpy(x).to(self.tdtype).cuda().contiguous()
                self.gpu.append([seq], [n], dev(k), dev(v), list(ids[t:t + n]))
                t += n
            elif op[0] == "drop":
                self.gpu.drop(seq, op[1])
            else:
                self.gpu.reposition([seq])
        torch.cuda.synchronize()
        return t

    def oracle(self, recs):
        """OracleCache sequence built directly from records."""
        c = OracleCache(self.hq, self.hkv, self.D, self.theta, self.dtype,
                        layers=range(self.L), page_size=self.S)
        sid = c.create()
        t = 0
        for r in recs:
            if r[0] == "T":
                k, v = self.kv(t, 1)
                c.append(sid, k, v, [r[1]])
                t += 1
            elif r[0] == "D":
                c.drop(sid, list(r[1]))
            else:
                c.reposition(sid)
        return c, sid

    def publish(self, program, ids):
        s = self.gpu.seq_create()
        self.run(s, program, ids)
        e = self.gpu.prefix_publish(self.idx, s, program, ids)
        self.gpu.seq_free(s)
        recs = P.records(program, ids)
        if e not in self.entries:
            self.entries[e] = recs
        self.clock += 1
        self.use[e] = self.clock
        return e


def _trunk(rng, n_ops, max_append=40):
    prog, n = [], 0
    for _ in range(n_ops):
        u = rng.random()
        if u < 0.55 or n == 0:
            k = int(rng.integers(1, max_append))
            prog.append(("append", k))
            n += k
        elif u < 0.85:
            b = int(rng.integers(0, n))
            prog.append(("drop", [(b, int(min(n, b + rng.integers(1, 25))))]))
        else:
            prog.append(("repos",))
    return prog, n


def _branch(rng, base, nb):
    tail, m = [], nb
    for _ in range(int(rng.integers(1, 6))):
        u = rng.random()
        if u < 0.5 or m == 0:
            k = int(rng.integers(1, 30))
            tail.append(("append", k))
            m += k
        elif u < 0.8:
            b = int(rng.integers(0, m))
            tail.append(("drop", [(b, int(min(m, b + rng.integers(1, 20))))]))
        else:
            tail.append(("repos",))
    return base + tail, m


def _remaining(program, m):
    """The part of the program after the match (op_index, op_tokens)."""
    if m["kind"] == "none":
        return list(program)
    rest = list(program[m["op_index"]:])
    if m["op_tokens"]:
        n = rest[0][1] - m["op_tokens"]
        rest = ([("append", n)] if n else []) + rest[1:]
    return rest


def _poison_free_pages(f):
    """NaN bit patterns in every free pool page (any slot a fork leaves
    unwritten would show them)."""
    free = [p for p in range(f.gpu.k_pool.shape[1]) if f.gpu.refcount(p) == 0]
    if free:
        idx = torch.tensor(free, dtype=torch.int64, device="cuda")
        f.gpu.k_pool[:, idx] = float("nan")
        f.gpu.v_pool[:, idx] = float("nan")
        torch.cuda.synchronize()


def _check_child(f, child, req, m, entry_recs):
    n = m["n_records"]
    plan = P.fork_plan(entry_recs, req, n, f.S)
    st = P.State(req[:n])
    info = f.gpu.info(child)
    assert info["n_held"] == plan["n_slots"] and info["n_logical"] == plan["n_logical"]
    held = [t for t in range(len(st.alive)) if st.held[t]]
    np.testing.assert_array_equal(f.gpu.logical(child), held)
    np.testing.assert_array_equal(f.gpu.keep_mask(child), [st.alive[t] for t in held])
    pages, act = f.gpu.page_table(child)
    epages, _ = f.gpu.page_table(m["entry"])
    for k, kind in enumerate(plan["pages"]):
        if kind == "none" and k == len(plan["pages"]) - 1 and plan["n_slots"] % f.S:
            # a partly filled tail page stays held (appends write into it)
            assert pages[k] >= 0 and f.gpu.refcount(int(pages[k])) == 1
        elif kind == "none":
            assert pages[k] < 0
        elif kind == "shared":
            assert pages[k] == epages[k] and f.gpu.refcount(int(pages[k])) >= 2
        else:
            assert pages[k] >= 0 and pages[k] not in set(epages.tolist())
            assert f.gpu.refcount(int(pages[k])) == 1
    np.testing.assert_array_equal(act, [k for k, kind in enumerate(plan["pages"]) if kind != "none"])
    # keys and values against a cache built directly from the request prefix
    oc, osid = f.oracle(req[:n])
    os_ = oc.seqs[osid]
    n_rot = sum(1 for r in entry_recs if r[0] == "R") + sum(1 for r in req[:n] if r[0] == "R") + 2
    live = np.array([st.alive[t] for t in held])
    for l in range(f.L):
        k, v = f.gpu.read_kv(child, l)
        ref = os_.K[l][live]
        err = np.abs(k[live] - ref)
        tol = key_tolerance(ref, f.dtype, n_rot)
        assert not (err > tol).any(), (l, err.max())
        np.testing.assert_array_equal(v[live], os_.V[l][live])
    # step-wise: each needed key is the entry's stored key, read from its slot
    # (its stored position) and rotated to the request's position; the
    # entry's stored keys are first checked against a cache built from the
    # entry's own records (chained bound)
    eo, esid = f.oracle(entry_recs)
    es = eo.seqs[esid]
    n_rot_e = sum(1 for r in entry_recs if r[0] == "R") + 1
    mv = sorted(plan["moves"].values())
    dst = np.array([x[0] for x in mv], dtype=np.int64)
    src = np.array([x[1] for x in mv], dtype=np.int64)
    for l in range(f.L):
        ke, _ = f.gpu.read_kv(m["entry"], l)
        k, _ = f.gpu.read_kv(child, l)
        ref = es.K[l][src]
        assert not (np.abs(ke[src] - ref) > key_tolerance(ref, f.dtype, n_rot_e)).any()
        check_key_step(k[dst], ke[src], src, dst, oc.freq, f.dtype, "prefix fork")


@pytest.mark.parametrize("dtype,D,G,S", [("bf16", 64, 4, 16), ("bf16", 128, 8, 16),
                                         ("fp32", 64, 2, 4), ("bf16", 128, 4, 1)])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_prefix_fork_matches_oracle(dtype, D, G, S, seed):
    rng = np.random.default_rng(seed * 31 + D + S)
    f = Family(dtype, D, G, S, seed=seed)
    trunk, n = _trunk(rng, int(rng.integers(4, 12)))
    ids = list(int(x) for x in rng.integers(0, 30000, size=n + 400))
    kinds = []
    for _ in range(6):
        cut = int(rng.integers(1, len(trunk) + 1))
        base = trunk[:cut]
        nb = sum(op[1] for op in base if op[0] == "append")
        prog, m = _branch(rng, base, nb)
        f.publish(prog, ids[:m])
    for r in range(4):
        cut = int(rng.integers(1, len(trunk) + 1))
        base = trunk[:cut]
        nb = sum(op[1] for op in base if op[0] == "append")
        prog, m = _branch(rng, base, nb)
        req = P.records(prog, ids[:m])
        want = P.match(f.entries, req, S)
        _poison_free_pages(f)
        child, got = f.gpu.prefix_fork(f.idx, prog, ids[:m])
        assert {k: got[k] for k in want} == want, (got, want)
        kinds.append(got["kind"])
        if got["kind"] == "none":
            assert child == -1
            continue
        f.clock += 1
        f.use[got["entry"]] = f.clock
        _check_child(f, child, req, got, f.entries[got["entry"]])
        # the rest of the request on the child, then decode against the oracle
        f.run(child, _remaining(prog, got), ids[:m], t0=got["n_tokens"])
        oc, osid = f.oracle(req)
        assert f.gpu.info(child)["n_logical"] == oc.seqs[osid].n_logical
        q = np.stack([synth.query(f.seed, 900 + r, l, 0, f.hq, f.D, f.width)
                      for l in range(f.L)])
        for l in range(f.L):
            out = f.gpu.decode_attention(l, torch.from_numpy(q[l][None]).to(f.tdtype).cuda(), [child])
            want_o = oc.attention(l, q[l][None], [osid])
            err = np.abs(out.double().cpu().numpy() - want_o)
            tmax, tmean = ATTN_TOL[dtype]
            assert err.max() <= tmax and err.mean() <= tmean, (l, err.max())
        # the history key equals that of the same program built from scratch
        s2 = f.gpu.seq_create()
        f.run(s2, prog, ids[:m])
        assert f.gpu.history_key(child) == f.gpu.history_key(s2)
        f.gpu.seq_free(s2)
        f.gpu.seq_free(child)
    assert f.gpu.sync_errors() == 0
    # eviction: the library's order is the oracle's; everything comes back
    assert f.idx.evict_order() == P.evict_order(f.entries, f.use)
    freed, n_ev = f.gpu.prefix_evict(f.idx, 1 << 30)
    assert n_ev == len(f.entries)
    assert f.gpu.pool_stats()[1] == 0 and freed > 0


def test_publish_and_fork_rules():
    f = Family("bf16", 64, 4, 16)
    ids = list(range(100, 160))
    prog = [("append", 40), ("drop", [(5, 20)]), ("append", 10)]
    e = f.publish(prog, ids[:50])
    # publishing the same history again returns the same entry
    assert f.publish(prog, ids[:50]) == e
    # snapshots are frozen
    k = torch.zeros((f.L, 1, f.hkv, f.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(abi.AkvError) as ex:
        f.gpu.append([e], [1], k, k, [1])
    assert ex.value.code == abi.AKV_EINVAL
    with pytest.raises(abi.AkvError):
        f.gpu.drop(e, [(0, 1)])
    with pytest.raises(abi.AkvError):
        f.gpu.reposition([e])
    # a program that is not the sequence's history is refused
    s = f.gpu.seq_create()
    f.run(s, prog, ids[:50])
    with pytest.raises(abi.AkvError) as ex:
        f.gpu.prefix_publish(f.idx, s, prog, ids[1:51])
    assert ex.value.code == abi.AKV_EINVAL
    # ... and so is a sequence built without token ids
    s2 = f.gpu.seq_create()
    kk, vv = f.kv(0, 5)
    dev = lambda x: torch.from_numpy(x).to(torch.bfloat16).cuda().contiguous()
    f.gpu.append([s2], [5], dev(kk), dev(vv))
    with pytest.raises(abi.AkvError):
        f.gpu.prefix_publish(f.idx, s2, [("append", 5)], ids[:5])
    # the exact prefix shares every page that keeps its slots
    child, m = f.gpu.prefix_fork(f.idx, prog + [("append", 5)], ids[:55])
    assert m["kind"] == "exact" and m["n_tokens"] == 50 and m["op_index"] == 3
    pc, _ = f.gpu.page_table(child)
    pe, _ = f.gpu.page_table(e)
    np.testing.assert_array_equal(pc[pc >= 0], pe[pc >= 0])
    assert f.gpu.kernel_launches() >= 0
    for x in (s, s2, child):
        f.gpu.seq_free(x)
    # eviction of the entry leaves the pool empty
    f.gpu.prefix_evict(f.idx, 1 << 30)
    assert f.gpu.pool_stats()[1] == 0
    assert f.gpu.sync_errors() == 0


def test_drop_aware_eviction_frees_dropped_turn_first():
    """A turn published before a drop is evicted before the newer turn (even
    though used more recently), and evicting it leaves the newer turn's
    pages and any child's bytes untouched."""
    f = Family("bf16", 128, 4, 16)
    ids = list(range(1000, 1400))
    turn1 = [("append", 200)]
    turn2 = [("append", 200), ("drop", [(20, 150)]), ("repos",), ("append", 40)]
    e1 = f.publish(turn1, ids[:200])
    e2 = f.publish(turn2, ids[:240])
    f.gpu.prefix_fork(f.idx, [("append", 100)], ids[:100])   # touches e1 (now the newest use)
    child, m = f.gpu.prefix_fork(f.idx, turn2 + [("append", 3)], ids[:243])
    assert m["entry"] == e2 and m["kind"] == "exact"
    assert f.idx.evict_order() == [e1, e2]
    before = [f.gpu.read_kv(child, l) for l in range(f.L)]
    freed, n = f.gpu.prefix_evict(f.idx, 1)
    assert n == 1 and freed > 0
    assert f.idx.evict_order() == [e2]
    after = [f.gpu.read_kv(child, l) for l in range(f.L)]
    for (k0, v0), (k1, v1) in zip(before, after):
        np.testing.assert_array_equal(k0, k1)
        np.testing.assert_array_equal(v0, v1)
    assert f.gpu.sync_errors() == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_retrigger_fork_rotates_keys(dtype):
    """Entry: 60 tokens, drop [10, 30), reposition, 8 more.  Request: the same
    60 tokens and drop, then 5 tokens without the reposition.  The drop's
    survivors 30..59 are stored at 10..39 and wanted at 30..59: a retrigger
    match of 61 records rotating 30 keys by +20 (the exact prefix is only
    tokens 0..9, since 10..29 are gone from the entry)."""
    f = Family(dtype, 128, 4, 16)
    ids = list(range(500, 600))
    entry = [("append", 60), ("drop", [(10, 30)]), ("repos",), ("append", 8)]
    req = [("append", 60), ("drop", [(10, 30)]), ("append", 5)]
    e = f.publish(entry, ids[:68])
    _poison_free_pages(f)
    child, m = f.gpu.prefix_fork(f.idx, req, ids[:65])
    assert m == dict(kind="retrigger", entry=e, n_records=61, n_tokens=60, n_rotated=30,
                     op_index=2, op_tokens=0)
    recs = P.records(req, ids[:65])
    _check_child(f, child, recs, m, f.entries[e])
    pages, _ = f.gpu.page_table(child)
    pe, _ = f.gpu.page_table(e)
    assert pages[0] == pe[0]                 # slots 0..9 keep their place: shared
    assert f.gpu.info(child)["next_pos"] == 60
    f.run(child, [("append", 5)], ids[:65], t0=60)
    oc, osid = f.oracle(recs)
    for l in range(f.L):
        q = synth.query(f.seed, 77, l, 0, f.hq, f.D, f.width)[None]
        out = f.gpu.decode_attention(l, torch.from_numpy(q).to(f.tdtype).cuda(), [child])
        err = np.abs(out.double().cpu().numpy() - oc.attention(l, q, [osid]))
        tmax, tmean = ATTN_TOL[dtype]
        assert err.max() <= tmax and err.mean() <= tmean
    assert f.gpu.sync_errors() == 0


def test_shared_decode_over_held_unwritten_slots():
    """A prefix fork whose tail page holds no needed token gets a fresh page
    whose held rows are never written (here NaN patterns: free pages were
    poisoned); appends then fill the page, and forks of that sequence hold it
    as a full page.  The tensor-core shared decode over those forks must mask
    the unwritten rows in the scores and the values alike."""
    f = Family("bf16", 128, 4, 16)
    ids = list(range(1000, 1200))
    entry = [("append", 120), ("drop", [(112, 120)])]
    f.publish(entry, ids[:120])
    _poison_free_pages(f)
    req = entry + [("append", 8)]
    child, m = f.gpu.prefix_fork(f.idx, req, ids[:128])
    assert m["kind"] == "exact" and m["n_tokens"] == 120, m
    f.run(child, _remaining(req, m), ids[:128], t0=120)
    assert f.gpu.info(child)["n_held"] == 128
    pages, _ = f.gpu.page_table(child)
    # the held, dropped slots 112..119 of the last page were never written
    assert torch.isnan(f.gpu.v_pool[:, int(pages[7]), :, :8].float()).any()
    kids = [f.gpu.seq_fork(child) for _ in range(3)]
    oc, osid = f.oracle(P.records(req, ids[:128]))
    for mode in (1, 2, 0):
        f.gpu.set_decode_sharing(mode)
        for l in range(f.L):
            q = np.stack([synth.query(f.seed, 700 + i, l, 0, f.hq, f.D, f.width)
                          for i in range(len(kids))])
            out = f.gpu.decode_attention(l, torch.from_numpy(q).to(f.tdtype).cuda(), kids)
            got = out.double().cpu().numpy()
            assert np.isfinite(got).all(), (mode, l)
            err = np.abs(got - oc.attention(l, q, [osid] * len(kids)))
            tmax, tmean = ATTN_TOL["bf16"]
            assert err.max() <= tmax and err.mean() <= tmean, (mode, l, err.max())
            if mode:
                assert f.gpu.decode_plan_stats()["shared_items"] > 0
    assert f.gpu.sync_errors() == 0
