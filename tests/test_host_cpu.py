"""The cache's host planner on a machine without a GPU.

The planner (``akv_host.cpp``, ``akv_prefix.cpp``) is built with g++ against
a host-memory stand-in for the CUDA runtime (``tests/host/fake_cuda.cpp``):
no kernel runs, so only state the planner keeps on the host is checked --
sequence counts (held slots, next position, pages, active pages, active
tokens), the logical index of every held slot, the planner's page table,
page reference counts and pool occupancy, history keys, and that a call
that fails leaves all of it unchanged.

References:
* counts, logical maps and history-key equality: the oracle
  (``oracle.akv_oracle.OracleCache`` without K/V), replayed alongside;
* page rules of the design (page 1, 3.2 / 4.2.3: forks share pages
  copy-on-write; a reposition keeps the pages before the first page holding
  a dropped slot and writes the rest to fresh pages; a drop releases full
  pages left without an active token; an append into a shared, partly
  filled tail page copies it first);
* reference counts: every held page counted once per sequence holding it,
  and nothing left after every sequence is freed.
"""
import ctypes
import os
import sys

import numpy as np
import pytest

from agent_kv_cache_gb300 import abi
from oracle.akv_oracle import OracleCache

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "host"))
import build_host  # noqa: E402


@pytest.fixture(scope="module")
def host_lib():
    """Point the binding at the host-only build for this module."""
    l = ctypes.CDLL(build_host.build())
    for name, (res, args) in abi.SIGNATURES.items():
        fn = getattr(l, name, None)
        if fn is not None:
            fn.restype, fn.argtypes = res, args
    saved = abi._lib
    abi._lib = l
    yield l
    abi._lib = saved


class HostCache:
    """A cache of the host-only build plus the oracle's metadata replay."""

    def __init__(self, S=16, max_pages=256, max_seqs=8, max_slots=2048, hq=4, hkv=2, D=64):
        self.S, self.hkv, self.D = S, hkv, D
        self.cfg = abi.make_config(1, hq, hkv, D, S, "fp32", max_pages, max_seqs, max_slots, 1e4)
        nbytes = abi.akv_pool_bytes(self.cfg)
        # pools: aligned host memory (the stand-in never runs a kernel on them)
        self._mem = [np.zeros(nbytes + 256, np.uint8) for _ in range(2)]
        ptr = [m.ctypes.data + (-m.ctypes.data % 256) for m in self._mem]
        self.h = abi.akv_cache_create(self.cfg, ptr[0], ptr[1], nbytes)
        self.orc = OracleCache(hq, hkv, D, 1e4, "fp32", layers=[], page_size=S)
        self.o = {}
        self.raw = np.zeros(16, np.float32)        # never read: no kernel runs
        self.max_pages = max_pages

    def close(self):
        abi.akv_cache_destroy(self.h)

    def create(self):
        s = abi.akv_seq_create(self.h)
        self.o[s] = self.orc.create()
        return s

    def fork(self, p):
        s = abi.akv_seq_fork(self.h, p)
        self.o[s] = self.orc.fork(self.o[p])
        return s

    def free(self, s):
        abi.akv_seq_free(self.h, s)
        self.orc.free(self.o.pop(s))

    def append(self, seqs, ns):
        abi.akv_append(self.h, seqs, ns, self.raw.ctypes.data, self.raw.ctypes.data)
        for s, n in zip(seqs, ns):
            self.orc.append(self.o[s], np.zeros((0, n, self.hkv, self.D)),
                            np.zeros((0, n, self.hkv, self.D)))

    def drop(self, s, ranges):
        abi.akv_drop(self.h, s, ranges)
        self.orc.drop(self.o[s], ranges)

    def reposition(self, seqs):
        abi.akv_reposition(self.h, seqs)
        for s in seqs:
            self.orc.reposition(self.o[s])

    def pages(self, s):
        return abi.akv_seq_host_pages(self.h, s)

    def refcounts(self):
        return np.array([abi.akv_page_refcount(self.h, p) for p in range(self.max_pages)])

    def snapshot(self):
        """Everything a failed call must leave unchanged."""
        return {s: (abi.akv_seq_info(self.h, s), self.pages(s).tolist(),
                    abi.akv_history_key(self.h, s)) for s in self.o}, \
            self.refcounts().tolist(), abi.akv_pool_stats(self.h)

    def check(self):
        """Every live sequence against the oracle and the page rules; the
        reference counts against the page tables."""
        S = self.S
        held_total = np.zeros(self.max_pages, np.int64)
        for s, os_ in self.o.items():
            info = abi.akv_seq_info(self.h, s)
            want = self.orc.info(os_)
            for k in ("n_logical", "n_held", "next_pos", "n_pages", "n_active_pages"):
                assert info[k] == want[k], (s, k, info[k], want[k])
            assert info["n_active"] == want["n_alive"]
            st = self.orc.seqs[os_]
            np.testing.assert_array_equal(abi.akv_seq_logical(self.h, s, info["n_held"]),
                                          st.logical)
            np.testing.assert_array_equal(abi.akv_seq_positions(self.h, s, info["n_held"]),
                                          np.arange(info["n_held"]))
            pages = self.pages(s)
            assert len(pages) == want["n_pages"]
            act = set(self.orc.active_pages(os_).tolist())
            n = info["n_held"]
            for k, p in enumerate(pages):
                tail = k == len(pages) - 1 and n % S != 0
                # a page is held iff it has an active token or is the partly
                # filled tail page (appends write into it)
                assert (p >= 0) == (k in act or tail), (s, k, p, sorted(act), n)
                if p >= 0:
                    assert 0 <= p < self.max_pages
                    held_total[p] += 1
            assert info["n_owned_pages"] + info["n_shared_pages"] == int((pages >= 0).sum())
        rc = self.refcounts()
        np.testing.assert_array_equal(rc, held_total)
        free, used = abi.akv_pool_stats(self.h)
        assert used == int((rc > 0).sum()) and free + used == self.max_pages
        # equal histories <=> equal keys
        ids = list(self.o)
        for i, a in enumerate(ids):
            for b in ids[i + 1:]:
                same_log = self.orc.history(self.o[a]) == self.orc.history(self.o[b])
                assert same_log == (abi.akv_history_key(self.h, a) == abi.akv_history_key(self.h, b))


def _random_program(c, rng, n_ops, max_tokens=512):
    seqs = [c.create()]
    c.append(seqs, [int(rng.integers(1, 80))])
    for _ in range(n_ops):
        u = rng.random()
        s = seqs[int(rng.integers(0, len(seqs)))]
        n_log = c.orc.seqs[c.o[s]].n_logical
        if u < 0.3 and n_log < max_tokens:
            k = int(rng.integers(1, min(120, max_tokens - n_log) + 1))
            targets = [x for x in seqs if c.orc.seqs[c.o[x]].n_logical + k <= max_tokens]
            pick = [x for x in targets if rng.random() < 0.6] or [s]
            pick = [x for x in pick if c.orc.seqs[c.o[x]].n_logical + k <= max_tokens]
            if pick:
                c.append(pick, [k] * len(pick))
        elif u < 0.55 and n_log:
            ranges = []
            for _ in range(int(rng.integers(1, 4))):
                b = int(rng.integers(0, n_log))
                ranges.append((b, int(min(n_log, b + rng.integers(1, 60)))))
            c.drop(s, ranges)
        elif u < 0.75:
            pick = [x for x in seqs if rng.random() < 0.5] or [s]
            c.reposition(pick)
        elif u < 0.9 and len(seqs) < 6:
            seqs.append(c.fork(s))
        elif len(seqs) > 1:
            seqs.remove(s)
            c.free(s)
        c.check()
    return seqs


@pytest.mark.parametrize("S", [16, 1, 4])
@pytest.mark.parametrize("seed", range(8))
def test_random_programs_against_oracle(host_lib, S, seed):
    """Random append / fork / drop / reposition / free programs (at most 512
    tokens per sequence): counts, logical maps, page rules, reference counts
    and history keys after every operation; the pool is empty at the end."""
    rng = np.random.default_rng(1000 * S + seed)
    c = HostCache(S=S, max_pages=4096 if S == 1 else 1024, max_slots=600)
    seqs = _random_program(c, rng, 40)
    for s in seqs:
        c.free(s)
    c.check()
    assert abi.akv_pool_stats(c.h)[1] == 0
    c.close()


def test_copy_on_write_decisions(host_lib):
    """Fork shares every page; an append into the shared partly filled tail
    copies that page only; a reposition keeps the pages before the first page
    holding a dropped slot and takes fresh pages for the rest."""
    c = HostCache(S=16)
    a = c.create()
    c.append([a], [100])                      # pages 0..6, tail page 6 holds 4 slots
    pa = c.pages(a)
    b = c.fork(a)
    np.testing.assert_array_equal(c.pages(b), pa)
    assert all(abi.akv_page_refcount(c.h, int(p)) == 2 for p in pa)
    c.append([b], [3])                        # writes into the shared tail page
    pb = c.pages(b)
    np.testing.assert_array_equal(pb[:6], pa[:6])
    assert pb[6] != pa[6] and abi.akv_page_refcount(c.h, int(pb[6])) == 1
    assert abi.akv_page_refcount(c.h, int(pa[6])) == 1
    c.check()
    c.drop(b, [(40, 45)])                     # first dropped slot 40: page 2
    c.reposition([b])
    pr = c.pages(b)
    np.testing.assert_array_equal(pr[:2], pa[:2])          # kept, still shared
    assert all(abi.akv_page_refcount(c.h, int(p)) == 2 for p in pr[:2])
    for p in pr[2:]:
        assert p not in set(pa.tolist()) and abi.akv_page_refcount(c.h, int(p)) == 1
    c.check()
    # a reposition with nothing dropped since the last one is an exact no-op
    before = c.snapshot()
    n0 = host_lib.akv_fake_launches()
    c.reposition([b])
    after = c.snapshot()
    assert before[0][b][:2] == after[0][b][:2] and before[1:] == after[1:]
    assert host_lib.akv_fake_launches() == n0
    c.free(a)
    c.free(b)
    assert abi.akv_pool_stats(c.h)[1] == 0
    c.close()


def test_drop_releases_pages_without_active_tokens(host_lib):
    c = HostCache(S=16)
    a = c.create()
    c.append([a], [70])                       # pages 0..4 (4 partly filled)
    c.drop(a, [(16, 48)])                     # pages 1, 2 left without an active token
    p = c.pages(a)
    assert p[1] == -1 and p[2] == -1 and p[0] >= 0 and p[3] >= 0
    c.drop(a, [(64, 70)])                     # the partly filled tail stays held
    assert c.pages(a)[4] >= 0
    c.check()
    assert abi.akv_pool_stats(c.h)[1] == 3
    c.free(a)
    assert abi.akv_pool_stats(c.h)[1] == 0
    c.close()


def _expect_error(code, fn, *args):
    with pytest.raises(abi.AkvError) as e:
        fn(*args)
    assert e.value.code == code, (e.value.code, code)


def test_out_of_pages_rolls_back(host_lib):
    """A call that needs more pages than are free fails with AKV_ENOPAGES and
    leaves every sequence, page table, reference count and the pool as they
    were -- also in a batched call where only a later sequence runs out."""
    c = HostCache(S=16, max_pages=12)
    a = c.create()
    c.append([a], [100])                      # 7 pages
    b = c.fork(a)
    c.check()
    snap = c.snapshot()
    # appending 100 more tokens to both needs 14 pages (5 free)
    _expect_error(abi.AKV_ENOPAGES, abi.akv_append, c.h, [a, b], [100, 100],
                  c.raw.ctypes.data, c.raw.ctypes.data)
    assert c.snapshot() == snap
    # a reposition of b after an early drop needs 6 fresh pages (5 free)
    c.drop(b, [(3, 4)])
    snap = c.snapshot()
    _expect_error(abi.AKV_ENOPAGES, abi.akv_reposition, c.h, [b])
    assert c.snapshot() == snap
    # batched: a's reposition fits alone, b's does not; nothing happens
    c.drop(a, [(90, 95)])
    snap = c.snapshot()
    _expect_error(abi.AKV_ENOPAGES, abi.akv_reposition, c.h, [a, b])
    assert c.snapshot() == snap
    c.check()                                 # the drops stand, the repositions never ran
    c.free(a)
    c.free(b)
    assert abi.akv_pool_stats(c.h)[1] == 0
    c.close()


def test_errors_leave_state_unchanged(host_lib):
    c = HostCache(S=16, max_seqs=3, max_slots=200)
    a = c.create()
    c.append([a], [50])
    snap = c.snapshot()
    _expect_error(abi.AKV_ERANGE, abi.akv_drop, c.h, a, [(10, 51)])          # past the end
    _expect_error(abi.AKV_ERANGE, abi.akv_drop, c.h, a, [(-1, 3)])
    _expect_error(abi.AKV_ENOSEQ, abi.akv_drop, c.h, 12345, [(0, 1)])
    _expect_error(abi.AKV_ECAPACITY, abi.akv_append, c.h, [a], [151],        # > max_slots
                  c.raw.ctypes.data, c.raw.ctypes.data)
    assert c.snapshot() == snap
    b = c.fork(a)
    c.free(b)
    _expect_error(abi.AKV_ENOSEQ, abi.akv_seq_fork, c.h, b)                  # forking a freed seq
    _expect_error(abi.AKV_ENOSEQ, abi.akv_append, c.h, [b], [1],             # use after free
                  c.raw.ctypes.data, c.raw.ctypes.data)
    _expect_error(abi.AKV_ENOSEQ, abi.akv_reposition, c.h, [a, b])
    _expect_error(abi.AKV_ENOSEQ, abi.akv_seq_free, c.h, b)
    assert c.snapshot() == snap
    s2, s3 = c.fork(a), c.create()
    _expect_error(abi.AKV_ECAPACITY, abi.akv_seq_create, c.h)                 # max_seqs
    assert abi.akv_pool_stats(c.h) == snap[2]
    for s in (s2, s3):
        c.free(s)
    c.check()
    c.free(a)
    assert abi.akv_pool_stats(c.h)[1] == 0
    c.close()


def test_interval_sets_under_overlapping_drops(host_lib):
    """Overlapping, repeated and out-of-order drop ranges (set semantics),
    across repositions that renumber slots (ranges stay logical)."""
    rng = np.random.default_rng(5)
    c = HostCache(S=4, max_pages=2048, max_slots=1500)
    a = c.create()
    c.append([a], [400])
    for r in range(30):
        n = c.orc.seqs[c.o[a]].n_logical
        ranges = [(int(b), int(min(n, b + rng.integers(1, 30))))
                  for b in rng.integers(0, n, size=int(rng.integers(1, 6)))]
        c.drop(a, ranges[::-1])
        c.drop(a, ranges[:1])                 # again: nothing changes but the history
        if r % 4 == 3:
            c.reposition([a])
        if r % 5 == 4:
            c.append([a], [int(rng.integers(1, 40))])
        c.check()
    c.free(a)
    c.close()


@pytest.fixture()
def tensor_core_plans(host_lib):
    """Plan as for a GPU where the tensor-core decode kernels run."""
    host_lib.akv_fake_set_tensor_cores(1)
    yield host_lib
    host_lib.akv_fake_set_tensor_cores(0)


def test_shared_prefix_items_fit_one_wave(tensor_core_plans):
    """Branches of one prefix, each with its own drops and repositions: the
    decode plan reads pages that several branches hold through shared-prefix
    items (page 1, 3.2: forks share pages copy-on-write), and those items fit
    one wave of the shared-prefix kernel (two CTAs per SM on the 152 SMs the
    stand-in reports, one CTA per KV head), whatever the segments' sizes."""
    from workloads import traces
    sh = traces.LLAMA8B
    NB, P = 48, 8192
    _, branches = traces.branching(11, n_branches=NB, prefix_len=P)
    cfg = abi.make_config(1, sh.hq, sh.hkv, sh.head_dim, 16, "bf16", P // 16 + NB * 700 + 256,
                          NB + 2, P + 64, sh.rope_theta)
    nbytes = abi.akv_pool_bytes(cfg)
    mem = [np.zeros(nbytes + 256, np.uint8) for _ in range(2)]
    ptr = [m.ctypes.data + (-m.ctypes.data % 256) for m in mem]
    h = abi.akv_cache_create(cfg, ptr[0], ptr[1], nbytes)
    raw = np.zeros(16, np.float32)
    root = abi.akv_seq_create(h)
    abi.akv_append(h, [root], [P], raw.ctypes.data, raw.ctypes.data)
    kids = [abi.akv_seq_fork(h, root) for _ in range(NB)]
    for i in range(max(len(b.ops) for b in branches)):
        rep = []
        for k, br in zip(kids, branches):
            if i < len(br.ops):
                if br.ops[i][0] == "drop":
                    abi.akv_drop(h, k, br.ops[i][1])
                else:
                    rep.append(k)
        if rep:
            abi.akv_reposition(h, rep)
    abi.akv_append(h, kids, [1] * NB, raw.ctypes.data, raw.ctypes.data)
    q = np.zeros(NB * sh.hq * sh.head_dim, np.uint16)
    out = np.zeros(NB * sh.hq * sh.head_dim, np.float32)
    abi.akv_decode_attention(h, 0, q.ctypes.data, kids, out.ctypes.data)
    st = abi.akv_decode_plan_stats(h)
    assert st["shared_items"] > 0
    assert st["shared_items"] * sh.hkv <= 2 * 152
    # every branch is merged by one item of the one-row kernel at least
    assert st["items"] - st["shared_items"] >= NB
    assert st["members"] >= 2 * st["shared_items"]
    for k in kids:
        abi.akv_seq_free(h, k)
    abi.akv_seq_free(h, root)
    assert abi.akv_pool_stats(h)[1] == 0
    abi.akv_cache_destroy(h)


def test_restore_token_list_checks(host_lib):
    """akv_restore_attention_tokens checks its token list before any GPU
    work: increasing and within the program's tokens; an empty list does
    nothing (no launch)."""
    c = HostCache(S=16)
    prog = [("append", 5), ("drop", [(1, 2)]), ("repos",), ("append", 3)]
    n = 8
    buf = np.zeros(n * 4 * 64, np.float32)
    p = buf.ctypes.data
    n0 = host_lib.akv_fake_launches()
    abi.akv_restore_attention_tokens(c.h, prog, 0, p, p, p, n, [], p)
    assert host_lib.akv_fake_launches() == n0
    for bad in ([3, 2], [1, 1], [-1], [n]):
        with pytest.raises(abi.AkvError) as e:
            abi.akv_restore_attention_tokens(c.h, prog, 0, p, p, p, n, bad, p)
        assert e.value.code == abi.AKV_EINVAL
    with pytest.raises(abi.AkvError) as e:        # the program appends 8 tokens, not 9
        abi.akv_restore_attention_tokens(c.h, prog, 0, p, p, p, n + 1, [0], p)
    assert e.value.code == abi.AKV_EINVAL
    assert host_lib.akv_fake_launches() == n0
    abi.akv_restore_attention_tokens(c.h, prog, 0, p, p, p, n, [0, 4, 7], p)
    assert host_lib.akv_fake_launches() > n0
    c.close()
