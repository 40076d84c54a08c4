#!/usr/bin/env python3
"""Benchmark of the active-KV hot path: drop + reposition + decode attention.

Headline workload (the largest of the single-GPU workloads): the
Llama-70B-shaped long-running agent steady state -- 80 layers (stored on 16
aliased physical slabs; every logical layer's kernels still run and move
their bytes), 64 query / 8 KV heads, head_dim 128, bf16 K/V, RoPE theta 5e5,
page 16; 64 sequences, each a 1024-token system prompt followed by agent
turns.  A turn appends one tool response (lognormal, median 1000 tokens,
clipped to 200..4000) and decodes 64 tokens (each: append the token's K/V,
decode attention on all 80 layers).  After every third turn the oldest tool
responses are dropped until at most 16384 tokens are active, and the
sequences are repositioned.  One step = one turn of the steady-state window
(turns 31 and later); the state before the warm-up turns is built untimed
by the same calls.  Inputs are seeded and synthetic and resident in HBM when
the timed region starts: the tool-response, query and new-token buffers are
filled once and re-read every turn (each far larger than L2).

The same run adds one block per other workload (each with its own cache,
timed after the headline): the Llama-3.1-8B-shaped trace (16 x 32768 tokens,
~60% dropped, one reposition, 128 decode steps), the GPT-OSS-120B-shaped
trace (4 x 131072 tokens, ~80% dropped, 256 decode steps) and the branching
histories (one 16384-token prefix forked into 64 branches, each applying 1-6
drop / reposition operations, then 128 batched decode steps over all 64).

``value`` is algorithmic bytes per second over the whole step: K/V of the
tool responses and decode tokens read and written by the appends, the active
K/V read by every decode-attention call (plus q, out and page metadata), the
K/V of relocated survivors read and written by the reposition, and the drop's
metadata.  ``--impl reference`` times the CPU oracle on the same workload.
"""
import argparse
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import synth, traces  # noqa: E402

METRIC = "active-KV GB/s & % HBM roofline (drop+repos+decode attn), decode tok/s, 1×GB300"
BYTES_EL = 2
CHUNK = 4096

# the 70B-shaped steady state (headline)
STEADY = traces.LLAMA70B
STEADY_SEQS = 64
STEADY_SLABS = 16
STEADY_DECODE = 64
STEADY_CAP = 16384
STEADY_SYS = 1024
STEADY_FIRST = 30          # index of the first timed turn (turn 31 of 100)
STEADY_TURNS = 100
STEADY_GROUPS = 4          # tool responses appended in batched calls of 16 sequences
STEADY_SEED = traces.seed_for(4)
SHAPE = traces.LLAMA8B     # restore attention and prefix-sharing lines

# the 8B- and 120B-shaped traces and the branching histories (blocks)
TRACE8B = dict(name="llama8b", shape=traces.LLAMA8B, batch=16, n_tokens=32768, decode=128,
               seed=traces.seed_for(1))
TRACE120B = dict(name="gptoss120b", shape=traces.GPTOSS120B, batch=4, n_tokens=131072,
                 decode=256, seed=traces.seed_for(2))
BRANCH = dict(shape=traces.LLAMA8B, prefix=16384, branches=64, decode=128,
              seed=traces.seed_for(3))
# profiler case of the 70B shape (not a block): 8 sequences of 40960 tokens
# with ~60% dropped, about the steady state's ~16K active tokens per sequence
TRACE70B = dict(name="llama70b", shape=traces.LLAMA70B, batch=8, n_tokens=40960, decode=4,
                seed=traces.seed_for(4))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    return json.load(open(p)) if os.path.exists(p) else {}


def hbm_peak():
    pk = load_peaks()
    return (pk["hbm_gbs"], "measured") if "hbm_gbs" in pk else (6800.0, "fallback")


def kvt_of(sh):
    """K + V bytes of one token on one layer."""
    return 2 * sh.hkv * sh.head_dim * BYTES_EL


# ---------------------------------------------------------------------------
# host mirror of a sequence, for algorithmic bytes and pool sizing
# ---------------------------------------------------------------------------

class Sim:
    """Held slots of one sequence (logical index and active flag per slot),
    following the library's rules: slots are positions; a drop releases the
    full pages left without an active token; a reposition keeps the pages
    before the first page that holds a dropped slot and rewrites the
    survivors from there into fresh pages.  ``first_private`` tracks, for a
    forked sequence, the first page it owns alone (pages before it are
    shared with its parent)."""

    def __init__(self, S, logical=None, shared_pages=0):
        self.S = S
        self.logical = np.zeros(0, np.int64) if logical is None else logical.copy()
        self.alive = np.ones(self.logical.size, bool)
        self.n_logical = int(self.logical.size)
        self.first_private = shared_pages

    def append(self, n):
        self.logical = np.concatenate([self.logical, self.n_logical + np.arange(n)])
        self.alive = np.concatenate([self.alive, np.ones(n, bool)])
        self.n_logical += n

    def drop(self, ranges):
        for b, e in ranges:
            self.alive &= ~((self.logical >= b) & (self.logical < e))

    def held(self):
        return int(self.alive.size)

    def active(self):
        return int(self.alive.sum())

    def active_pages(self):
        return int(np.unique(np.flatnonzero(self.alive) // self.S).size)

    def held_pages(self):
        pages = set((np.flatnonzero(self.alive) // self.S).tolist())
        if self.alive.size % self.S:
            pages.add(self.alive.size // self.S)
        return len(pages)

    def private_pages(self):
        pages = set((np.flatnonzero(self.alive) // self.S).tolist())
        if self.alive.size % self.S:
            pages.add(self.alive.size // self.S)
        return sum(1 for p in pages if p >= self.first_private)

    def reposition(self):
        """Returns (survivors relocated, fresh pages taken)."""
        dead = np.flatnonzero(~self.alive)
        if dead.size == 0:
            return 0, 0
        kept = (int(dead[0]) // self.S) * self.S
        r = int(self.alive.sum())
        self.logical = self.logical[self.alive]
        self.alive = np.ones(r, bool)
        self.first_private = min(self.first_private, kept // self.S)
        return r - kept, -(-r // self.S) - kept // self.S


def decode_call_bytes(sh, actives, pages):
    """Algorithmic bytes of one decode-attention call over rows with these
    active-token and active-page counts."""
    n = len(actives)
    return (sum(actives) * kvt_of(sh) + n * sh.hq * sh.head_dim * (BYTES_EL + 4)
            + sum(pages) * (4 + 4 + sh.page_size // 8))


def drop_bytes(sim):
    """Metadata a drop touches: keep bits of the held slots, the page list."""
    return sim.held() // 8 + 10 * (-(-sim.held() // sim.S))


# ---------------------------------------------------------------------------
# the steady-state schedule: per-turn bytes, pool size, buffer sizes
# ---------------------------------------------------------------------------

def steady_schedule(n_turns):
    return traces.steady_state(STEADY_SEED, n_seqs=STEADY_SEQS, n_turns=n_turns,
                               sys_len=STEADY_SYS, decode_per_turn=STEADY_DECODE,
                               active_cap=STEADY_CAP)


def steady_groups():
    g = STEADY_SEQS // STEADY_GROUPS
    return [list(range(i * g, (i + 1) * g)) for i in range(STEADY_GROUPS)]


def steady_plan(turns, seqs, n_turns, timed_from):
    """Walk the schedule of sequences ``seqs`` for turns 0..n_turns-1.
    Turns before ``timed_from`` are replayed in bulk (tool response and the
    decode tokens appended at once); from it on, each turn is accounted as the
    benchmark runs it.  Returns per-turn byte accounts, the pool's peak page
    count and the largest batched append (tokens) of each kind."""
    sh = STEADY
    L, kvt, S = sh.layers, kvt_of(sh), sh.page_size
    sims = {s: Sim(S) for s in seqs}
    for s in seqs:
        sims[s].append(STEADY_SYS)
    peak = sum(sims[s].held_pages() for s in seqs)
    groups = [[s for s in g if s in sims] for g in steady_groups()]
    bulk_max = STEADY_SYS * max(len(g) for g in groups)
    tool_max = 0
    acct = []
    for k in range(n_turns):
        tool = {s: turns[s][k].tool_len for s in seqs}
        a = {"tool": sum(tool.values()), "calls": [], "repos_moved": 0, "drop": 0,
             "repos": False, "dropped": False}
        if k < timed_from:
            for g in groups:
                bulk_max = max(bulk_max, sum(tool[s] + STEADY_DECODE for s in g))
            for s in seqs:
                sims[s].append(tool[s] + STEADY_DECODE)
        else:
            for g in groups:
                tool_max = max(tool_max, sum(tool[s] for s in g))
            for s in seqs:
                sims[s].append(tool[s])
            act = [sims[s].active() for s in seqs]
            pg = [sims[s].active_pages() for s in seqs]
            held = [sims[s].held() for s in seqs]
            for t in range(STEADY_DECODE):
                a_t = [x + t + 1 for x in act]
                p_t = [p + (-(-(h + t + 1) // S)) - (-(-h // S)) for p, h in zip(pg, held)]
                a["calls"].append(decode_call_bytes(sh, a_t, p_t))
            for s in seqs:
                sims[s].append(STEADY_DECODE)
        peak = max(peak, sum(sims[s].held_pages() for s in seqs))
        for s in seqs:
            if turns[s][k].drop_ranges:
                a["drop"] += drop_bytes(sims[s])
                sims[s].drop(turns[s][k].drop_ranges)
                a["dropped"] = True
        if any(turns[s][k].repos for s in seqs):
            a["repos"] = True
            before = sum(sims[s].held_pages() for s in seqs)
            fresh = 0
            for s in seqs:
                if turns[s][k].repos:
                    moved, fr = sims[s].reposition()
                    a["repos_moved"] += moved
                    fresh += fr
            peak = max(peak, before + fresh)
        a["append_bytes"] = 2 * L * (a["tool"] + STEADY_DECODE * len(seqs)) * kvt
        a["decode_bytes"] = L * sum(a["calls"])
        a["repos_bytes"] = 2 * L * a["repos_moved"] * kvt
        a["total"] = a["append_bytes"] + a["decode_bytes"] + a["repos_bytes"] + a["drop"]
        acct.append(a)
    return acct, peak, bulk_max, tool_max


# ---------------------------------------------------------------------------
# CPU oracle leg: worker processes, one per sampled (sequence, layer)
# ---------------------------------------------------------------------------

ORACLE_DECODE = 2        # decode steps the oracle times per turn (of 64)


def _steady_worker(conn, seq, layer, n_turns, start):
    """Oracle state of one (sequence, layer) of the steady-state workload,
    built to turn ``start`` untimed; then, per request, one turn: timed are
    the tool append, the first ORACLE_DECODE decode steps (append + attention)
    and the turn's drop and reposition; the turn's other decode tokens are
    appended untimed (in one call), so the state follows the schedule.
    Input generation is excluded from the time."""
    os.environ["OMP_NUM_THREADS"] = "1"
    from oracle.akv_oracle import OracleCache
    sh = STEADY
    turns = traces.steady_state(STEADY_SEED, n_seqs=seq + 1, n_turns=n_turns, sys_len=STEADY_SYS,
                                decode_per_turn=STEADY_DECODE, active_cap=STEADY_CAP)[seq]
    o = OracleCache(sh.hq, sh.hkv, sh.head_dim, sh.rope_theta, sh.dtype, layers=[layer],
                    page_size=sh.page_size)
    s = o.create()
    w = synth.width_for(sh.dtype)
    tag = seq + 1
    t = [0]

    def kv(n):
        k = synth.kv_tokens(STEADY_SEED, tag, synth.KIND_K, [layer], t[0], n, sh.hkv,
                            sh.head_dim, w)
        v = synth.kv_tokens(STEADY_SEED, tag, synth.KIND_V, [layer], t[0], n, sh.hkv,
                            sh.head_dim, w)
        t[0] += n
        return k, v

    o.append(s, *kv(STEADY_SYS))
    for k in range(start):
        o.append(s, *kv(turns[k].tool_len + STEADY_DECODE))
        if turns[k].drop_ranges:
            o.drop(s, turns[k].drop_ranges)
        if turns[k].repos:
            o.reposition(s)
    conn.send("ready")
    D = ORACLE_DECODE
    while True:
        k = conn.recv()
        if k is None:
            break
        tn = turns[k]
        kt, vt = kv(tn.tool_len)
        kn, vn = kv(STEADY_DECODE)
        qs = [synth.query(STEADY_SEED, tag, layer, k * STEADY_DECODE + i, sh.hq, sh.head_dim, w)
              for i in range(D)]
        t0 = time.perf_counter()
        o.append(s, kt, vt)
        for i in range(D):
            o.append(s, kn[:, i:i + 1], vn[:, i:i + 1])
            o.attention(0, qs[i][None], [s])
        el = time.perf_counter() - t0
        o.append(s, kn[:, D:], vn[:, D:])
        t0 = time.perf_counter()
        if tn.drop_ranges:
            o.drop(s, tn.drop_ranges)
        if tn.repos:
            o.reposition(s)
        conn.send(el + time.perf_counter() - t0)
    conn.close()


class OracleTurns:
    """The oracle on a bounded sample of the steady-state workload: one
    single-threaded process per sampled (sequence, layer), all advancing one
    turn per request; a turn's time is the slowest unit's."""

    def __init__(self, seqs=(0, 1), layers=(0, 1), start=STEADY_FIRST, n_turns=STEADY_TURNS):
        self.seqs, self.layers = list(seqs), list(layers)
        self.n_turns = n_turns
        ctx = mp.get_context("spawn")
        self.procs, self.conns = [], []
        for s in self.seqs:
            for l in self.layers:
                a, b = ctx.Pipe()
                p = ctx.Process(target=_steady_worker, args=(b, s, l, n_turns, start), daemon=True)
                p.start()
                self.procs.append(p)
                self.conns.append(a)
        for c in self.conns:
            assert c.recv() == "ready"
        turns = steady_schedule(n_turns)
        self.acct, _, _, _ = steady_plan(turns, self.seqs, n_turns, start)

    def turn_bytes(self, k):
        """Algorithmic bytes of the sampled work of turn k (same accounting as
        the GPU path, for the sampled sequences and layers)."""
        a, kvt, n = self.acct[k], kvt_of(STEADY), len(self.seqs)
        per_layer = (2 * a["tool"] * kvt + sum(a["calls"][:ORACLE_DECODE])
                     + ORACLE_DECODE * 2 * n * kvt + 2 * a["repos_moved"] * kvt + a["drop"])
        return per_layer * len(self.layers)

    def turn(self, k):
        for c in self.conns:
            c.send(k)
        secs = max(c.recv() for c in self.conns)
        return self.turn_bytes(k), secs

    def close(self):
        for c in self.conns:
            c.send(None)
        for p in self.procs:
            p.join(timeout=30)

    def sample(self):
        return (f"{len(self.seqs)} sequences x {len(self.layers)} layers of the workload; per "
                f"turn the tool append, the first {ORACLE_DECODE} of its {STEADY_DECODE} decode "
                "steps (append + attention) and the turn's drop and reposition (the other decode "
                "tokens appended untimed); one single-threaded process per (sequence, layer), "
                "input generation excluded; bytes counted as on the GPU for that work")


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu_id)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id(local):
    import torch
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        return uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        return local


# ---------------------------------------------------------------------------
# ranks: one replica per GPU, sequences partitioned, no data-path collective
# ---------------------------------------------------------------------------

def rank_tags(rank, batch):
    """Input-stream tags of the sequences a rank owns (disjoint across ranks)."""
    return [rank * 1000 + b + 1 for b in range(batch)]


def reduce_max(value, dist, device):
    """Max over ranks of a per-rank time (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def events(torch, n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def isolated_decode(torch, cache, layers, q, seqs, out, reps=3):
    """Decode-attention calls one at a time, each after an unrelated kernel
    that streams a buffer larger than L2 (a stand-in for the projections and
    MLP between two layers' attention): returns the mean per-call time (us)."""
    st = cache.stream
    junk = torch.empty(3 << 27, dtype=torch.float32, device="cuda")     # 1.5 GB
    ev = events(torch, reps * len(layers))
    i = 0
    with torch.cuda.stream(st):
        for _ in range(reps):
            for l in layers:
                junk.mul_(1.0)
                ev[i][0].record(st)
                cache.decode_attention(l, q[l], seqs, out[l])
                ev[i][1].record(st)
                i += 1
    torch.cuda.synchronize()
    del junk
    return float(np.mean([a.elapsed_time(b) for a, b in ev])) * 1e3


# ---------------------------------------------------------------------------
# the steady-state workload on the GPU (headline)
# ---------------------------------------------------------------------------

class Steady:
    """64 sequences of the 70B-shaped steady state, one turn per step."""

    def __init__(self, rank, warmup, steps, e2e_steps):
        import torch
        from agent_kv_cache_gb300 import Cache, build
        from workloads import device as dev
        self.torch, self.dev = torch, dev
        build()
        dev.build()
        sh = self.sh = STEADY
        self.W = min(warmup, STEADY_FIRST)
        self.first = STEADY_FIRST - self.W          # first turn run as a full turn
        self.n_turns = max(STEADY_TURNS, STEADY_FIRST + steps + e2e_steps)
        self.turns = steady_schedule(self.n_turns)
        self.acct, peak, bulk_max, tool_max = steady_plan(
            self.turns, list(range(STEADY_SEQS)), self.n_turns, self.first)
        S, L, H, D, Hq = sh.page_size, sh.layers, sh.hkv, sh.head_dim, sh.hq
        self.max_pages = peak + 4 * STEADY_SEQS + 256
        held_max = STEADY_CAP + 3 * (4000 + STEADY_DECODE) + STEADY_SYS
        self.cache = Cache(L, Hq, H, D, S, sh.dtype, self.max_pages, STEADY_SEQS + 2,
                           held_max, sh.rope_theta, phys_layers=STEADY_SLABS)
        self.stream = self.cache.stream
        self.tags = rank_tags(rank, STEADY_SEQS)
        self.width = synth.width_for(sh.dtype)
        seed = STEADY_SEED + 7919 * rank
        # tool-response K/V (re-read every turn; sized for the largest batched
        # append), the decode steps' queries and new-token K/V
        self.raw_tokens = max(bulk_max, tool_max)
        self.tool_max = tool_max
        n_raw = L * self.raw_tokens * H * D
        self.kraw = torch.empty(n_raw, dtype=torch.bfloat16, device="cuda")
        self.vraw = torch.empty(n_raw, dtype=torch.bfloat16, device="cuda")
        self.q = torch.empty((STEADY_DECODE, L, STEADY_SEQS, Hq, D), dtype=torch.bfloat16,
                             device="cuda")
        self.knew = torch.empty((STEADY_DECODE, L, STEADY_SEQS, H, D), dtype=torch.bfloat16,
                                device="cuda")
        self.vnew = torch.empty_like(self.knew)
        keep = [dev.fill(x, [(synth.stream_key(seed, 1, kind, j), 0, 0)], x.numel(), self.width)
                for j, (x, kind) in enumerate(((self.kraw, synth.KIND_K), (self.vraw, synth.KIND_V),
                                               (self.q, synth.KIND_Q), (self.knew, synth.KIND_K),
                                               (self.vnew, synth.KIND_V)))]
        self.out = torch.empty((L, STEADY_SEQS, Hq, D), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        del keep
        self.groups = steady_groups()
        self._build()

    def raw(self, n, buf=None):
        """[L][n][hkv][D] views of the raw tool-response buffers."""
        sh = self.sh
        kb, vb = buf if buf is not None else (self.kraw, self.vraw)
        m = sh.layers * n * sh.hkv * sh.head_dim
        shape = (sh.layers, n, sh.hkv, sh.head_dim)
        return kb[:m].view(shape), vb[:m].view(shape)

    def _build(self):
        """Sequences at the start of turn ``first``: the system prompt, then
        every earlier turn's tool response and decode tokens appended at once,
        with the turn's drops and reposition."""
        c, torch = self.cache, self.torch
        self.seqs = [c.seq_create() for _ in range(STEADY_SEQS)]
        for g in self.groups:
            k, v = self.raw(STEADY_SYS * len(g))
            c.append([self.seqs[i] for i in g], [STEADY_SYS] * len(g), k, v)
        for k in range(self.first):
            for g in self.groups:
                lens = [self.turns[i][k].tool_len + STEADY_DECODE for i in g]
                kk, vv = self.raw(sum(lens))
                c.append([self.seqs[i] for i in g], lens, kk, vv)
            self._drop_repos(k)
        torch.cuda.synchronize()
        assert c.sync_errors() == 0

    def _drop_repos(self, k, ev=None):
        c = self.cache
        if ev is not None:
            ev["drop"][0].record(self.stream)
        for i, s in enumerate(self.seqs):
            if self.turns[i][k].drop_ranges:
                c.drop(s, self.turns[i][k].drop_ranges)
        if ev is not None:
            ev["drop"][1].record(self.stream)
            ev["repos"][0].record(self.stream)
        rep = [s for i, s in enumerate(self.seqs) if self.turns[i][k].repos]
        if rep:
            c.reposition(rep)
        if ev is not None:
            ev["repos"][1].record(self.stream)

    def events(self):
        E = lambda: events(self.torch, 1)[0]
        return {"append": E(), "dec": events(self.torch, STEADY_DECODE), "drop": E(), "repos": E()}

    def turn(self, k, ev=None, host=None):
        """One turn.  ``ev``: events per phase; ``host``: pinned host inputs
        and outputs (end-to-end variant: each turn's tool responses go up
        during the previous turn's decode, into one device slot per group of
        sequences; each turn's queries and new-token K/V go up while its own
        decode steps run, each step waiting for its own)."""
        c, torch, st = self.cache, self.torch, self.stream
        L = self.sh.layers
        if host is not None:
            if not hasattr(self, "_h2d"):
                self._h2d = torch.cuda.Stream()            # this turn's queries / new K/V
                self._h2d_tool = torch.cuda.Stream()       # the next turn's tool responses
                self._d2h = torch.cuda.Stream()
                self._tool_ready = [torch.cuda.Event() for _ in self.groups]
                self._ready = [torch.cuda.Event() for _ in range(STEADY_DECODE)]
                self._done = [torch.cuda.Event() for _ in range(STEADY_DECODE)]
                self._prefetched = None
                self._tool_ev, self._tool_host_s = {}, {}
            if self._prefetched != k:          # nothing prefetched: copy now
                self._h2d_tool.wait_stream(st)
                self._tool_copy(k, host)
            st.wait_stream(self._d2h)          # the previous turn's outputs have been read
        if ev is not None:
            ev["append"][0].record(st)
        for gi, g in enumerate(self.groups):
            lens = [self.turns[i][k].tool_len for i in g]
            n = sum(lens)
            if host is None:
                kk, vv = self.raw(n)
            else:
                kk, vv = self.raw(n, host["slots"][gi])
                st.wait_event(self._tool_ready[gi])
            c.append([self.seqs[i] for i in g], lens, kk, vv)
        if ev is not None:
            ev["append"][1].record(st)
        if host is not None:
            # the previous turn's decode has read q / new K/V, and this turn's
            # appends have read the tool slots (both enqueued on the stream);
            # the two kinds of copies go on streams of their own, so that the
            # queries never queue behind the next turn's tool responses
            self._h2d.wait_stream(st)
            with torch.cuda.stream(self._h2d):
                for t in range(STEADY_DECODE):
                    self.q[t].copy_(host["q"][t], non_blocking=True)
                    self.knew[t].copy_(host["kn"][t], non_blocking=True)
                    self.vnew[t].copy_(host["vn"][t], non_blocking=True)
                    self._ready[t].record(self._h2d)
        for t in range(STEADY_DECODE):
            if host is not None and t == 8 and k + 1 < self.n_turns:
                # the next turn's tool responses go up once this turn's
                # queries have (started at the turn start, the 27 GB copy
                # held the first decode step's 0.1 GB of queries back)
                self._h2d_tool.wait_stream(st)
                h0 = time.perf_counter()
                self._tool_copy(k + 1, host, timed=True)
                self._tool_host_s[k + 1] = time.perf_counter() - h0
                self._prefetched = k + 1
            if host is not None:
                st.wait_event(self._ready[t])
            c.append(self.seqs, [1] * STEADY_SEQS, self.knew[t], self.vnew[t])
            # one event pair around the step's L calls: an event between two
            # decode calls would end the overlap of their launches
            if ev is not None:
                ev["dec"][t][0].record(st)
            for l in range(L):
                # the last layer's output of every step has its own device
                # slot, read back on a stream of its own (a read-back on the
                # compute stream would wait behind the input copies)
                dst = host["out_dev"][t] if host is not None and l == L - 1 else self.out[l]
                c.decode_attention(l, self.q[t, l], self.seqs, dst)
            if ev is not None:
                ev["dec"][t][1].record(st)
            if host is not None:
                self._done[t].record(st)
                self._d2h.wait_event(self._done[t])
                with torch.cuda.stream(self._d2h):
                    host["out"][t].copy_(host["out_dev"][t], non_blocking=True)
        self._drop_repos(k, ev)

    def _tool_copy(self, k, host, timed=False):
        """Turn k's tool-response K/V from pinned host memory into the group
        slots, on the copy stream (``timed``: an event pair around it)."""
        torch = self.torch
        if timed:
            self._tool_ev[k] = events(torch, 1)[0]
        with torch.cuda.stream(self._h2d_tool):
            if timed:
                self._tool_ev[k][0].record(self._h2d_tool)
            for gi, g in enumerate(self.groups):
                n = sum(self.turns[i][k].tool_len for i in g)
                kk, vv = self.raw(n, host["slots"][gi])
                hk, hv = self.raw(n, (host["k"], host["v"]))
                kk.copy_(hk, non_blocking=True)
                vv.copy_(hv, non_blocking=True)
                self._tool_ready[gi].record(self._h2d_tool)
            if timed:
                self._tool_ev[k][1].record(self._h2d_tool)

    def host_buffers(self):
        """Pinned host copies of one turn's inputs and outputs (tool responses
        sized for the largest group), plus one device slot per group for the
        tool responses (the first is the device-resident run's buffer)."""
        torch = self.torch
        pin = lambda x: torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x)
        n = self.sh.layers * self.tool_max * self.sh.hkv * self.sh.head_dim
        h = {"k": pin(self.kraw[:n]), "v": pin(self.vraw[:n]), "q": pin(self.q),
             "kn": pin(self.knew), "vn": pin(self.vnew),
             "out": torch.empty((STEADY_DECODE, STEADY_SEQS, self.sh.hq, self.sh.head_dim),
                                dtype=torch.float32, pin_memory=True)}
        h["out_dev"] = torch.empty(h["out"].shape, dtype=torch.float32, device="cuda")
        h["slots"] = [(self.kraw, self.vraw)] + [
            (torch.empty(n, dtype=torch.bfloat16, device="cuda"),
             torch.empty(n, dtype=torch.bfloat16, device="cuda"))
            for _ in range(len(self.groups) - 1)]
        return h

    def h2d_bytes(self, k):
        a = self.acct[k]
        per_tok = self.sh.layers * self.sh.hkv * self.sh.head_dim * BYTES_EL * 2
        return (a["tool"] * per_tok + self.q.numel() * BYTES_EL
                + (self.knew.numel() + self.vnew.numel()) * BYTES_EL)

    def close(self):
        self.cache.close()
        for name in ("kraw", "vraw", "q", "knew", "vnew", "out", "cache"):
            setattr(self, name, None)
        self.torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# the 8B- and 120B-shaped traces (blocks): fork, drop, reposition, decode
# ---------------------------------------------------------------------------

class TraceBench:
    """One step = fork the prepared sequences (pages shared), drop their tool
    spans, one batched reposition, then decode steps x (append one token per
    sequence + decode attention on every layer), free the forks."""

    def __init__(self, spec, rank, batch=None, layers=None, decode=None):
        import dataclasses
        import torch
        from agent_kv_cache_gb300 import Cache, build
        from workloads import device as dev
        self.torch, self.dev = torch, dev
        build()
        dev.build()
        sh = spec["shape"]
        if layers:
            sh = dataclasses.replace(sh, layers=layers)
        self.sh, self.name = sh, spec["name"]
        self.B = batch or spec["batch"]
        self.N, self.DEC, self.seed = spec["n_tokens"], decode or spec["decode"], spec["seed"]
        mk = traces.gptoss_batch if spec["name"] == "gptoss120b" else traces.llama8b_batch
        self.trajs = mk(self.seed, batch=max(self.B, spec["batch"]), n_total=self.N)[:self.B]
        S, L, H, D, Hq = sh.page_size, sh.layers, sh.hkv, sh.head_dim, sh.hq
        kvt = kvt_of(sh)
        # algorithmic bytes of one step (host mirror of the sequences)
        moved, rs, drop = [], [], 0
        for tr in self.trajs:
            sim = Sim(S)
            sim.append(self.N)
            drop += drop_bytes(sim)
            sim.drop(tr.drop_ranges)
            moved.append(sim.reposition()[0])
            rs.append(sim.held())
        self.calls = [decode_call_bytes(sh, [r + t + 1 for r in rs],
                                        [-(-(r + t + 1) // S) for r in rs])
                      for t in range(self.DEC)]
        self.bytes = dict(repos=2 * L * sum(moved) * kvt, moved=sum(moved),
                          decode=L * sum(self.calls), append=self.DEC * self.B * L * kvt * 2,
                          drop=drop)
        self.bytes["total"] = sum(self.bytes[k] for k in ("repos", "decode", "append", "drop"))
        max_pages = self.B * (self.N // S) + sum(-(-(r + self.DEC) // S) + 2 for r in rs) + 256
        self.cache = Cache(L, Hq, H, D, S, sh.dtype, max_pages, 2 * self.B + 2,
                           self.N + self.DEC + S, sh.rope_theta)
        self.stream = self.cache.stream
        self.tags = rank_tags(rank, self.B)
        w = synth.width_for(sh.dtype)
        kbuf = torch.empty((L, CHUNK, H, D), dtype=torch.bfloat16, device="cuda")
        vbuf = torch.empty_like(kbuf)
        self.base = []
        for b in range(self.B):
            s = self.cache.seq_create()
            for t0 in range(0, self.N, CHUNK):
                n = min(CHUNK, self.N - t0)
                k1 = dev.kv_tokens(kbuf, self.seed, self.tags[b], synth.KIND_K, range(L), t0, n, H, D, w)
                v1 = dev.kv_tokens(vbuf, self.seed, self.tags[b], synth.KIND_V, range(L), t0, n, H, D, w)
                self.cache.append([s], [n], kbuf[:, :n].contiguous() if n < CHUNK else kbuf,
                                  vbuf[:, :n].contiguous() if n < CHUNK else vbuf)
                torch.cuda.synchronize()
                del k1, v1
            self.base.append(s)
        del kbuf, vbuf
        self.q = torch.empty((self.DEC, L, self.B, Hq, D), dtype=torch.bfloat16, device="cuda")
        self.knew = torch.empty((self.DEC, L, self.B, H, D), dtype=torch.bfloat16, device="cuda")
        self.vnew = torch.empty_like(self.knew)
        keep = []
        for t in range(self.DEC):
            for l in range(L):
                keep.append(dev.queries(self.q[t, l], self.seed, self.tags, l, t, Hq, D, w))
            keep.append(dev.kv_tokens_multi(self.knew[t], self.seed, self.tags, synth.KIND_K,
                                            range(L), [self.N + t] * self.B, 1, H, D, w))
            keep.append(dev.kv_tokens_multi(self.vnew[t], self.seed, self.tags, synth.KIND_V,
                                            range(L), [self.N + t] * self.B, 1, H, D, w))
        self.out = torch.empty((L, self.B, Hq, D), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        del keep
        assert self.cache.sync_errors() == 0

    def events(self):
        return {"ops": events(self.torch, 1)[0], "dec": events(self.torch, self.DEC)}

    def step(self, ev=None, host=None):
        """One pass.  ``ev``: events for per-call timing; ``host``: pinned host
        inputs/outputs for the end-to-end variant."""
        c, torch, st = self.cache, self.torch, self.stream
        L = self.sh.layers
        if host is not None:
            # every decode step's inputs go up on a copy stream (each step has
            # its own device slot), overlapping the fork / drop / reposition
            # and the earlier decode steps; decode step t waits for its copy
            if not hasattr(self, "_h2d"):
                self._h2d = torch.cuda.Stream()
                self._ready = [torch.cuda.Event() for _ in range(self.DEC)]
            self._h2d.wait_stream(st)   # the previous pass has read the slots
            with torch.cuda.stream(self._h2d):
                for t in range(self.DEC):
                    self.q[t].copy_(host["q"][t], non_blocking=True)
                    self.knew[t].copy_(host["k"][t], non_blocking=True)
                    self.vnew[t].copy_(host["v"][t], non_blocking=True)
                    self._ready[t].record(self._h2d)
        forks = [c.seq_fork(b) for b in self.base]
        if ev is not None:
            ev["ops"][0].record(st)
        for f, tr in zip(forks, self.trajs):
            c.drop(f, tr.drop_ranges)
        c.reposition(forks)
        if ev is not None:
            ev["ops"][1].record(st)
        for t in range(self.DEC):
            if host is not None:
                st.wait_event(self._ready[t])
            c.append(forks, [1] * self.B, self.knew[t], self.vnew[t])
            if ev is not None:
                ev["dec"][t][0].record(st)
            for l in range(L):
                c.decode_attention(l, self.q[t, l], forks, self.out[l])
            if ev is not None:
                ev["dec"][t][1].record(st)
            if host is not None:
                host["out"][t].copy_(self.out[L - 1], non_blocking=True)
        for f in forks:
            c.seq_free(f)

    def run(self, warmup, steps):
        """Warm-up passes, then timed passes; returns the block's figures."""
        torch = self.torch
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        assert self.cache.sync_errors() == 0
        evs = [self.events() for _ in range(steps)]
        start, stop = events(torch, 1)[0]
        start.record(self.stream)
        for i in range(steps):
            self.step(ev=evs[i])
        stop.record(self.stream)
        torch.cuda.synchronize()
        assert self.cache.sync_errors() == 0
        ms = start.elapsed_time(stop) / steps
        L = self.sh.layers
        dec_ms = np.array([[s.elapsed_time(e) / L for s, e in ev["dec"]] for ev in evs])
        ops_ms = float(np.mean([ev["ops"][0].elapsed_time(ev["ops"][1]) for ev in evs]))
        call_b = np.array(self.calls)
        achieved = float(np.sum(call_b) * steps / (np.sum(dec_ms) * 1e-3) / 1e9)
        # one call at a time (after an unrelated kernel), on the first decode
        # step's state: fork, drop, reposition, one append
        forks = [self.cache.seq_fork(b) for b in self.base]
        for f, tr in zip(forks, self.trajs):
            self.cache.drop(f, tr.drop_ranges)
        self.cache.reposition(forks)
        self.cache.append(forks, [1] * self.B, self.knew[0], self.vnew[0])
        iso_us = isolated_decode(torch, self.cache, range(L), self.q[0], forks, self.out)
        for f in forks:
            self.cache.seq_free(f)
        peak, _ = hbm_peak()
        by = self.bytes
        return {
            "ms_per_step": round(ms, 3), "steps": steps, "warmup": warmup,
            "gbs": round(by["total"] / (ms * 1e-3) / 1e9, 1),
            "frac": round(by["total"] / (ms * 1e-3) / 1e9 / peak, 4),
            "bytes_per_step": by["total"],
            "decode_tok_s": round(self.B * self.DEC / (float(np.sum(dec_ms)) * L / steps * 1e-3), 1),
            "decode": {"kernel": "k_decode_mma", "avg_call_us": round(float(np.mean(dec_ms)) * 1e3, 2),
                       "algorithmic_bytes_per_call": int(np.mean(call_b)),
                       "gbs": round(achieved, 1), "frac": round(achieved / peak, 4),
                       "isolated_call_us": round(iso_us, 2),
                       "isolated_gbs": round(call_b[0] / (iso_us * 1e-6) / 1e9, 1),
                       "isolated_frac": round(call_b[0] / (iso_us * 1e-6) / 1e9 / peak, 4)},
            "reposition": {"kernel": "k_compact + k_gather (drop included)", "ms": round(ops_ms, 3),
                           "moved_tokens": by["moved"], "algorithmic_bytes": by["repos"],
                           "gbs": round(by["repos"] / (ops_ms * 1e-3) / 1e9, 1),
                           "frac": round(by["repos"] / (ops_ms * 1e-3) / 1e9 / peak, 4)},
        }

    def workload(self):
        sh = self.sh
        pct = {"llama8b": "~60%", "gptoss120b": "~80%", "llama70b": "~60%"}[self.name]
        return (f"{sh.name}-shaped agent trace: {sh.layers} layers, {sh.hq}/{sh.hkv} heads, "
                f"head_dim {sh.head_dim}, {sh.dtype}, rope theta {sh.rope_theta:g}, page "
                f"{sh.page_size}; batch {self.B} x {self.N} logical tokens, tool spans dropped "
                f"({pct}), 1 reposition, {self.DEC} decode steps")

    def close(self):
        self.cache.close()
        for name in ("q", "knew", "vnew", "out", "cache"):
            setattr(self, name, None)
        self.torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# the branching histories (block): 64 forks of one prefix, their operations,
# batched decode over all of them
# ---------------------------------------------------------------------------

class BranchBench:
    """One step = fork the prefix into 64 branches (pages shared), apply every
    branch's 1-6 drop / reposition operations (round by round: the round's
    drops, then one batched reposition of the branches whose operation it
    is), 128 decode steps x (append + decode attention on all 32 layers)
    over all 64 branches, free the branches."""

    def __init__(self, rank, layers=None):
        import dataclasses
        import torch
        from agent_kv_cache_gb300 import Cache, build
        from workloads import device as dev
        self.torch, self.dev = torch, dev
        build()
        dev.build()
        sh = BRANCH["shape"]
        if layers:
            sh = dataclasses.replace(sh, layers=layers)
        self.sh = sh
        P, NB, DEC, seed = BRANCH["prefix"], BRANCH["branches"], BRANCH["decode"], BRANCH["seed"]
        self.P, self.NB, self.DEC, self.seed = P, NB, DEC, seed
        _, self.branches = traces.branching(seed, n_branches=NB, prefix_len=P)
        self.rounds = max(len(b.ops) for b in self.branches)
        S, L, H, D, Hq = sh.page_size, sh.layers, sh.hkv, sh.head_dim, sh.hq
        kvt = kvt_of(sh)
        moved = drop = 0
        peak_private, actives, pages, held = 0, [], [], []
        for br in self.branches:
            sim = Sim(S, logical=np.arange(P), shared_pages=P // S)
            top = 0
            for op in br.ops:
                if op[0] == "drop":
                    drop += drop_bytes(sim)
                    sim.drop(op[1])
                else:
                    before = sim.private_pages()
                    mv, fr = sim.reposition()
                    moved += mv
                    top = max(top, before + fr)
            peak_private += max(top, sim.private_pages()) + -(-DEC // S) + 2
            actives.append(sim.active())
            pages.append(sim.active_pages())
            held.append(sim.held())
        self.calls = [decode_call_bytes(sh, [a + t + 1 for a in actives],
                                        [p + (-(-(h + t + 1) // S)) - (-(-h // S))
                                         for p, h in zip(pages, held)])
                      for t in range(DEC)]
        self.bytes = dict(repos=2 * L * moved * kvt, moved=moved, decode=L * sum(self.calls),
                          append=DEC * NB * L * kvt * 2, drop=drop)
        self.bytes["total"] = sum(self.bytes[k] for k in ("repos", "decode", "append", "drop"))
        max_pages = P // S + peak_private + 512
        self.cache = Cache(L, Hq, H, D, S, sh.dtype, max_pages, NB + 4, P + DEC + 64,
                           sh.rope_theta)
        self.stream = self.cache.stream
        w = synth.width_for(sh.dtype)
        tag = rank * 1000 + 1
        self.root = self.cache.seq_create()
        kbuf = torch.empty((L, CHUNK, H, D), dtype=torch.bfloat16, device="cuda")
        vbuf = torch.empty_like(kbuf)
        for t0 in range(0, P, CHUNK):
            n = min(CHUNK, P - t0)
            k1 = dev.kv_tokens(kbuf, seed, tag, synth.KIND_K, range(L), t0, n, H, D, w)
            v1 = dev.kv_tokens(vbuf, seed, tag, synth.KIND_V, range(L), t0, n, H, D, w)
            self.cache.append([self.root], [n], kbuf[:, :n].contiguous() if n < CHUNK else kbuf,
                              vbuf[:, :n].contiguous() if n < CHUNK else vbuf)
            torch.cuda.synchronize()
            del k1, v1
        del kbuf, vbuf
        tags = [tag + 1 + b for b in range(NB)]
        self.q = torch.empty((DEC, L, NB, Hq, D), dtype=torch.bfloat16, device="cuda")
        self.knew = torch.empty((DEC, L, NB, H, D), dtype=torch.bfloat16, device="cuda")
        self.vnew = torch.empty_like(self.knew)
        keep = [dev.fill(x, [(synth.stream_key(seed, tag, kind, 99), 0, 0)], x.numel(), w)
                for x, kind in ((self.q, synth.KIND_Q), (self.knew, synth.KIND_K),
                                (self.vnew, synth.KIND_V))]
        del tags
        self.out = torch.empty((L, NB, Hq, D), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        del keep
        self.unique = None

    def _ops(self, kids):
        c = self.cache
        for i in range(self.rounds):
            rep = []
            for k, br in zip(kids, self.branches):
                if i < len(br.ops):
                    if br.ops[i][0] == "drop":
                        c.drop(k, br.ops[i][1])
                    else:
                        rep.append(k)
            if rep:
                c.reposition(rep)

    def _unique_bytes(self, kids):
        """Decode-call bytes with each pool page read once (pages shared by
        several branches counted once)."""
        sh = self.sh
        uniq = set()
        pages = 0
        for k in kids:
            pt, act = self.cache.page_table(k)
            uniq.update(int(pt[a]) for a in act)
            pages += len(act)
        return (len(uniq) * sh.page_size * kvt_of(sh) + len(kids) * sh.hq * sh.head_dim
                * (BYTES_EL + 4) + pages * (4 + 4 + sh.page_size // 8))

    def step(self, ev=None, count_unique=False):
        c, st = self.cache, self.stream
        L = self.sh.layers
        kids = [c.seq_fork(self.root) for _ in range(self.NB)]
        if ev is not None:
            ev["ops"][0].record(st)
        self._ops(kids)
        if ev is not None:
            ev["ops"][1].record(st)
        uniq = []
        for t in range(self.DEC):
            c.append(kids, [1] * self.NB, self.knew[t], self.vnew[t])
            if count_unique and t in (0, self.DEC - 1):
                uniq.append(self._unique_bytes(kids))
            if ev is not None:
                ev["dec"][t][0].record(st)
            for l in range(L):
                c.decode_attention(l, self.q[t, l], kids, self.out[l])
            if ev is not None:
                ev["dec"][t][1].record(st)
        if count_unique:
            self.unique = list(np.linspace(uniq[0], uniq[1], self.DEC))
            self.plan = c.decode_plan_stats()
        for k in kids:
            c.seq_free(k)

    def run(self, warmup, steps):
        torch = self.torch
        for i in range(warmup):
            self.step(count_unique=(i == 0))
        torch.cuda.synchronize()
        assert self.cache.sync_errors() == 0
        evs = [{"ops": events(torch, 1)[0], "dec": events(torch, self.DEC)} for _ in range(steps)]
        start, stop = events(torch, 1)[0]
        start.record(self.stream)
        for i in range(steps):
            self.step(ev=evs[i])
        stop.record(self.stream)
        torch.cuda.synchronize()
        assert self.cache.sync_errors() == 0
        ms = start.elapsed_time(stop) / steps
        L = self.sh.layers
        dec_ms = np.array([[s.elapsed_time(e) / L for s, e in ev["dec"]] for ev in evs])
        ops_ms = float(np.mean([ev["ops"][0].elapsed_time(ev["ops"][1]) for ev in evs]))
        call_b = np.array(self.calls)
        uniq_b = np.array(self.unique)
        sec = float(np.sum(dec_ms)) * 1e-3          # per-call times: bytes per call / sec
        per_branch = float(np.sum(call_b) * steps / sec / 1e9)
        unique = float(np.sum(uniq_b) * steps / sec / 1e9)
        kids = [self.cache.seq_fork(self.root) for _ in range(self.NB)]
        self._ops(kids)
        self.cache.append(kids, [1] * self.NB, self.knew[0], self.vnew[0])
        iso_us = isolated_decode(torch, self.cache, range(L), self.q[0], kids, self.out)
        for k in kids:
            self.cache.seq_free(k)
        peak, _ = hbm_peak()
        by = self.bytes
        total = by["total"] - by["decode"] + L * float(np.sum(uniq_b))
        return {
            "ms_per_step": round(ms, 3), "steps": steps, "warmup": warmup,
            "gbs": round(total / (ms * 1e-3) / 1e9, 1),
            "frac": round(total / (ms * 1e-3) / 1e9 / peak, 4),
            "bytes_per_step": int(total),
            "bytes_note": "decode counted by unique pool pages (a page several branches hold "
                          "is read once)",
            "decode_tok_s": round(self.NB * self.DEC / (sec * L / steps), 1),
            "decode": {"kernel": "k_decode_share_tc + k_decode_mma",
                       "avg_call_us": round(float(np.mean(dec_ms)) * 1e3, 2),
                       "unique_page_bytes_per_call": int(np.mean(uniq_b)),
                       "per_branch_bytes_per_call": int(np.mean(call_b)),
                       "gbs": round(unique, 1), "frac": round(unique / peak, 4),
                       "gbs_per_branch": round(per_branch, 1), "plan": self.plan,
                       "isolated_call_us": round(iso_us, 2),
                       "isolated_gbs": round(uniq_b[0] / (iso_us * 1e-6) / 1e9, 1),
                       "isolated_frac": round(uniq_b[0] / (iso_us * 1e-6) / 1e9 / peak, 4)},
            "reposition": {"kernel": "k_drop + k_compact + k_gather (every branch's operations)",
                           "ms": round(ops_ms, 3), "moved_tokens": by["moved"],
                           "algorithmic_bytes": by["repos"],
                           "gbs": round(by["repos"] / (ops_ms * 1e-3) / 1e9, 1),
                           "frac": round(by["repos"] / (ops_ms * 1e-3) / 1e9 / peak, 4)},
        }

    def workload(self):
        sh = self.sh
        return (f"branching histories, {sh.name}-shaped ({sh.layers} layers, {sh.hq}/{sh.hkv} "
                f"heads, head_dim {sh.head_dim}): one {self.P}-token prefix forked into all "
                f"{self.NB} branches, each applying its 1-6 drop / reposition operations, then "
                f"{self.DEC} batched decode steps over the {self.NB} branches")

    def close(self):
        self.cache.close()
        for name in ("q", "knew", "vnew", "out", "cache"):
            setattr(self, name, None)
        self.torch.cuda.empty_cache()


def run_blocks(rank, names, steps, warmup=3):
    out = {}
    for name in names:
        if name == "branching":
            b = BranchBench(rank)
        else:
            b = TraceBench(TRACE8B if name == "llama8b" else TRACE120B, rank)
        res = b.run(warmup, steps)
        res["workload"] = b.workload()
        out[name] = res
        b.close()
        del b
    return out


# ---------------------------------------------------------------------------
# segment-batch restore attention (its own line: --restore)
# ---------------------------------------------------------------------------

RESTORE_SEED = traces.seed_for(5)


def restore_visible(prog):
    """Sum over appended tokens of the keys each one attends (itself included)."""
    alive = vis = 0
    for op in prog:
        if op[0] == "append":
            n = op[1]
            vis += n * alive + n * (n + 1) // 2
            alive += n
        elif op[0] == "drop":
            alive -= sum(e - b for b, e in op[1])
    return vis


def restore_arm(args):
    """Restore attention of one long agent sequence on every layer: per layer
    one akv_restore_attention call over the whole program (~34k tokens,
    10 repositions).  FLOPs are algorithmic: 4 * D * hq per visible
    (query, key) pair (Q K^T and P V)."""
    import torch
    from agent_kv_cache_gb300 import Cache, build
    from workloads import device as dev
    build()
    dev.build()
    sh = SHAPE
    prog = traces.restore_program(RESTORE_SEED)
    n = sum(op[1] for op in prog if op[0] == "append")
    cache = Cache(sh.layers, sh.hq, sh.hkv, sh.head_dim, sh.page_size, sh.dtype, 16, 2, n + 64,
                  sh.rope_theta)
    if args.restore_cuda_cores:
        cache.set_restore_tensor_cores(False)
    w = synth.width_for(sh.dtype)
    st = cache.stream
    q = torch.empty((n, sh.hq, sh.head_dim), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((n, sh.hkv, sh.head_dim), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    keep = [dev.fill(x, [(synth.stream_key(RESTORE_SEED, 1, kind, 0), 0, 0)], x.numel(), w)
            for x, kind in ((q, synth.KIND_Q), (k, synth.KIND_K), (v, synth.KIND_V))]
    out = torch.empty((n, sh.hq, sh.head_dim), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    del keep
    flops = 4.0 * sh.head_dim * sh.hq * restore_visible(prog)
    for _ in range(args.warmup):
        for l in range(sh.layers):
            cache.restore_attention(prog, l, q, k, v, out=out)
    torch.cuda.synchronize()
    w = cache.sync_errors()
    assert w == 0, f"device error word 0x{w:x} after the warm-up"
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps * sh.layers)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = cache.kernel_launches()
    with torch.cuda.stream(st):
        start.record(st)
        for i in range(args.steps):
            for l in range(sh.layers):
                e = evs[i * sh.layers + l]
                e[0].record(st)
                cache.restore_attention(prog, l, q, k, v, out=out)
                e[1].record(st)
        stop.record(st)
    torch.cuda.synchronize()
    assert cache.sync_errors() == 0
    launches = (cache.kernel_launches() - n0) // args.steps
    ms = start.elapsed_time(stop) / args.steps
    call_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = peaks.get("bf16_tflops_sustained", 1700.0)
    achieved = flops / (call_ms * 1e-3) / 1e12
    line = {
        "metric": "segment-batch restore attention TFLOP/s (algorithmic, visible pairs)",
        "value": round(sh.layers * flops / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded SplitMix64 q/K/V)",
        "config": {"workload": f"{sh.name}-shaped long-running agent sequence: {n} tokens, "
                               f"{sum(op[0] == 'repos' for op in prog)} repositions, "
                               f"{sum(op[0] == 'drop' for op in prog)} drop operations; one step "
                               f"= restore attention on all {sh.layers} layers",
                   "kernel": "CUDA cores" if args.restore_cuda_cores
                   else "tensor cores (tcgen05, accumulators in tensor memory)",
                   "flops_per_layer": flops, "tokens": n},
        "roofline": {"kernel": "restore attention (temporary key versions + attention)",
                     "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": "measured sustained" if "bf16_tflops_sustained" in peaks
                     else "fallback", "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": None, "avg_call_ms": round(call_ms, 3)},
        "gpu_launches": int(launches),
    }
    # recovery: the older half of the sequence lost its KV; the plan picks
    # the missing tokens the end state reads and everything their
    # recomputation reads, and restore attention runs over those only
    missing = np.zeros(n, np.uint8)
    missing[:n // 2] = 1
    h0 = time.perf_counter()
    plan = Cache.plan_recovery(prog, n, missing)
    plan_ms = (time.perf_counter() - h0) * 1e3
    for l in range(sh.layers):
        cache.restore_attention_tokens(prog, l, q, k, v, plan, out=out)
    torch.cuda.synchronize()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        r0.record(st)
        for _ in range(args.steps):
            for l in range(sh.layers):
                cache.restore_attention_tokens(prog, l, q, k, v, plan, out=out)
        r1.record(st)
    torch.cuda.synchronize()
    assert cache.sync_errors() == 0
    line["recovery"] = {
        "what": "the first half of the tokens missing; restore attention over the planned "
                "tokens only (akv_restore_plan_recovery + akv_restore_attention_tokens), "
                "all layers",
        "missing": int(missing.sum()), "recomputed": len(plan), "plan_host_ms": round(plan_ms, 3),
        "ms_per_step": round(r0.elapsed_time(r1) / args.steps, 3),
        "full_restore_ms_per_step": round(ms, 3)}
    print(json.dumps(line), flush=True)
    cache.close()


# ---------------------------------------------------------------------------
# history-keyed prefix sharing and drop-aware eviction (its own line: --prefix)
# ---------------------------------------------------------------------------

def prefix_arm(args):
    """One long-running agent sequence (8B shape, ~34k tokens, 30 turns,
    drops of old tool spans and a reposition every 3 turns) published at the
    end of every turn (30 entries).  Timed: host matching of two requests,
    an exact fork that continues the conversation (every page shared), a
    retrigger fork of a request that skipped the last reposition (every
    survivor after the first dropped span rotated into fresh pages: the
    k_transplant kernel, HBM-bound), and drop-aware eviction of all
    entries."""
    import torch
    from agent_kv_cache_gb300 import Cache, PrefixIndex, build
    from workloads import device as dev
    build()
    dev.build()
    sh = SHAPE
    seed = RESTORE_SEED
    turns = traces.turn_programs(seed)
    n_total = sum(op[1] for t in turns for op in t if op[0] == "append")
    ids = traces.token_ids(seed, n_total + 64)
    S = sh.page_size
    max_pages = 16384
    cache = Cache(sh.layers, sh.hq, sh.hkv, sh.head_dim, S, sh.dtype, max_pages, 64,
                  n_total + 64, sh.rope_theta)
    idx = PrefixIndex(S)
    st = cache.stream
    w = synth.width_for(sh.dtype)
    live = cache.seq_create()
    hist, t = [], 0
    entries = []
    for ops in turns:
        for op in ops:
            if op[0] == "append":
                n = op[1]
                for c0 in range(0, n, CHUNK):
                    m = min(CHUNK, n - c0)
                    k = torch.empty((sh.layers, m, sh.hkv, sh.head_dim), dtype=torch.bfloat16,
                                    device="cuda")
                    v = torch.empty_like(k)
                    keep = [dev.kv_tokens(k, seed, 1, synth.KIND_K, range(sh.layers), t, m,
                                          sh.hkv, sh.head_dim, w),
                            dev.kv_tokens(v, seed, 1, synth.KIND_V, range(sh.layers), t, m,
                                          sh.hkv, sh.head_dim, w)]
                    torch.cuda.synchronize()
                    cache.append([live], [m], k, v, ids[t:t + m].tolist())
                    torch.cuda.synchronize()
                    del keep
                    t += m
            elif op[0] == "drop":
                cache.drop(live, op[1])
            else:
                cache.reposition([live])
        hist += ops
        entries.append(cache.prefix_publish(idx, live, hist, ids[:t].tolist()))
    torch.cuda.synchronize()
    assert cache.sync_errors() == 0
    n_tok = t
    # requests: continue the conversation (exact), and the history without its
    # last reposition followed by one new turn (retrigger)
    cont = hist + [("append", 64)]
    cont_ids = ids[:n_tok + 64].tolist()
    assert hist[-1][0] == "repos"
    skip = hist[:-1] + [("append", 64)]

    def timed_host(fn, reps):
        fn()
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        return (time.perf_counter() - t0) / reps

    match_cont = timed_host(lambda: idx.match(cont, cont_ids), 20)
    match_skip = timed_host(lambda: idx.match(skip, cont_ids), 20)
    m_skip = idx.match(skip, cont_ids)
    m_cont = idx.match(cont, cont_ids)
    # forks: GPU time by events on the cache stream (a spin on the stream
    # first, so that the call's host planning is over before the start event
    # fires and only the GPU work is timed), host time by the clock
    def fork_times(prog, reps):
        gpu_ms, host_s = [], []
        for i in range(args.warmup + reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(st):
                torch.cuda._sleep(20_000_000)
            t0 = time.perf_counter()
            a.record(st)
            child, m = cache.prefix_fork(idx, prog, cont_ids)
            b.record(st)
            t1 = time.perf_counter()
            torch.cuda.synchronize()
            if i >= args.warmup:
                gpu_ms.append(a.elapsed_time(b))
                host_s.append(t1 - t0)
            info = cache.info(child)
            cache.seq_free(child)
        return float(np.mean(gpu_ms)), float(np.mean(host_s)), m, info

    n0 = cache.kernel_launches()
    ex_gpu, ex_host, m1, info1 = fork_times(cont, args.steps)
    re_gpu, re_host, m2, info2 = fork_times(skip, args.steps)
    launches = cache.kernel_launches() - n0
    assert cache.sync_errors() == 0
    moved = m2["n_rotated"]
    # algorithmic bytes of the retrigger fork: every rotated key and its value
    # read and written once on every layer, plus the keys copied unrotated
    # into fresh pages (tokens of a moved page that keep their position)
    per_tok = sh.layers * 2 * sh.hkv * sh.head_dim * BYTES_EL
    plan_tokens = info2["n_active"]
    # tokens in fresh pages = rotated keys + unrotated ones sharing their pages;
    # count from the page table: pages not shared with the entry
    child, _ = cache.prefix_fork(idx, skip, cont_ids)
    pc, _ = cache.page_table(child)
    pe, _ = cache.page_table(m2["entry"])
    keep = cache.keep_mask(child)
    fresh_pages = [k for k in range(len(pc)) if pc[k] >= 0 and (k >= len(pe) or pc[k] != pe[k])]
    fresh_tok = int(sum(keep[k * S:(k + 1) * S].sum() for k in fresh_pages))
    cache.seq_free(child)
    algo = 2 * fresh_tok * per_tok
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = peaks.get("hbm_gbs", 6800.0)
    gbs = algo / (re_gpu * 1e-3) / 1e9
    used_before = cache.pool_stats()[1]
    t0 = time.perf_counter()
    freed, n_ev = cache.prefix_evict(idx, 1 << 30)
    ev_s = time.perf_counter() - t0
    cache.seq_free(live)
    line = {
        "metric": "prefix fork (retrigger) GB/s & history-keyed matching / eviction latency",
        "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (seeded K/V and token ids, seeded agent turn schedule)",
        "config": {"workload": f"{sh.name}-shaped long-running agent sequence: {n_tok} tokens, "
                               f"{len(turns)} turns published as {len(set(entries))} entries; "
                               "requests: continue (exact), skip the last reposition (retrigger)",
                   "page_size": S},
        "match_us": {"continue": round(match_cont * 1e6, 1), "skip_repos": round(match_skip * 1e6, 1)},
        "exact_fork": {"match": m1, "gpu_ms": round(ex_gpu, 4), "host_ms": round(ex_host * 1e3, 3),
                       "tokens": info1["n_active"]},
        "retrigger_fork": {"match": m2, "gpu_ms": round(re_gpu, 4),
                           "host_ms": round(re_host * 1e3, 3), "fresh_pages": len(fresh_pages),
                           "tokens_in_fresh_pages": fresh_tok, "tokens": plan_tokens,
                           "algorithmic_bytes": algo},
        "roofline": {"kernel": "k_transplant (retrigger fork)", "bound": "hbm",
                     "achieved": round(gbs, 1), "peak": peak,
                     "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
                     "unit": "GB/s", "frac": round(gbs / peak, 4), "traffic": None},
        "eviction": {"entries": n_ev, "pages_freed": freed, "pages_used_before": used_before,
                     "host_ms": round(ev_s * 1e3, 3)},
        "gpu_launches": int(launches),
    }
    print(json.dumps(line), flush=True)
    cache.close()


# ---------------------------------------------------------------------------
# decode and reposition bandwidth on the other workload shapes
# (--config-kernels gptoss120b,branching,llama70b): one line per workload
# ---------------------------------------------------------------------------

def _decode_bytes(cache, seqs, sh):
    """Algorithmic bytes of one decode call: per sequence (every sequence's
    active K/V), and with pages shared by several sequences counted once."""
    kvt = 2 * sh.hkv * sh.head_dim * BYTES_EL
    act = sum(cache.info(s)["n_active"] for s in seqs)
    pages = sum(cache.info(s)["n_active_pages"] for s in seqs)
    fixed = len(seqs) * sh.hq * sh.head_dim * (BYTES_EL + 4) + pages * (8 + sh.page_size // 8)
    uniq = set()
    for s in seqs:
        pt, act_pages = cache.page_table(s)
        uniq.update(int(pt[k]) for k in act_pages)
    return act * kvt + fixed, len(uniq) * sh.page_size * kvt + fixed


def _moved(cache, seq, sh):
    """Survivors a reposition relocates: those at or after the first full page
    that holds a dropped slot."""
    keep = cache.keep_mask(seq)
    dead = np.flatnonzero(~keep)
    if dead.size == 0:
        return 0
    kept = (int(dead[0]) // sh.page_size) * sh.page_size
    return int(keep.sum()) - kept


def kernels_arm(args):
    import torch
    from agent_kv_cache_gb300 import Cache, build
    from workloads import device as dev
    build()
    dev.build()
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    peak = peaks.get("hbm_gbs", 6800.0)
    st_events = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))

    def append(cache, seq, tag, t0, n, sh, seed):
        L, H, D = sh.layers, sh.hkv, sh.head_dim
        w = synth.width_for(sh.dtype)
        for c0 in range(0, n, CHUNK):
            m = min(CHUNK, n - c0)
            k = torch.empty((L, m, H, D), dtype=torch.bfloat16, device="cuda")
            v = torch.empty_like(k)
            keep = [dev.kv_tokens(k, seed, tag, synth.KIND_K, range(L), t0 + c0, m, H, D, w),
                    dev.kv_tokens(v, seed, tag, synth.KIND_V, range(L), t0 + c0, m, H, D, w)]
            torch.cuda.synchronize()
            cache.append([seq], [m], k, v)
            torch.cuda.synchronize()
            del keep

    def measure(name, cache, sh, bases, drops, seed, note, decode_steps=2, sharing=None):
        """Fork the prepared sequences, drop, time one batched reposition and
        decode_steps x (append + decode on every layer); repeated args.steps
        times after args.warmup.  sharing: decode sharing mode (None: default)."""
        st = cache.stream
        if sharing is not None:
            cache.set_decode_sharing(sharing)
        L, Hq, H, D = sh.layers, sh.hq, sh.hkv, sh.head_dim
        w = synth.width_for(sh.dtype)
        B = len(bases)
        q = torch.empty((L, B, Hq, D), dtype=torch.bfloat16, device="cuda")
        kn = torch.empty((L, B, H, D), dtype=torch.bfloat16, device="cuda")
        keep = [dev.queries(q[l], seed, list(range(B)), l, 0, Hq, D, w) for l in range(L)]
        keep.append(dev.kv_tokens_multi(kn, seed, list(range(B)), synth.KIND_K, range(L),
                                        [0] * B, 1, H, D, w))
        out = torch.empty((L, B, Hq, D), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        rep_ms, dec_ms, rep_bytes, dec_bytes, dec_ubytes = [], [], 0, [], []
        for it in range(args.warmup + args.steps):
            forks = [cache.seq_fork(b) for b in bases]
            for f, dr in zip(forks, drops):
                if dr:
                    cache.drop(f, dr)
            moved = sum(_moved(cache, f, sh) for f in forks)
            e = st_events()
            e[0].record(st)
            cache.reposition(forks)
            e[1].record(st)
            devs = []
            for t in range(decode_steps):
                cache.append(forks, [1] * B, kn, kn)
                db, dub = _decode_bytes(cache, forks, sh)
                ev = st_events()          # around the L back-to-back calls
                ev[0].record(st)
                for l in range(L):
                    cache.decode_attention(l, q[l], forks, out[l])
                ev[1].record(st)
                devs.append((ev, db, dub))
            torch.cuda.synchronize()
            assert cache.sync_errors() == 0
            if it >= args.warmup:
                rep_ms.append(e[0].elapsed_time(e[1]))
                rep_bytes = 2 * L * moved * 2 * H * D * BYTES_EL
                for ev, db, dub in devs:
                    dec_ms += [ev[0].elapsed_time(ev[1]) / L] * L
                    dec_bytes += [db] * L
                    dec_ubytes += [dub] * L
            for f in forks:
                cache.seq_free(f)
        del keep
        dgbs = float(np.sum(dec_bytes) / (np.sum(dec_ms) * 1e-3) / 1e9)
        ugbs = float(np.sum(dec_ubytes) / (np.sum(dec_ms) * 1e-3) / 1e9)
        rgbs = rep_bytes / (np.mean(rep_ms) * 1e-3) / 1e9 if rep_bytes else 0.0
        line = {
            "metric": f"decode attention and reposition HBM GB/s on the {name} workload",
            "value": round(ugbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic (seeded SplitMix64 K/V/q, seeded trace structure)",
            "config": {"workload": note, "batch": B, "layers": L, "heads": f"{Hq}/{H}",
                       "head_dim": D, "decode_steps_timed": decode_steps,
                       "decode_sharing": {None: "default (on)", 0: "off", 1: "on"}.get(sharing, sharing)},
            "decode": {"avg_call_us": round(float(np.mean(dec_ms)) * 1e3, 2),
                       "plan": cache.decode_plan_stats(),
                       "algorithmic_bytes_per_call": int(np.mean(dec_bytes)),
                       "gbs": round(dgbs, 1), "frac": round(dgbs / peak, 4),
                       "unique_page_bytes_per_call": int(np.mean(dec_ubytes)),
                       "gbs_unique_pages": round(ugbs, 1), "frac_unique_pages": round(ugbs / peak, 4)},
            "reposition": {"ms": round(float(np.mean(rep_ms)), 3), "moved_tokens": moved,
                           "algorithmic_bytes": rep_bytes, "gbs": round(rgbs, 1),
                           "frac": round(rgbs / peak, 4)},
            "peak": peak, "peak_source": "measured" if "hbm_gbs" in peaks else "fallback",
        }
        print(json.dumps(line), flush=True)

    for name in args.config_kernels.split(","):
        if name == "gptoss120b":
            sh, seed, B, N = traces.GPTOSS120B, traces.seed_for(2), 4, 131072
            trajs = traces.gptoss_batch(seed, batch=B, n_total=N)
            mp = B * (N // 16) + B * (N // 16 // 4) + 512
            cache = Cache(sh.layers, sh.hq, sh.hkv, sh.head_dim, sh.page_size, sh.dtype, mp,
                          2 * B + 2, N + 64, sh.rope_theta)
            bases = [cache.seq_create() for _ in range(B)]
            for b, s in enumerate(bases):
                append(cache, s, b + 1, 0, N, sh, seed)
            measure(name, cache, sh, bases, [t.drop_ranges for t in trajs], seed,
                    f"{sh.name}-shaped: {B} x {N} tokens, ~80% dropped, 1 reposition")
        elif name == "branching":
            # 32 of the workload's 64 branches: each fork's reposition takes
            # fresh 2 MB pages, and 64 prepared branches plus 64 timed forks
            # would not fit the pool next to the other state
            sh, seed, P, NB = traces.LLAMA8B, traces.seed_for(3), 16384, 32
            segs, branches = traces.branching(seed, n_branches=64, prefix_len=P)
            mp = P // 16 + 2 * NB * (P // 16 + 8) + 512
            cache = Cache(sh.layers, sh.hq, sh.hkv, sh.head_dim, sh.page_size, sh.dtype, mp,
                          2 * NB + 4, P + 64, sh.rope_theta)
            root = cache.seq_create()
            append(cache, root, 1, 0, P, sh, seed)
            # a branch's prepared state is its operations before its last
            # reposition; the timed call is that last reposition, batched
            kids = []
            for br in branches[:NB]:
                k = cache.seq_fork(root)
                last = max(i for i, op in enumerate(br.ops) if op[0] == "repos")
                for op in br.ops[:last]:
                    if op[0] == "drop":
                        cache.drop(k, op[1])
                    else:
                        cache.reposition([k])
                kids.append(k)
            for sharing in (0, 1):
                measure(name, cache, sh, kids, [None] * NB, seed,
                        f"{sh.name}-shaped: one {P}-token prefix forked into {NB} of the 64 "
                        "branches (1-6 drop / reposition operations each); every branch's last "
                        "reposition batched and timed, then batched decode over the branches",
                        sharing=sharing)
        elif name == "branching_fork":
            # the same workload at the moment of the fork, before any branch
            # operation: all 64 branches hold every page of the prefix
            sh, seed, P, NB = traces.LLAMA8B, traces.seed_for(3), 16384, 64
            mp = P // 16 + 2 * NB + 512
            cache = Cache(sh.layers, sh.hq, sh.hkv, sh.head_dim, sh.page_size, sh.dtype, mp,
                          2 * NB + 4, P + 64, sh.rope_theta)
            root = cache.seq_create()
            append(cache, root, 1, 0, P, sh, seed)
            kids = [cache.seq_fork(root) for _ in range(NB)]
            for sharing in (0, 1):
                measure(name, cache, sh, kids, [None] * NB, seed,
                        f"{sh.name}-shaped: one {P}-token prefix forked into {NB} branches, "
                        "decoded before any branch operation (every prefix page shared by "
                        "all branches; the reposition is a no-op)", sharing=sharing)
        elif name == "llama70b":
            # turns 0..13 as scheduled, then turn 14's tool response; the timed
            # operation is turn 14's drop of the oldest tool spans + reposition
            # (every third turn drops once more than 16384 tokens are active)
            sh, seed, B, TT = traces.LLAMA70B, traces.seed_for(4), 64, 14
            turns = traces.steady_state(seed, n_seqs=B, n_turns=TT + 1, decode_per_turn=64,
                                        active_cap=16384)
            longest = max(1024 + sum(t.tool_len + 64 for t in ts) for ts in turns)
            mp = B * (-(-longest // 16) + 8) * 2 + 1024
            cache = Cache(sh.layers, sh.hq, sh.hkv, sh.head_dim, sh.page_size, sh.dtype, mp,
                          2 * B + 2, longest + 64, sh.rope_theta, phys_layers=16)
            bases, drops = [], []
            for b, ts in enumerate(turns):
                s = cache.seq_create()
                t0 = 0
                append(cache, s, b + 1, t0, 1024, sh, seed)
                t0 += 1024
                for k, tn in enumerate(ts[:TT]):
                    append(cache, s, b + 1, t0, tn.tool_len + 64, sh, seed)
                    t0 += tn.tool_len + 64
                    if tn.drop_ranges:
                        cache.drop(s, tn.drop_ranges)
                    if tn.repos:
                        cache.reposition([s])
                append(cache, s, b + 1, t0, ts[TT].tool_len + 64, sh, seed)
                bases.append(s)
                drops.append(ts[TT].drop_ranges or None)
            measure(name, cache, sh, bases, drops, seed,
                    f"{sh.name}-shaped steady state: {B} sequences at turn {TT + 1} (80 logical "
                    "layers on 16 slabs): the turn's drop of the oldest tool spans and one "
                    "batched reposition timed, then decode on all 80 layers")
        else:
            raise SystemExit(f"unknown workload {name}")
        cache.close()
        del cache
        torch.cuda.empty_cache()



# ---------------------------------------------------------------------------
# GPU arm (headline line)
# ---------------------------------------------------------------------------

def decode_traffic(name, algorithmic):
    """DRAM bytes per decode launch, from the committed ncu summary of the
    decode kernel (``profiles/<name>``), if that summary was taken on the
    kernel's source as it is now: the measured traffic / algorithmic ratio of
    the captured case times this call's algorithmic bytes.  None otherwise."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", name)
    src = os.path.join(ROOT, "agent_kv_cache_gb300", "csrc", "akv_decode_mma.cu")
    try:
        text = open(prof).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None, None
    fields = dict(l.split(":", 1) for l in text.splitlines()
                  if l.startswith(("kernel_source_sha256:", "traffic_bytes_per_launch:",
                                   "algorithmic_bytes_per_launch:")))
    if fields.get("kernel_source_sha256", "").strip() != digest:
        return None, None
    try:
        ratio = (int(fields["traffic_bytes_per_launch"].strip())
                 / int(fields["algorithmic_bytes_per_launch"].strip()))
    except (KeyError, ValueError):
        return None, None
    return int(ratio * algorithmic), (f"ncu dram__bytes_read.sum + dram__bytes_write.sum of the "
                                      f"captured case in profiles/{name} (kernel source hash "
                                      f"matches), scaled by this call's algorithmic bytes "
                                      f"(traffic / algorithmic = {ratio:.4f})")


def gpu_arm(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    barrier = (lambda: dist.barrier()) if dist else (lambda: None)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        ot = OracleTurns()
        by, secs = ot.turn(STEADY_FIRST)
        ot.close()
        cpu = {"value": round(by / secs / 1e9, 4), "unit": "GB/s",
               "cores": os.cpu_count(), "workers": len(ot.conns), "kind": "oracle",
               "sample": ot.sample() + f"; turn {STEADY_FIRST + 1}; {secs:.1f} s"}

    K = args.steps
    e2e_turns = 0 if args.no_e2e else K + 1
    b = Steady(rank, args.warmup, K, e2e_turns)
    for k in range(b.first, STEADY_FIRST):
        b.turn(k)
    torch.cuda.synchronize()
    w = b.cache.sync_errors()
    assert w == 0, f"device error word 0x{w:x} after the warm-up turns"

    evs = [b.events() for _ in range(K)]
    start, stop = events(torch, 1)[0]
    n0 = b.cache.kernel_launches()
    barrier()
    torch.cuda.synchronize()
    with Clocks(gpu_id(local)) as clk:
        start.record(b.stream)
        host_dev = time.perf_counter()
        for i in range(K):
            if args.nvtx:
                torch.cuda.nvtx.range_push("turn")
            b.turn(STEADY_FIRST + i, ev=evs[i])
            if args.nvtx:
                torch.cuda.nvtx.range_pop()
        host_dev = (time.perf_counter() - host_dev) / K
        stop.record(b.stream)
        torch.cuda.synchronize()
    barrier()
    launches = (b.cache.kernel_launches() - n0) // K
    ms = reduce_max(start.elapsed_time(stop) / K, dist, "cuda")
    assert b.cache.sync_errors() == 0

    sh = b.sh
    L = sh.layers
    timed = [b.acct[STEADY_FIRST + i] for i in range(K)]
    total = sum(a["total"] for a in timed)
    peak, peak_src = hbm_peak()
    call_b = np.array([a["calls"] for a in timed])                        # [K][DEC]
    dec_ms = np.array([[s.elapsed_time(e) / L for s, e in ev["dec"]] for ev in evs])
    achieved = float(np.sum(call_b) / np.sum(dec_ms * 1e-3) / 1e9)
    dec_sec = float(np.sum(dec_ms)) * L * 1e-3
    rep = [(ev["repos"][0].elapsed_time(ev["repos"][1]), a["repos_bytes"], a["repos_moved"])
           for ev, a in zip(evs, timed) if a["repos"]]
    drp = [ev["drop"][0].elapsed_time(ev["drop"][1]) for ev, a in zip(evs, timed) if a["dropped"]]
    app = [(ev["append"][0].elapsed_time(ev["append"][1]), 2 * L * a["tool"] * kvt_of(sh))
           for ev, a in zip(evs, timed)]
    # time between one decode step's last call and the next step's first
    # (the next token's append, and in the end-to-end run any wait for inputs)
    gap_dev = float(np.mean([sum(ev["dec"][t][1].elapsed_time(ev["dec"][t + 1][0])
                                 for t in range(STEADY_DECODE - 1)) for ev in evs]))
    value = world * total / (ms * K * 1e-3) / 1e9

    # one decode call at a time (after an unrelated kernel streaming 1.5 GB),
    # on the state after the timed turns
    act = [b.cache.info(s) for s in b.seqs]
    iso_bytes = decode_call_bytes(sh, [i["n_active"] for i in act],
                                  [i["n_active_pages"] for i in act])
    iso_us = isolated_decode(torch, b.cache, range(L), b.q[0], b.seqs, b.out)
    traffic, traffic_src = decode_traffic("decode_mma_llama70b.md", int(np.mean(call_b)))

    e2e = None
    if not args.no_e2e:
        host = b.host_buffers()
        k0 = STEADY_FIRST + K
        b.turn(k0, host=host)
        torch.cuda.synchronize()
        barrier()
        s2, e2 = events(torch, 1)[0]
        evs2 = [b.events() for _ in range(K)]
        s2.record(b.stream)
        host_s = time.perf_counter()
        for i in range(K):
            b.turn(k0 + 1 + i, ev=evs2[i], host=host)
        host_s = (time.perf_counter() - host_s) / K
        e2.record(b.stream)
        torch.cuda.synchronize()
        barrier()
        assert b.cache.sync_errors() == 0
        ms2 = reduce_max(s2.elapsed_time(e2) / K, dist, "cuda")
        tot2 = sum(b.acct[k0 + 1 + i]["total"] for i in range(K))
        dec2 = np.array([[s_.elapsed_time(e_) / L for s_, e_ in ev["dec"]] for ev in evs2])
        gap2 = float(np.mean([sum(ev["dec"][t][1].elapsed_time(ev["dec"][t + 1][0])
                                  for t in range(STEADY_DECODE - 1)) for ev in evs2]))
        app2 = [ev["append"][0].elapsed_time(ev["append"][1]) for ev in evs2]
        e2e = {"value": round(world * tot2 / (ms2 * K * 1e-3) / 1e9, 1), "unit": "GB/s",
               "h2d_bytes_per_step": int(np.mean([b.h2d_bytes(k0 + 1 + i) for i in range(K)])),
               "d2h_bytes_per_step": int(host["out"].numel() * 4),
               "ms_per_step": round(ms2, 3),
               "turns": f"{k0 + 2}..{k0 + 1 + K}",
               "decode_avg_call_us": round(float(np.mean(dec2)) * 1e3, 2),
               "decode_ms_per_turn": round(float(np.sum(dec2)) * L / K, 1),
               "decode_call_us_per_8_steps": [round(float(np.mean(dec2[:, j:j + 8])) * 1e3, 1)
                                              for j in range(0, STEADY_DECODE, 8)],
               "append_ms_per_turn": round(float(np.mean(app2)), 3),
               "between_decode_steps_ms_per_turn": round(gap2, 2),
               "host_enqueue_ms_per_turn": round(host_s * 1e3, 1),
               "appends_to_first_decode_ms": round(float(np.mean(
                   [ev["append"][1].elapsed_time(ev["dec"][0][0]) for ev in evs2])), 2),
               "last_decode_to_turn_end_ms": round(float(np.mean(
                   [ev["dec"][-1][1].elapsed_time(ev["repos"][1]) for ev in evs2])), 2),
               "tool_prefetch_ms": round(float(np.mean(
                   [b._tool_ev[k][0].elapsed_time(b._tool_ev[k][1])
                    for k in range(k0 + 2, k0 + 2 + K) if k in b._tool_ev])), 2),
               "tool_prefetch_start_after_first_decode_ms": round(float(np.mean(
                   [ev["dec"][0][0].elapsed_time(b._tool_ev[k0 + 2 + i][0])
                    for i, ev in enumerate(evs2) if k0 + 2 + i in b._tool_ev])), 2),
               "tool_prefetch_host_ms": round(float(np.mean(
                   [b._tool_host_s[k] * 1e3 for k in range(k0 + 2, k0 + 2 + K)
                    if k in b._tool_host_s])), 2),
               "turn_start_to_first_append_ms": round(float(np.mean(
                   [e_prev["repos"][1].elapsed_time(e_cur["append"][0])
                    for e_prev, e_cur in zip(evs2[:-1], evs2[1:])])), 2) if K > 1 else None,
               "what": "public C-ABI calls (append / decode / drop / reposition) with every "
                       "turn's inputs copied from pinned host memory on copy streams: its "
                       "tool responses' raw K/V during the previous turn's decode (from its "
                       "eighth decode step on, one device "
                       "slot per group of 16 sequences; each group's append waits for its "
                       "copy), its decode steps' queries and new-token K/V while its decode "
                       "runs (each step waits for its own); every decode step's last-layer "
                       "attention output copied back on a third stream"}
        del host
    b.close()

    blocks = None
    if world == 1 and not args.no_blocks:
        blocks = run_blocks(rank, ["llama8b", "gptoss120b", "branching"], min(K, 5))

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded SplitMix64 K/V/q, seeded agent turn schedule)",
            "config": {
                "workload": steady_workload(K),
                "global_batch": world * STEADY_SEQS, "seq_len": "<= 16384 active after each drop",
                "decode_steps_per_turn": STEADY_DECODE,
                "parallelism": f"replicas x{world} (sequences partitioned, no collective)",
                "l2": "inputs larger than L2 (each decode call reads 4-5 GB); no flush",
                "bytes_per_step": int(total / K)},
            "decode_tok_s": round(world * STEADY_SEQS * STEADY_DECODE * K / dec_sec, 1),
            "roofline": {"kernel": "k_decode_mma (one launch per decode-attention call, split "
                                   "merge fused; per-call time = span of a decode step's "
                                   f"{L} back-to-back calls / {L})",
                         "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "peak_source": peak_src, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "traffic_source": traffic_src,
                         "avg_call_us": round(float(np.mean(dec_ms)) * 1e3, 2),
                         "algorithmic_bytes_per_call": int(np.mean(call_b)),
                         "share_of_step": round(dec_sec / K / (ms * 1e-3), 4)},
            "decode_isolated": {"what": "one decode-attention call at a time, each after an "
                                        "unrelated kernel streaming 1.5 GB",
                                "avg_call_us": round(iso_us, 2),
                                "algorithmic_bytes_per_call": int(iso_bytes),
                                "gbs": round(iso_bytes / (iso_us * 1e-6) / 1e9, 1),
                                "frac": round(iso_bytes / (iso_us * 1e-6) / 1e9 / peak, 4)},
            "reposition": {"kernel": "k_compact + k_gather", "turns": len(rep),
                           "ms": round(float(np.mean([r[0] for r in rep])), 3) if rep else None,
                           "moved_tokens": int(np.mean([r[2] for r in rep])) if rep else 0,
                           "algorithmic_bytes": int(np.mean([r[1] for r in rep])) if rep else 0,
                           "gbs": round(sum(r[1] for r in rep) / (sum(r[0] for r in rep) * 1e-3)
                                        / 1e9, 1) if rep else None,
                           "frac": round(sum(r[1] for r in rep) / (sum(r[0] for r in rep) * 1e-3)
                                         / 1e9 / peak, 4) if rep else None},
            "between_decode_steps_ms_per_turn": round(gap_dev, 2),
            "host_enqueue_ms_per_turn": round(host_dev * 1e3, 1),
            "drop": {"kernel": "k_drop", "us_per_turn": round(float(np.mean(drp)) * 1e3, 1)
                     if drp else None, "calls_per_turn": STEADY_SEQS},
            "append": {"kernel": "k_append (tool responses, 80 layers)",
                       "ms": round(float(np.mean([a[0] for a in app])), 3),
                       "gbs": round(sum(a[1] for a in app) / (sum(a[0] for a in app) * 1e-3)
                                    / 1e9, 1)},
            "gpu_launches": int(launches),
            "clocks": clk.summary(),
        }
        if cpu:
            line["cpu_baseline"] = cpu
        if e2e:
            line["e2e"] = e2e
        if blocks:
            line["configs"] = blocks
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def steady_workload(K):
    sh = STEADY
    return (f"{sh.name}-shaped steady state: {sh.layers} layers ({STEADY_SLABS} physical slabs), "
            f"{sh.hq}/{sh.hkv} heads, head_dim {sh.head_dim}, {sh.dtype}, rope theta "
            f"{sh.rope_theta:g}, page {sh.page_size}; {STEADY_SEQS} sequences, {STEADY_SYS}-token "
            "system prompt, per turn one tool response (lognormal median 1000, 200..4000 tokens) "
            f"and {STEADY_DECODE} decode tokens; every 3 turns the oldest tool responses dropped "
            f"to <= {STEADY_CAP} active and a reposition; one step = one turn (turns "
            f"{STEADY_FIRST + 1}..{STEADY_FIRST + K} of the steady-state window)")


def only_arm(args):
    """One workload as its own line (for focused measurement or a profiler's
    small case): the 8B / 120B trace or the branching block."""
    import torch
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    name = args.only
    if name == "branching":
        b = BranchBench(0, layers=args.layers)
    else:
        spec = {"llama8b": TRACE8B, "gptoss120b": TRACE120B, "llama70b": TRACE70B}[name]
        b = TraceBench(spec, 0, batch=args.batch, layers=args.layers, decode=args.decode_steps)
    res = b.run(args.warmup, args.steps)
    line = {"metric": METRIC, "value": res["gbs"], "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": b.workload()}, "block": res}
    if args.batch or args.layers or args.decode_steps:
        line["config"]["profiling_case"] = "reduced shape for a profiler capture"
    print(json.dumps(line), flush=True)
    b.close()


def reference_arm(args):
    """The oracle as the reference arm: one process per sampled (sequence,
    layer) of the steady-state workload; a step is one turn of that sample."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    W, K = min(args.warmup, STEADY_FIRST), args.steps
    ot = OracleTurns(start=STEADY_FIRST - W, n_turns=max(STEADY_TURNS, STEADY_FIRST + K))
    for k in range(STEADY_FIRST - W, STEADY_FIRST):
        ot.turn(k)
    res = [ot.turn(STEADY_FIRST + i) for i in range(K)]
    ot.close()
    by, secs = sum(r[0] for r in res), sum(r[1] for r in res)
    value = by / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": K, "warmup": args.warmup,
        "ms_per_step": round(secs / K * 1e3, 1), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": steady_workload(K)},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": os.cpu_count(),
                         "workers": len(ot.conns), "kind": "oracle", "sample": ot.sample()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["akv", "reference"], default="akv")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-blocks", action="store_true",
                    help="headline only (no 8B / 120B / branching blocks)")
    ap.add_argument("--only", choices=["llama8b", "gptoss120b", "branching", "llama70b"],
                    default=None, help="one block's workload (or the 70B-shaped profiler "
                                       "case) as its own line")
    ap.add_argument("--nvtx", action="store_true",
                    help="wrap each timed turn in an NVTX range 'turn' (profiler launch lists)")
    ap.add_argument("--restore", action="store_true",
                    help="time segment-batch restore attention instead (its own line)")
    ap.add_argument("--restore-cuda-cores", action="store_true")
    ap.add_argument("--config-kernels", default=None,
                    help="comma list of gptoss120b, branching, branching_fork, llama70b: decode and "
                         "reposition bandwidth on those workloads (one line each)")
    ap.add_argument("--prefix", action="store_true",
                    help="time prefix matching / forks / eviction instead (its own line)")
    # smaller cases of --only llama8b / gptoss120b for profiler captures; a
    # line printed with any of these is marked "profiling case"
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--decode-steps", type=int, default=None)
    args = ap.parse_args()
    if args.config_kernels:
        kernels_arm(args)
    elif args.prefix:
        prefix_arm(args)
    elif args.restore or args.restore_cuda_cores:
        restore_arm(args)
    elif args.only:
        only_arm(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        if args.warmup < 3:
            ap.error("the headline line takes at least 3 warm-up steps")
        gpu_arm(args)


if __name__ == "__main__":
    main()
