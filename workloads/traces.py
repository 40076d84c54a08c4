"""Shapes of synthetic agent trajectories.

The pages measure on replayed agent runs over public benchmarks (coding,
browsing and research tasks).  None of that data is used here; these seeded
generators stand in for it with the structure the pages describe: a system
prompt, then alternating assistant segments and long tool responses, and a
rolling-drop policy that removes old tool responses while keeping reasoning
("Cache Engineering for Agents" review, 3.2 Design Motivation: rolling drop of
old tool responses; Figure 14 for active-context growth).

Every function returns plain Python data (lists of half-open logical token
ranges and operation schedules).  Nothing here computes any part of the
method.
"""
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Shape:
    """Attention shape of a model family (no weights are involved)."""
    name: str
    layers: int
    hq: int
    hkv: int
    head_dim: int
    dtype: str          # pool dtype: 'bf16' or 'fp32'
    rope_theta: float
    page_size: int = 16


TINY = Shape("tiny", 1, 8, 2, 64, "fp32", 1.0e4)
LLAMA8B = Shape("llama3.1-8b", 32, 32, 8, 128, "bf16", 5.0e5)
GPTOSS120B = Shape("gpt-oss-120b", 36, 64, 8, 64, "bf16", 1.5e5)
LLAMA70B = Shape("llama-70b", 80, 64, 8, 128, "bf16", 5.0e5)

MASTER_SEED = 20261202


def seed_for(workload_id):
    return MASTER_SEED + int(workload_id)


# --------------------------------------------------------------------------
# trajectories
# --------------------------------------------------------------------------

def _draw(rng, n, asst_range, tool_median, tool_sigma, tool_clip):
    a = rng.integers(asst_range[0], asst_range[1] + 1, size=n)
    z = rng.standard_normal(n)
    t = np.rint(tool_median * np.exp(tool_sigma * z))
    t = np.clip(t, tool_clip[0], tool_clip[1]).astype(np.int64)
    return a.astype(np.int64), t


def _build(n_total, sys_len, a, t, scale):
    segs = [("system", 0, min(sys_len, n_total))]
    pos = segs[0][2]
    k = 0
    while pos < n_total:
        la = min(max(1, int(round(float(a[k]) * scale))), n_total - pos)
        segs.append(("assistant", pos, la))
        pos += la
        if pos >= n_total:
            break
        lt = min(int(t[k]), n_total - pos)
        segs.append(("tool", pos, lt))
        pos += lt
        k += 1
    return segs


def agent_trajectory(rng, n_total, sys_len=1024, asst_range=(200, 900),
                     tool_median=1500, tool_sigma=0.75, tool_clip=(500, 8000),
                     scale=1.0, n_draw=4096):
    """Segments ``[(kind, start, length)]`` covering logical tokens [0, n_total)."""
    a, t = _draw(rng, n_draw, asst_range, tool_median, tool_sigma, tool_clip)
    return _build(n_total, sys_len, a, t, scale)


def _tool_drop(segs, keep_last):
    tools = [(s, s + n) for kind, s, n in segs if kind == "tool"]
    cut = max(0, len(tools) - keep_last)
    return tools[:cut]


@dataclass
class RollingDrop:
    n_total: int
    segments: list
    drop_ranges: list           # half-open logical ranges removed by the policy
    dropped_fraction: float
    scale: float
    keep_last: int


def rolling_drop(seed, n_total, tool_median, tool_clip, frac_range,
                 keep_last_choices=(3,), sys_len=1024, asst_range=(200, 900),
                 tool_sigma=0.75):
    """Trajectory whose rolling drop removes a fraction of tokens in ``frac_range``.

    All tool spans but the last ``keep_last`` are dropped.  The assistant
    segment lengths are scaled (and ``keep_last`` chosen among the choices)
    so that dropped/N falls in ``frac_range``; among the feasible choices the
    one closest to the middle of the range wins, then the smallest scale
    change.  If no scale works for a draw (the kept tail of three tool spans
    moves the fraction in large steps), the lengths are drawn again from the
    next sub-stream ``[seed, attempt]``.
    """
    target = 0.5 * (frac_range[0] + frac_range[1])
    for attempt in range(256):
        rng = np.random.default_rng([seed, attempt])
        a, t = _draw(rng, 4096, asst_range, tool_median, tool_sigma, tool_clip)
        best = None
        for keep_last in keep_last_choices:
            for scale in np.geomspace(0.25, 4.0, 161):
                segs = _build(n_total, sys_len, a, t, float(scale))
                drops = _tool_drop(segs, keep_last)
                frac = sum(e - b for b, e in drops) / n_total
                if not (frac_range[0] <= frac <= frac_range[1]):
                    continue
                score = (round(abs(frac - target), 3), abs(np.log(scale)))
                if best is None or score < best[0]:
                    best = (score, RollingDrop(n_total, segs, drops, frac,
                                               float(scale), keep_last))
        if best is not None:
            return best[1]
    raise RuntimeError("no trajectory reaches the dropped fraction")


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

def tiny_spans(seed, n_total=512, n_spans=3, lo=40, hi=80):
    """Three non-overlapping spans of uniform length [lo, hi] in [0, n_total)."""
    rng = np.random.default_rng(seed)
    while True:
        spans = []
        for _ in range(n_spans):
            ln = int(rng.integers(lo, hi + 1))
            b = int(rng.integers(0, n_total - ln + 1))
            spans.append((b, b + ln))
        spans.sort()
        if all(spans[i][1] <= spans[i + 1][0] for i in range(n_spans - 1)):
            return spans


def llama8b_batch(seed, batch=16, n_total=32768):
    """Per-sequence rolling-drop trajectories (~60% dropped, last 3 tools kept)."""
    return [rolling_drop(seed * 1000 + b, n_total, 1500, (500, 8000),
                         (0.57, 0.63), keep_last_choices=(3,))
            for b in range(batch)]


def gptoss_batch(seed, batch=4, n_total=131072):
    """Per-sequence trajectories with ~80% dropped (tool median 3000)."""
    return [rolling_drop(seed * 1000 + b, n_total, 3000, (1000, 16000),
                         (0.77, 0.83), keep_last_choices=tuple(range(1, 31)))
            for b in range(batch)]


@dataclass
class Branch:
    ops: list     # [("drop", [(b, e), ...]) | ("repos",)]


def branching(seed, n_branches=64, prefix_len=16384):
    """One shared prefix and per-branch drop/reposition sequences.

    Each branch applies 1..6 operations; each is a drop (probability 2/3;
    half of the drops take one of the prefix's tool spans, half a uniform span
    of 64..2048 tokens) or a reposition; a branch whose draw has no
    reposition gets its last operation replaced by one.
    """
    rng = np.random.default_rng(seed)
    segs = agent_trajectory(rng, prefix_len)
    tools = [(s, s + n) for kind, s, n in segs if kind == "tool"]
    branches = []
    for b in range(n_branches):
        r = np.random.default_rng([seed, b])
        n_ops = int(r.integers(1, 7))
        ops = []
        for _ in range(n_ops):
            if r.random() < 2.0 / 3.0:
                if tools and r.random() < 0.5:
                    span = tools[int(r.integers(0, len(tools)))]
                else:
                    ln = int(r.integers(64, 2049))
                    st = int(r.integers(0, prefix_len - ln + 1))
                    span = (st, st + ln)
                ops.append(("drop", [span]))
            else:
                ops.append(("repos",))
        if not any(o[0] == "repos" for o in ops):
            ops[-1] = ("repos",)
        branches.append(Branch(ops))
    return segs, branches


@dataclass
class Turn:
    tool_len: int
    drop_ranges: list    # applied after the turn's decode steps (may be empty)
    repos: bool


def steady_state(seed, n_seqs=64, n_turns=100, sys_len=1024, decode_per_turn=64,
                 tool_median=1000, tool_clip=(200, 4000), tool_sigma=0.75,
                 every=3, active_cap=16384):
    """Per-sequence turn schedules of the long-running agent workload.

    A turn appends one tool response (lognormal length) and then decodes
    ``decode_per_turn`` tokens.  After every ``every``-th turn the oldest
    tool responses still active are dropped until the active count is at
    most ``active_cap`` (or none are left), then the sequence is
    repositioned.
    """
    out = []
    for s in range(n_seqs):
        rng = np.random.default_rng([seed, s])
        z = rng.standard_normal(n_turns)
        lens = np.clip(np.rint(tool_median * np.exp(tool_sigma * z)),
                       tool_clip[0], tool_clip[1]).astype(np.int64)
        pos = sys_len
        active = sys_len
        live_tools = []
        turns = []
        for k in range(n_turns):
            tl = int(lens[k])
            live_tools.append((pos, pos + tl))
            pos += tl + decode_per_turn
            active += tl + decode_per_turn
            drops = []
            repos = False
            if (k + 1) % every == 0:
                while active > active_cap and live_tools:
                    b, e = live_tools.pop(0)
                    drops.append((b, e))
                    active -= e - b
                repos = True
            turns.append(Turn(tl, drops, repos))
        out.append(turns)
    return out


def restore_program(seed, n_turns=30, sys_len=1024, decode_per_turn=64, active_cap=16384):
    """Operation program of one long-running agent sequence (the steady-state
    schedule above, one sequence) for restore attention: the system prompt,
    then per turn the tool response and its decoded tokens as one append, the
    turn's drops of the oldest tool responses and its reposition."""
    turns = steady_state(seed, n_seqs=1, n_turns=n_turns, sys_len=sys_len,
                         decode_per_turn=decode_per_turn, active_cap=active_cap)[0]
    prog = [("append", sys_len)]
    for t in turns:
        prog.append(("append", t.tool_len + decode_per_turn))
        if t.drop_ranges:
            prog.append(("drop", list(t.drop_ranges)))
        if t.repos:
            prog.append(("repos",))
    return prog


def turn_programs(seed, n_turns=30, sys_len=1024, decode_per_turn=64, active_cap=16384):
    """The same long-running sequence as ``restore_program``, cut at the end
    of every turn: element k is the list of operations of turn k (turn 0
    starts with the system prompt).  Concatenating elements 0..k gives the
    sequence's history after turn k."""
    turns = steady_state(seed, n_seqs=1, n_turns=n_turns, sys_len=sys_len,
                         decode_per_turn=decode_per_turn, active_cap=active_cap)[0]
    out = []
    for k, t in enumerate(turns):
        ops = [("append", sys_len)] if k == 0 else []
        ops.append(("append", t.tool_len + decode_per_turn))
        if t.drop_ranges:
            ops.append(("drop", list(t.drop_ranges)))
        if t.repos:
            ops.append(("repos",))
        out.append(ops)
    return out


def token_ids(seed, n, vocab=128256):
    """Seeded synthetic token ids (uniform over a Llama-3-sized vocabulary)."""
    return np.random.default_rng([seed, 77]).integers(0, vocab, size=n).astype(np.int32)
