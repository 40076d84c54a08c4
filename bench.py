#!/usr/bin/env python3
"""Benchmark of the active-KV hot path: drop + reposition + decode attention.

Workload (Llama-3.1-8B-shaped agent trace): 32 layers, 32 query / 8 KV heads,
head_dim 128, bf16 K/V, RoPE theta 5e5, page 16; 16 sequences of 32768
logical tokens whose tool-response spans (lognormal, median 1500, clipped to
500..8000) are all dropped but the last 3 (~60% of the tokens), then one
reposition and 128 decode steps (each appends one token per sequence and runs
decode attention on all 32 layers).  Inputs are seeded and synthetic.

One timed step = fork the 16 prepared sequences (pages shared), drop, one
batched reposition, 128 x (append + 32 x decode attention), free the forks.
Every step redoes the same work from the same prepared cache.

``value`` is algorithmic bytes per second over the whole step: the K/V of
relocated survivors read and written by the reposition, the active K/V read
by every decode-attention call (plus q, out and page metadata), and the K/V
written by the appends.  ``--impl reference`` times the CPU oracle instead.
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
SHAPE = traces.LLAMA8B
BATCH = 16
N_TOKENS = 32768
DECODE_STEPS = 128
SEED = traces.seed_for(1)
BYTES_EL = 2
CHUNK = 4096


def workload_name():
    return (f"{SHAPE.name}-shaped agent trace: {SHAPE.layers} layers, {SHAPE.hq}/{SHAPE.hkv} heads, "
            f"head_dim {SHAPE.head_dim}, {SHAPE.dtype}, rope theta {SHAPE.rope_theta:g}, page "
            f"{SHAPE.page_size}; batch {BATCH} x {N_TOKENS} logical tokens, tool spans dropped "
            f"(all but last 3, ~60%), 1 reposition, {DECODE_STEPS} decode steps")


def trajectories():
    return traces.llama8b_batch(SEED, batch=16, n_total=N_TOKENS)[:BATCH]


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def kv_bytes_per_token():
    return 2 * SHAPE.hkv * SHAPE.head_dim * BYTES_EL      # K + V, one layer


def repos_moved(traj):
    """Survivors a reposition relocates (those before the first drop stay)."""
    first = min(b for b, _ in traj.drop_ranges) if traj.drop_ranges else N_TOKENS
    r = N_TOKENS - sum(e - b for b, e in traj.drop_ranges)
    kept = (first // SHAPE.page_size) * SHAPE.page_size
    return r, r - kept


def step_bytes(trajs):
    L = SHAPE.layers
    kvt = kv_bytes_per_token()
    rs = [repos_moved(t) for t in trajs]
    repos = sum(2 * L * moved * kvt for _, moved in rs)          # read + write
    decode_calls = []
    for t in range(DECODE_STEPS):
        active = sum(r + t + 1 for r, _ in rs)
        pages = sum(-(-(r + t + 1) // SHAPE.page_size) for r, _ in rs)
        qo = BATCH * SHAPE.hq * SHAPE.head_dim * (BYTES_EL + 4)
        meta = pages * (4 + 4 + SHAPE.page_size // 8)
        decode_calls.append(active * kvt + qo + meta)
    decode = L * sum(decode_calls)
    append = DECODE_STEPS * BATCH * L * kvt * 2                  # read raw + write
    drop = sum(N_TOKENS // 8 + 10 * (N_TOKENS // SHAPE.page_size) for _ in trajs)
    return dict(repos=repos, decode=decode, append=append, drop=drop,
                decode_per_call=decode_calls, total=repos + decode + append + drop)


def decode_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if that
    summary was taken on the decode kernel as it is now (else None)."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "decode_mma_llama8b.md")
    src = os.path.join(ROOT, "agent_kv_cache_gb300", "csrc", "akv_decode_mma.cu")
    try:
        text = open(prof).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    fields = dict(l.split(":", 1) for l in text.splitlines()
                  if l.startswith(("kernel_source_sha256:", "traffic_bytes_per_launch:")))
    if fields.get("kernel_source_sha256", "").strip() != digest:
        return None
    return int(fields["traffic_bytes_per_launch"].strip())


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


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------

def _oracle_unit(args):
    """Drop + reposition + decode of one (sequence, layer) of the workload."""
    os.environ["OMP_NUM_THREADS"] = "1"
    seq, layer, n_decode, traj_ranges = args
    from oracle.akv_oracle import OracleCache
    o = OracleCache(SHAPE.hq, SHAPE.hkv, SHAPE.head_dim, SHAPE.rope_theta, SHAPE.dtype,
                    layers=[layer], page_size=SHAPE.page_size)
    s = o.create()
    w = synth.width_for(SHAPE.dtype)
    k = synth.kv_tokens(SEED, seq + 1, synth.KIND_K, [layer], 0, N_TOKENS, SHAPE.hkv, SHAPE.head_dim, w)
    v = synth.kv_tokens(SEED, seq + 1, synth.KIND_V, [layer], 0, N_TOKENS, SHAPE.hkv, SHAPE.head_dim, w)
    o.append(s, k, v)
    new_k = synth.kv_tokens(SEED, seq + 1, synth.KIND_K, [layer], N_TOKENS, n_decode, SHAPE.hkv,
                            SHAPE.head_dim, w)
    new_v = synth.kv_tokens(SEED, seq + 1, synth.KIND_V, [layer], N_TOKENS, n_decode, SHAPE.hkv,
                            SHAPE.head_dim, w)
    qs = [synth.query(SEED, seq + 1, layer, t, SHAPE.hq, SHAPE.head_dim, w) for t in range(n_decode)]
    t0 = time.perf_counter()
    o.drop(s, traj_ranges)
    o.reposition(s)
    for t in range(n_decode):
        o.append(s, new_k[:, t:t + 1], new_v[:, t:t + 1])
        o.attention(0, qs[t][None], [s])
    return time.perf_counter() - t0


def oracle_sample(trajs, n_seqs=2, n_layers=4, n_decode=16, workers=None):
    """Times the oracle on a bounded sample: n_seqs x n_layers (seq, layer) units."""
    units = [(b, l, n_decode, trajs[b].drop_ranges) for b in range(n_seqs) for l in range(n_layers)]
    workers = workers or min(len(units), os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(workers) as pool:
        times = pool.map(_oracle_unit, units)
    wall = time.perf_counter() - t0
    # algorithmic bytes of the sample, same accounting as the GPU path
    kvt = kv_bytes_per_token()
    total = 0
    for b in range(n_seqs):
        r, moved = repos_moved(trajs[b])
        per_layer = 2 * moved * kvt + sum((r + t + 1) * kvt + SHAPE.hq * SHAPE.head_dim * 6
                                          for t in range(n_decode)) + n_decode * kvt * 2
        total += n_layers * per_layer
    busy = max(times)
    return dict(bytes=total, seconds=busy, wall=wall, workers=workers, unit_times=times,
                sample=f"{n_seqs} sequences x {n_layers} layers of the workload (drop, reposition, "
                       f"{n_decode} decode steps each), one single-threaded process per "
                       f"(sequence, layer) unit, input generation excluded")


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


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class Bench:
    def __init__(self, rank):
        import torch
        from agent_kv_cache_gb300 import Cache, build
        from workloads import device as dev
        self.torch, self.dev = torch, dev
        build()
        dev.build()
        self.rank = rank
        self.trajs = trajectories()
        S = SHAPE.page_size
        rs = [repos_moved(t)[0] for t in self.trajs]
        base_pages = BATCH * (N_TOKENS // S)
        step_pages = sum(-(-(r + DECODE_STEPS) // S) + 2 for r in rs)
        self.max_pages = base_pages + step_pages + 256
        self.cache = Cache(SHAPE.layers, SHAPE.hq, SHAPE.hkv, SHAPE.head_dim, S, SHAPE.dtype,
                           self.max_pages, 2 * BATCH + 2, N_TOKENS + DECODE_STEPS + S,
                           SHAPE.rope_theta)
        self.stream = self.cache.stream
        self.tags = rank_tags(rank, BATCH)
        self.width = synth.width_for(SHAPE.dtype)
        self._build_base()
        self._make_inputs()
        self.bytes = step_bytes(self.trajs)

    def _build_base(self):
        torch, dev = self.torch, self.dev
        L, H, D = SHAPE.layers, SHAPE.hkv, SHAPE.head_dim
        kbuf = torch.empty((L, CHUNK, H, D), dtype=torch.bfloat16, device="cuda")
        vbuf = torch.empty_like(kbuf)
        self.base = []
        for b in range(BATCH):
            s = self.cache.seq_create()
            for t0 in range(0, N_TOKENS, CHUNK):
                n = min(CHUNK, N_TOKENS - t0)
                k1 = dev.kv_tokens(kbuf, SEED, self.tags[b], synth.KIND_K, range(L), t0, n, H, D, self.width)
                v1 = dev.kv_tokens(vbuf, SEED, self.tags[b], synth.KIND_V, range(L), t0, n, H, D, self.width)
                self.cache.append([s], [n], kbuf[:, :n].contiguous() if n < CHUNK else kbuf,
                                  vbuf[:, :n].contiguous() if n < CHUNK else vbuf)
                torch.cuda.synchronize()
                del k1, v1
            self.base.append(s)
        assert self.cache.sync_errors() == 0

    def _make_inputs(self):
        torch, dev = self.torch, self.dev
        L, Hq, H, D = SHAPE.layers, SHAPE.hq, SHAPE.hkv, SHAPE.head_dim
        self.q = torch.empty((DECODE_STEPS, L, BATCH, Hq, D), dtype=torch.bfloat16, device="cuda")
        self.knew = torch.empty((DECODE_STEPS, L, BATCH, H, D), dtype=torch.bfloat16, device="cuda")
        self.vnew = torch.empty_like(self.knew)
        keep = []
        for t in range(DECODE_STEPS):
            for l in range(L):
                keep.append(dev.queries(self.q[t, l], SEED, self.tags, l, t, Hq, D, self.width))
            keep.append(dev.kv_tokens_multi(self.knew[t], SEED, self.tags, synth.KIND_K, range(L),
                                            [N_TOKENS + t] * BATCH, 1, H, D, self.width))
            keep.append(dev.kv_tokens_multi(self.vnew[t], SEED, self.tags, synth.KIND_V, range(L),
                                            [N_TOKENS + t] * BATCH, 1, H, D, self.width))
        torch.cuda.synchronize()
        self.out = torch.empty((L, BATCH, Hq, D), dtype=torch.float32, device="cuda")

    def step(self, ev=None, host=None):
        """One pass of the hot path.  ``ev``: events for per-call timing;
        ``host``: pinned host inputs/outputs for the end-to-end variant."""
        c, torch = self.cache, self.torch
        L = SHAPE.layers
        if host is not None:
            # every decode step's inputs go up on a copy stream (each step has
            # its own device slot), overlapping the fork / drop / reposition
            # and the earlier decode steps; decode step t waits for its copy
            if not hasattr(self, "_h2d"):
                self._h2d = torch.cuda.Stream()
                self._ready = [torch.cuda.Event() for _ in range(DECODE_STEPS)]
            self._h2d.wait_stream(self.stream)   # the previous pass has read the slots
            with torch.cuda.stream(self._h2d):
                for t in range(DECODE_STEPS):
                    self.q[t].copy_(host["q"][t], non_blocking=True)
                    self.knew[t].copy_(host["k"][t], non_blocking=True)
                    self.vnew[t].copy_(host["v"][t], non_blocking=True)
                    self._ready[t].record(self._h2d)
        forks = [c.seq_fork(b) for b in self.base]
        for f, tr in zip(forks, self.trajs):
            c.drop(f, tr.drop_ranges)
        if ev is not None:
            ev["repos"][0].record(self.stream)
        c.reposition(forks)
        if ev is not None:
            ev["repos"][1].record(self.stream)
        for t in range(DECODE_STEPS):
            if host is not None:
                self.stream.wait_event(self._ready[t])
            c.append(forks, [1] * BATCH, self.knew[t], self.vnew[t])
            # one event pair around the step's L decode calls: an event between
            # two decode calls would end the overlap of their launches
            if ev is not None:
                ev["dec"][t][0].record(self.stream)
            for l in range(L):
                c.decode_attention(l, self.q[t, l], forks, self.out[l])
            if ev is not None:
                ev["dec"][t][1].record(self.stream)
            if host is not None:
                host["out"][t].copy_(self.out[L - 1], non_blocking=True)
        for f in forks:
            c.seq_free(f)

    def events(self):
        E = self.torch.cuda.Event
        return {"repos": (E(enable_timing=True), E(enable_timing=True)),
                "dec": [(E(enable_timing=True), E(enable_timing=True))
                        for _ in range(DECODE_STEPS)]}


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
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(trajectories())

    b = Bench(rank)
    barrier = (lambda: dist.barrier()) if dist else (lambda: None)
    for _ in range(args.warmup):
        b.step()
    torch.cuda.synchronize()
    w = b.cache.sync_errors()
    assert w == 0, f"device error word 0x{w:x} after the warm-up steps"

    evs = [b.events() for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        uuid = str(torch.cuda.get_device_properties(local).uuid)
        gid = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
    except Exception:
        gid = local
    n0 = b.cache.kernel_launches()
    barrier()
    torch.cuda.synchronize()
    with Clocks(gid) as clk:
        start.record(b.stream)
        for k in range(args.steps):
            b.step(ev=evs[k])
        stop.record(b.stream)
        torch.cuda.synchronize()
    barrier()
    launches = (b.cache.kernel_launches() - n0) // args.steps
    ms = reduce_max(start.elapsed_time(stop) / args.steps, dist, "cuda")
    assert b.cache.sync_errors() == 0

    by = b.bytes
    # per decode step: the span of its L back-to-back calls; per call: span / L
    dec_ms = [s.elapsed_time(e) / SHAPE.layers for ev in evs for s, e in ev["dec"]
              for _ in range(SHAPE.layers)]
    repos_ms = [ev["repos"][0].elapsed_time(ev["repos"][1]) for ev in evs]
    # calls are ordered step-major, layer-minor: expand the per-step bytes per layer
    per_call = np.repeat(np.array(by["decode_per_call"]), SHAPE.layers)
    per_call = np.tile(per_call, args.steps)
    achieved = float(np.sum(per_call) / (np.sum(dec_ms) * 1e-3) / 1e9)
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    traffic = decode_traffic() if not args.profiling_case else None
    peak = peaks.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    value = world * by["total"] / (ms * 1e-3) / 1e9
    dec_time = float(np.sum(dec_ms)) / args.steps * 1e-3
    tok_s = world * BATCH * DECODE_STEPS / dec_time

    # end to end: the same step with inputs from pinned host memory and the
    # last layer's attention output read back every decode step
    e2e = None
    if not args.no_e2e:
        host = {"q": b.q.cpu().pin_memory(), "k": b.knew.cpu().pin_memory(),
                "v": b.vnew.cpu().pin_memory(),
                "out": torch.empty((DECODE_STEPS, BATCH, SHAPE.hq, SHAPE.head_dim),
                                   dtype=torch.float32).pin_memory()}
        b.step(host=host)
        torch.cuda.synchronize()
        barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(b.stream)
        for _ in range(args.steps):
            b.step(host=host)
        e2.record(b.stream)
        torch.cuda.synchronize()
        barrier()
        ms2 = reduce_max(s2.elapsed_time(e2) / args.steps, dist, "cuda")
        h2d = (b.q.numel() + b.knew.numel() + b.vnew.numel()) * BYTES_EL
        d2h = host["out"].numel() * 4
        e2e = {"value": world * by["total"] / (ms2 * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ms2,
               "what": "public C-ABI calls (fork/drop/reposition/append/decode) with every "
                       "decode step's q and new K/V copied from pinned host memory (on a "
                       "copy stream, overlapping compute; each decode step waits for its "
                       "inputs) and the last layer's attention output copied back"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded SplitMix64 K/V/q, seeded agent-trace span structure)",
            "config": {"workload": workload_name(), "global_batch": world * BATCH,
                       "seq_len": N_TOKENS, "decode_steps": DECODE_STEPS,
                       "parallelism": f"replicas x{world} (sequences partitioned, no collective)",
                       "l2": "inputs larger than L2 (each decode call reads ~0.9 GB); no flush",
                       "bytes_per_step": by["total"]},
            "decode_tok_s": round(tok_s, 1),
            "roofline": {"kernel": "k_decode_mma (one launch per decode-attention call, "
                                   "split merge fused; per-call time = span of a step's "
                                   f"{SHAPE.layers} back-to-back calls / {SHAPE.layers})",
                         "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic,
                         "avg_call_us": round(float(np.mean(dec_ms)) * 1e3, 2),
                         "algorithmic_bytes_per_call": int(np.mean(per_call))},
            "repos_ms": round(float(np.mean(repos_ms)), 3),
            "repos_gbs": round(by["repos"] / (np.mean(repos_ms) * 1e-3) / 1e9, 1),
            "gpu_launches": int(launches),
            "clocks": clk.summary(),
        }
        if args.profiling_case:
            line["config"]["profiling_case"] = (f"reduced for a profiler capture: batch {BATCH}, "
                                                f"{SHAPE.layers} layers, {DECODE_STEPS} decode steps")
        if cpu:
            line["cpu_baseline"] = {"value": round(cpu["bytes"] / cpu["seconds"] / 1e9, 4),
                                    "unit": "GB/s", "cores": cpu["workers"], "kind": "oracle",
                                    "sample": cpu["sample"]}
        if e2e:
            line["e2e"] = e2e
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


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
    assert cache.sync_errors() == 0
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


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    trajs = trajectories()
    n_seqs, n_layers, n_dec = 2, 2, 16
    for _ in range(args.warmup):
        oracle_sample(trajs, n_seqs, n_layers, n_dec)
    res = [oracle_sample(trajs, n_seqs, n_layers, n_dec) for _ in range(args.steps)]
    secs = sum(r["seconds"] for r in res)
    value = sum(r["bytes"] for r in res) / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_name()},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": res[0]["workers"],
                         "kind": "oracle", "sample": res[0]["sample"]},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    global BATCH, DECODE_STEPS, SHAPE
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["akv", "reference"], default="akv")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--restore", action="store_true",
                    help="time segment-batch restore attention instead (its own line)")
    ap.add_argument("--restore-cuda-cores", action="store_true")
    ap.add_argument("--config-kernels", default=None,
                    help="comma list of gptoss120b, branching, branching_fork, llama70b: decode and "
                         "reposition bandwidth on those workloads (one line each)")
    ap.add_argument("--prefix", action="store_true",
                    help="time prefix matching / forks / eviction instead (its own line)")
    # smaller cases for profiler captures only; a line printed with any of
    # these is marked "profiling case" and is not the benchmark's number
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--decode-steps", type=int, default=None)
    args = ap.parse_args()
    if args.batch or args.layers or args.decode_steps:
        import dataclasses
        BATCH = args.batch or BATCH
        DECODE_STEPS = args.decode_steps or DECODE_STEPS
        SHAPE = dataclasses.replace(SHAPE, layers=args.layers or SHAPE.layers)
        args.profiling_case = True
    else:
        args.profiling_case = False
    if args.config_kernels:
        kernels_arm(args)
    elif args.prefix:
        prefix_arm(args)
    elif args.restore or args.restore_cuda_cores:
        restore_arm(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
