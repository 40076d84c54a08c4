"""Full-size workloads: every sequence's metadata bit-exact against the
oracle, sampled keys/values/attention element by element; restore attention
of a full-length agent sequence on sampled tokens.

The four large workloads run at their full shapes and batch sizes, through
the same batched calls as the benchmark (so the same decode launch plan).
The long-running 70B-shaped workload runs 6 turns instead of 100 (with the
active-token cap lowered to 4096 so that its drop/reposition cycle still
fires); its shapes, batch and layer aliasing are the full ones.
"""
import gc

import numpy as np
import pytest
import torch

from agent_kv_cache_gb300 import Cache, abi, build
from fullsize import FullSize
from oracle.akv_oracle import OracleCache
from twin import ATTN_TOL
from workloads import device, synth, traces

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean():
    build()
    gc.collect()
    torch.cuda.empty_cache()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _pages(lengths, S, extra):
    return sum(-(-n // S) for n in lengths) + extra


def test_llama8b_trace_fullsize():
    """16 x 32768 tokens, ~60% dropped, reposition of forks, 2 decode steps x 32 layers."""
    sh, seed, B, N = traces.LLAMA8B, traces.seed_for(1), 16, 32768
    trajs = traces.llama8b_batch(seed, batch=B, n_total=N)
    rs = [N - sum(e - b for b, e in t.drop_ranges) for t in trajs]
    max_pages = B * (N // 16) + _pages([r + 8 for r in rs], 16, 2 * B + 64)
    fs = FullSize(sh, seed, 2 * B, max_pages, N + 64, sample_seqs=[0, 9], sample_layers=[0, 31])
    base = [fs.create(b, b + 1) for b in range(B)]
    fs.append_tokens(base, N)
    forks = [fs.fork(s, i, fs.tags[s]) for i, s in enumerate(base)]
    for f, tr in zip(forks, trajs):
        fs.drop(f, tr.drop_ranges)
    fs.check_metadata()
    fs.reposition(forks)
    fs.check_metadata()
    fs.check_kv()
    for step in range(2):
        fs.append_tokens(forks, 1)
        fs.decode(forks, step, range(sh.layers), check_layers=[0, 31])
    fs.check_metadata()
    fs.check_kv()
    fs.close()


def test_gptoss120b_trace_fullsize():
    """4 x 131072 tokens, ~80% dropped, D = 64, group 8, 2 decode steps x 36 layers."""
    sh, seed, B, N = traces.GPTOSS120B, traces.seed_for(2), 4, 131072
    trajs = traces.gptoss_batch(seed, batch=B, n_total=N)
    rs = [N - sum(e - b for b, e in t.drop_ranges) for t in trajs]
    max_pages = _pages([N] * B, 16, 0) + _pages([r + 8 for r in rs], 16, 64)
    fs = FullSize(sh, seed, B, max_pages, N + 64, sample_seqs=[1, 3], sample_layers=[0, 35])
    seqs = [fs.create(b, b + 1) for b in range(B)]
    fs.append_tokens(seqs, N)
    for s, tr in zip(seqs, trajs):
        fs.drop(s, tr.drop_ranges)
    fs.reposition(seqs)
    fs.check_metadata()
    fs.check_kv()
    for step in range(2):
        fs.append_tokens(seqs, 1)
        fs.decode(seqs, step, range(sh.layers), check_layers=[0, 35])
    fs.check_metadata()
    fs.close()


def test_branching_histories_fullsize():
    """A 16384-token prefix forked into 64 branches with 1-6 drop/reposition
    operations each; batched decode over all 64 branches.  Shared prefix
    pages stay shared and unchanged; repositioned pages are private."""
    sh, seed, P = traces.LLAMA8B, traces.seed_for(3), 16384
    segs, branches = traces.branching(seed, n_branches=64, prefix_len=P)
    max_pages = P // 16 + 64 * (P // 16 + 4) + 256
    fs = FullSize(sh, seed, 66, max_pages, P + 64, sample_seqs=[-1, 0, 13, 40],
                  sample_layers=[0, 31])
    root = fs.create(-1, 1)
    fs.append_tokens([root], P)
    pages0, _ = fs.gpu.page_table(root)
    idx = torch.from_numpy(pages0.astype(np.int64)).cuda()
    snap = fs.gpu.k_pool[:, idx].view(torch.int16).sum(dtype=torch.int64).item()
    kids = [fs.fork(root, i, 1) for i in range(64)]
    for k, br in zip(kids, branches):
        for op in br.ops:
            if op[0] == "drop":
                fs.drop(k, op[1])
            else:
                fs.reposition([k])
    fs.check_metadata()
    fs.check_kv()
    # the root's pages were never written by any branch
    assert fs.gpu.k_pool[:, idx].view(torch.int16).sum(dtype=torch.int64).item() == snap
    # every branch shares the pages before its first dropped slot
    for k in kids:
        pk, _ = fs.gpu.page_table(k)
        info = fs.gpu.info(k)
        assert info["n_shared_pages"] >= 0 and info["n_owned_pages"] >= 0
        shared = [p for p in pk if p >= 0 and fs.gpu.refcount(int(p)) > 1]
        assert set(shared) <= set(pages0.tolist())
    for step in range(2):
        fs.append_tokens(kids, 1)
        fs.decode(kids, step, range(sh.layers), check_layers=[0, 31])
    fs.check_metadata()
    for k in kids:
        fs.free(k)
    fs.free(root)
    assert fs.gpu.pool_stats()[1] == 0
    fs.close()


def test_llama70b_steady_state_fullsize():
    """64 sequences, 80 logical layers on 16 aliased slabs, 64/8 heads, D 128:
    6 turns of (tool response append, decode), drop oldest tool responses and
    reposition every 3 turns."""
    sh, seed, B = traces.LLAMA70B, traces.seed_for(4), 64
    turns = traces.steady_state(seed, n_seqs=B, n_turns=6, decode_per_turn=2, active_cap=4096)
    longest = max(1024 + sum(t.tool_len + 2 for t in ts) for ts in turns)
    max_pages = B * (-(-longest // 16) + 8) * 2
    fs = FullSize(sh, seed, B, max_pages, longest + 64, sample_seqs=[5, 50],
                  sample_layers=[3, 15], phys_layers=16)
    seqs = [fs.create(b, b + 1) for b in range(B)]
    fs.append_tokens(seqs, 1024)
    step = 0
    for k in range(6):
        for s, ts in zip(seqs, turns):
            fs.append_tokens([s], ts[k].tool_len)
        for _ in range(2):
            fs.append_tokens(seqs, 1)
            fs.decode(seqs, step, range(sh.layers), check_layers=[3, 79])
            step += 1
        did = []
        for s, ts in zip(seqs, turns):
            if ts[k].drop_ranges:
                fs.drop(s, ts[k].drop_ranges)
            if ts[k].repos:
                did.append(s)
        if did:
            fs.reposition(did)
    fs.check_metadata()
    fs.check_kv()
    fs.close()


def test_restore_llama8b_fullsize():
    """Restore attention of the long-running agent sequence (~34k tokens,
    10 repositions, 8B shape) on the tensor-core kernel, exactly as the
    restore benchmark calls it; 26 sampled tokens (first, last, random)
    checked against the oracle replay, and a windowed layer."""
    sh = traces.LLAMA8B
    seed = traces.seed_for(5)
    prog = traces.restore_program(seed)
    n = sum(op[1] for op in prog if op[0] == "append")
    H, D, Hq = sh.hkv, sh.head_dim, sh.hq
    w = synth.width_for(sh.dtype)
    gpu = Cache(2, Hq, H, D, sh.page_size, sh.dtype, 16, 2, n + 64, sh.rope_theta)
    gpu.set_layer_window(1, 4096)
    q = torch.empty((n, Hq, D), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((n, H, D), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    keep = [device.fill(x, [(synth.stream_key(seed, 1, kind, 0), 0, 0)], x.numel(), w)
            for x, kind in ((q, synth.KIND_Q), (k, synth.KIND_K), (v, synth.KIND_V))]
    torch.cuda.synchronize()
    del keep
    outs = [gpu.restore_attention(prog, l, q, k, v).double().cpu().numpy() for l in (0, 1)]
    assert gpu.sync_errors() == 0
    rng = np.random.default_rng(11)
    only = sorted(set([0, n - 1] + rng.integers(0, n, 24).tolist()))
    kk = synth.block(seed, 1, synth.KIND_K, 0, 0, n * H * D, w).reshape(1, n, H, D)
    vv = synth.block(seed, 1, synth.KIND_V, 0, 0, n * H * D, w).reshape(1, n, H, D)
    qq = np.stack([synth.block(seed, 1, synth.KIND_Q, 0, t * Hq * D, Hq * D, w).reshape(Hq, D)
                   for t in only])[None]
    for l, win in ((0, 0), (1, 4096)):
        o = OracleCache(Hq, H, D, sh.rope_theta, sh.dtype, layers=(0,), page_size=sh.page_size)
        want, _ = o.replay_attention(prog, qq, kk, vv, window=win, only=only)
        err = np.abs(outs[l][only] - want[0])
        tmax, tmean = ATTN_TOL[sh.dtype]
        assert err.max() <= tmax and err.mean() <= tmean, (l, err.max(), err.mean())
    gpu.close()


def test_prefix_fork_llama8b_fullsize():
    """The prefix-sharing workload at full size (8B shape, ~34k-token agent
    sequence published at every turn end), as the prefix benchmark runs it:
    the retrigger fork of the request that skipped the last reposition and
    the exact fork of the continuing request.  Checked: the match against
    properties the oracle's records fix at any size (equal records up to n,
    the next record differs, every needed key stored, rotated count), the
    child's keep mask / logical map bit-exact, and layer-0 keys and values
    against a cache built directly from the request prefix on sampled
    tokens."""
    import oracle.akv_prefix as P
    from agent_kv_cache_gb300 import PrefixIndex
    from twin import check_key_step, key_tolerance
    sh = traces.LLAMA8B
    seed = traces.seed_for(5)
    turns = traces.turn_programs(seed)
    n_total = sum(op[1] for t in turns for op in t if op[0] == "append")
    ids = traces.token_ids(seed, n_total + 64)
    S, L, H, D = sh.page_size, sh.layers, sh.hkv, sh.head_dim
    w = synth.width_for(sh.dtype)
    gpu = Cache(L, sh.hq, H, D, S, sh.dtype, 16384, 64, n_total + 64, sh.rope_theta)
    idx = PrefixIndex(S)
    live = gpu.seq_create()
    hist, t, entries = [], 0, {}
    for ops in turns:
        for op in ops:
            if op[0] == "append":
                for c0 in range(0, op[1], 4096):
                    m = min(4096, op[1] - c0)
                    k = torch.empty((L, m, H, D), dtype=torch.bfloat16, device="cuda")
                    v = torch.empty_like(k)
                    keep = [device.kv_tokens(k, seed, 1, synth.KIND_K, range(L), t, m, H, D, w),
                            device.kv_tokens(v, seed, 1, synth.KIND_V, range(L), t, m, H, D, w)]
                    torch.cuda.synchronize()
                    gpu.append([live], [m], k, v, ids[t:t + m].tolist())
                    torch.cuda.synchronize()
                    del keep
                    t += m
            elif op[0] == "drop":
                gpu.drop(live, op[1])
            else:
                gpu.reposition([live])
        hist += ops
        e = gpu.prefix_publish(idx, live, hist, ids[:t].tolist())
        entries[e] = P.records(hist, ids[:t])
    assert gpu.sync_errors() == 0
    cont_ids = ids[:t + 64].tolist()
    skip = hist[:-1] + [("append", 64)]
    cont = hist + [("append", 64)]
    last = max(entries)
    for prog, kind in ((skip, "retrigger"), (cont, "exact")):
        req = P.records(prog, cont_ids)
        child, m = gpu.prefix_fork(idx, prog, cont_ids)
        assert m["kind"] == kind and m["entry"] == last
        n = m["n_records"]
        er = entries[last]
        assert req[:n] == er[:n] and (n == len(er) or n == len(req) or req[n] != er[n])
        st = P.State(req[:n])
        stored = P.State(er).stored(S)
        need = [x for x in range(len(st.alive)) if st.alive[x]]
        assert all(x in stored for x in need)
        assert m["n_rotated"] == sum(stored[x] != st.pos[x] for x in need)
        if kind == "retrigger":
            assert m["n_rotated"] > 1000
        held = [x for x in range(len(st.alive)) if st.held[x]]
        np.testing.assert_array_equal(gpu.logical(child), held)
        np.testing.assert_array_equal(gpu.keep_mask(child), [st.alive[x] for x in held])
        # layer-0 keys of sampled needed tokens against the direct oracle replay
        oc = OracleCache(sh.hq, H, D, sh.rope_theta, sh.dtype, layers=(0,), page_size=S)
        osid = oc.create()
        tt = 0
        covered = list(prog[:m["op_index"]])
        if m["op_tokens"]:
            covered.append(("append", m["op_tokens"]))
        for op in covered:
            if op[0] == "append":
                cnt = op[1]
                kk = synth.kv_tokens(seed, 1, synth.KIND_K, [0], tt, cnt, H, D, w)
                vv = synth.kv_tokens(seed, 1, synth.KIND_V, [0], tt, cnt, H, D, w)
                oc.append(osid, kk, vv)
                tt += cnt
            elif op[0] == "drop":
                oc.drop(osid, op[1])
            else:
                oc.reposition(osid)
        os_ = oc.seqs[osid]
        assert np.array_equal(os_.logical, held)
        # step-wise, every needed token: the child's key is the entry's stored
        # key rotated from its stored position to the request's; the entry's
        # keys are first checked against the oracle replay of its own program
        eo = OracleCache(sh.hq, H, D, sh.rope_theta, sh.dtype, layers=(0,), page_size=S)
        esid = eo.create()
        tt = 0
        for op in hist:
            if op[0] == "append":
                eo.append(esid, synth.kv_tokens(seed, 1, synth.KIND_K, [0], tt, op[1], H, D, w),
                          synth.kv_tokens(seed, 1, synth.KIND_V, [0], tt, op[1], H, D, w))
                tt += op[1]
            elif op[0] == "drop":
                eo.drop(esid, op[1])
            else:
                eo.reposition(esid)
        src = np.array([stored[x] for x in need], dtype=np.int64)
        dst = np.array([st.pos[x] for x in need], dtype=np.int64)
        ke, _ = gpu.read_kv(last, 0)
        kg, vg = gpu.read_kv(child, 0)
        eref = eo.seqs[esid].K[0][src]
        n_rot_e = 1 + sum(1 for r in er if r[0] == "R")
        assert not (np.abs(ke[src] - eref) > key_tolerance(eref, sh.dtype, n_rot_e)).any()
        check_key_step(kg[dst], ke[src], src, dst, oc.freq, sh.dtype, kind)
        rng = np.random.default_rng(3)
        live_slots = np.flatnonzero(os_.alive)
        pick = rng.choice(live_slots, size=min(512, live_slots.size), replace=False)
        ref = os_.K[0][pick]
        n_rot = 1 + sum(1 for r in er if r[0] == "R") + 1
        assert not (np.abs(kg[pick] - ref) > key_tolerance(ref, sh.dtype, n_rot)).any()
        np.testing.assert_array_equal(vg[pick], os_.V[0][pick])
        gpu.seq_free(child)
    assert gpu.sync_errors() == 0
    freed, n_ev = gpu.prefix_evict(idx, 1 << 30)
    assert n_ev == len(entries) and freed > 0
    gpu.seq_free(live)
    assert gpu.pool_stats()[1] == 0
    gpu.close()
