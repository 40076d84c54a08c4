"""The allocation-free decode-attention entry point matches the regular one.

akv_decode_attention_noalloc() is for callers that cannot allocate device
memory (applications that reserve all GPU memory at start-up and forbid
cudaMalloc/cudaFree while serving, such as a plugin living in another
runtime's memory pool).  It keeps its split-KV partials in a file-scope
device array instead of a workspace.  These tests build a cache through the
regular API, give the same pool and the same page metadata to the
allocation-free call, and compare its output with akv_decode_attention() and
with the oracle on two calls in a row: the second call starts from the array
contents the first one left behind.  One case has enough long rows that the
first split plan's partials would not fit the array, so the splits are
widened.  The argument checks run without a GPU (nothing is launched).
"""
import numpy as np
import pytest
import torch

from agent_kv_cache_gb300 import abi, build
from twin import ATTN_TOL, Twin
from workloads import synth


def _metadata(t, seqs):
    """Device page table / active list / keep words in the library's layout."""
    infos = [t.gpu.info(s) for s in seqs]
    row_stride = max(1, max(i["n_pages"] for i in infos))
    keep_stride = max(1, max(-(-i["n_held"] // 32) for i in infos))
    pt = np.full((len(seqs), row_stride), -1, np.int32)
    act = np.full((len(seqs), row_stride), -1, np.int32)
    keep = np.zeros((len(seqs), keep_stride), np.uint32)
    for i, s in enumerate(seqs):
        pages, a = t.gpu.page_table(s)
        pt[i, :len(pages)] = pages
        act[i, :len(a)] = a
        bits = np.zeros(keep_stride * 32, np.uint64)
        km = t.gpu.keep_mask(s)
        bits[:len(km)] = km
        keep[i] = (bits.reshape(-1, 32) << np.arange(32, dtype=np.uint64)).sum(axis=1).astype(np.uint32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return (dev(pt), dev(act), dev(keep.view(np.int32)), row_stride, keep_stride,
            np.array([i["n_active_pages"] for i in infos], np.int32),
            np.array([i["n_held"] for i in infos], np.int32))


def _compare_twice(t, seqs, dtype, theta, oracle_rows=None):
    """Two allocation-free calls per layer against the regular call and the
    oracle (rows ``oracle_rows``, default all)."""
    pt, act, keep, row_stride, keep_stride, n_act, n_held = _metadata(t, seqs)
    tmax, tmean = ATTN_TOL[dtype]
    stream = torch.cuda.current_stream().cuda_stream
    rows = range(len(seqs)) if oracle_rows is None else oracle_rows
    for layer in range(t.L):
        q = np.stack([synth.query(t.seed, t.tag[s], layer, 0, t.hq, t.d, t.width) for s in seqs])
        qd = torch.from_numpy(q).to(t.tdtype).cuda()
        ref = t.gpu.decode_attention(layer, qd, seqs).clone()
        want = t.orc.attention(layer, q[list(rows)], [t.o[seqs[i]] for i in rows])
        slab = layer % t.gpu.phys
        for call in range(2):
            out = torch.full_like(ref, float("nan"))
            abi.akv_decode_attention_noalloc(
                t.gpu.k_pool[slab].data_ptr(), t.gpu.v_pool[slab].data_ptr(),
                t.gpu.cfg.max_pages, t.hq, t.hkv, t.d, t.S, dtype, theta,
                pt.data_ptr(), act.data_ptr(), keep.data_ptr(), row_stride, keep_stride,
                n_act, n_held, qd.data_ptr(), out.data_ptr(), stream)
            torch.cuda.synchronize()
            assert torch.isfinite(out).all(), (layer, call)
            err = (out - ref).abs()
            assert err.max().item() <= tmax and err.mean().item() <= tmean, (layer, call)
            err_o = np.abs(out.double().cpu().numpy()[list(rows)] - want)
            assert err_o.max() <= tmax and err_o.mean() <= tmean, (layer, call, err_o.max())
    return n_act


@pytest.mark.gpu
def test_noalloc_decode_matches_regular_decode_twice():
    build()
    t = Twin(layers=2, hq=32, hkv=8, head_dim=128, page_size=16, dtype="bf16",
             rope_theta=5e5, max_pages=2048, max_seqs=8, max_slots=8192, seed=11)
    seqs = [t.create() for _ in range(4)]
    t.append(seqs, [3000, 2500, 40, 1800])
    t.drop(seqs[0], [(100, 900), (2000, 2100)])
    t.drop(seqs[2], [(0, 40)])                  # nothing active left in seq 2
    t.drop(seqs[3], [(5, 6)])
    t.reposition([seqs[0], seqs[3]])
    t.append([seqs[0], seqs[1], seqs[3]], [1, 1, 1])
    _compare_twice(t, seqs, "bf16", 5e5)


@pytest.mark.gpu
def test_noalloc_widens_splits_to_fit_the_array():
    """64 rows of ~256 active pages with 64 query heads (group 16, D 128):
    the first split plan needs more partials than the 8 MiB array holds."""
    build()
    B, N = 64, 4096
    t = Twin(layers=1, hq=64, hkv=4, head_dim=128, page_size=16, dtype="bf16",
             rope_theta=5e5, max_pages=B * (N // 16 + 2), max_seqs=B, max_slots=N + 64, seed=12)
    seqs = [t.create() for _ in range(B)]
    t.append(seqs, [N] * B)
    for i, s in enumerate(seqs[::3]):
        t.drop(s, [(100 + i, 400 + 7 * i)])
    t.append(seqs, [1] * B)
    n_act = np.array([t.gpu.info(s)["n_active_pages"] for s in seqs], np.int64)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    pps = max(4, int(n_act.sum()) * t.hkv // (sms * 8))
    items = sum(-(-int(n) // pps) for n in n_act if -(-int(n) // pps) > 1)
    scratch_floats = abi.AKV_NOALLOC_SCRATCH_BYTES // 4
    assert items * t.hq * (t.d + 2) > scratch_floats, "the case must need wider splits"
    _compare_twice(t, seqs, "bf16", 5e5, oracle_rows=[0, 1, 31, 63])


@pytest.mark.gpu
def test_noalloc_fp32_head_dim_64():
    build()
    t = Twin(layers=1, hq=4, hkv=2, head_dim=64, page_size=4, dtype="fp32",
             rope_theta=1e4, max_pages=1024, max_seqs=4, max_slots=2048, seed=13)
    seqs = [t.create() for _ in range(3)]
    t.append(seqs, [700, 33, 1200])
    t.drop(seqs[2], [(10, 500)])
    t.reposition([seqs[2]])
    t.append(seqs, [1, 1, 1])
    _compare_twice(t, seqs, "fp32", 1e4)


def _call(**kw):
    a = dict(k_slab=1, v_slab=1, max_pages=8, hq=8, hkv=2, head_dim=64, page_size=16,
             dtype="bf16", rope_theta=1e4, page_table=1, active_pages=1, keep_bits=1,
             row_stride=4, keep_stride=2, n_active_pages=np.ones(2, np.int32),
             n_held=np.full(2, 16, np.int32), q=1, out=1)
    a.update(kw)
    with pytest.raises(abi.AkvError) as e:
        abi.akv_decode_attention_noalloc(**a)
    return e.value.code


def test_noalloc_argument_checks():
    """Each rejected argument returns its error before any device work (the
    pointers here are never dereferenced)."""
    build()
    assert _call(n_active_pages=np.zeros(257, np.int32),
                 n_held=np.zeros(257, np.int32)) == abi.AKV_ECAPACITY
    for name in ("k_slab", "v_slab", "page_table", "active_pages", "keep_bits", "q", "out"):
        assert _call(**{name: 0}) == abi.AKV_EINVAL, name
    for bad in (dict(hkv=0), dict(hkv=3), dict(hq=6), dict(hq=64, hkv=2),   # group 32
                dict(head_dim=96), dict(page_size=0), dict(page_size=12), dict(page_size=128),
                dict(dtype=7), dict(max_pages=0), dict(row_stride=0), dict(keep_stride=0),
                dict(rope_theta=1.0), dict(rope_theta=float("nan")),
                dict(n_active_pages=np.array([5, 1], np.int32)),              # > row_stride
                dict(n_active_pages=np.array([-1, 1], np.int32)),
                dict(n_held=np.array([65, 1], np.int32)),                      # > 32 * keep_stride
                dict(n_held=np.array([-1, 1], np.int32)),
                dict(n_held=np.array([0, 1], np.int32))):                      # active, none held
        assert _call(**bad) == abi.AKV_EINVAL, bad
