"""The allocation-free decode-attention entry point matches the regular one.

akv_decode_attention_noalloc() is for callers that cannot allocate device
memory (applications that reserve all GPU memory at start-up and forbid
cudaMalloc/cudaFree while serving, such as a plugin living in another
runtime's memory pool).  It keeps its split-KV partials in a file-scope
device array instead of a workspace.  This test builds a cache through the
regular API, gives the same pool and the same page metadata to the
allocation-free call, and compares its output with akv_decode_attention()
on two calls in a row: the second call starts from the array contents the
first one left behind.
"""
import numpy as np
import pytest
import torch

from agent_kv_cache_gb300 import abi, build
from twin import ATTN_TOL, Twin
from workloads import synth

pytestmark = pytest.mark.gpu


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
    pt, act, keep, row_stride, keep_stride, n_act, n_held = _metadata(t, seqs)
    tmax, tmean = ATTN_TOL["bf16"]
    stream = torch.cuda.current_stream().cuda_stream
    for layer in range(t.L):
        q = np.stack([synth.query(t.seed, t.tag[s], layer, 0, t.hq, t.d, t.width) for s in seqs])
        qd = torch.from_numpy(q).to(torch.bfloat16).cuda()
        ref = t.gpu.decode_attention(layer, qd, seqs).clone()
        slab = layer % t.gpu.phys
        for call in range(2):
            out = torch.full_like(ref, float("nan"))
            abi.akv_decode_attention_noalloc(
                t.gpu.k_pool[slab].data_ptr(), t.gpu.v_pool[slab].data_ptr(),
                t.gpu.cfg.max_pages, t.hq, t.hkv, t.d, t.S, "bf16", 5e5,
                pt.data_ptr(), act.data_ptr(), keep.data_ptr(), row_stride, keep_stride,
                n_act, n_held, qd.data_ptr(), out.data_ptr(), stream)
            torch.cuda.synchronize()
            err = (out - ref).abs()
            assert torch.isfinite(out).all(), (layer, call)
            assert err.max().item() <= tmax and err.mean().item() <= tmean, (layer, call)
            assert torch.all(out[2] == 0), "a sequence with no active token gives zeros"


def test_noalloc_rejects_too_many_sequences():
    build()
    n = abi.lib()  # loaded
    with pytest.raises(abi.AkvError) as e:
        abi.akv_decode_attention_noalloc(1, 1, 1, 8, 2, 64, 16, "bf16", 1e4, 1, 1, 1, 1, 1,
                                         np.zeros(257, np.int32), np.zeros(257, np.int32),
                                         1, 1)
    assert e.value.code == abi.AKV_ECAPACITY
    del n
