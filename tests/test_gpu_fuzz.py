"""Hundreds of tiny seeded operation programs against the oracle.

Every configuration of pool dtype (bf16, fp32) x page size (16, 1) x GQA
group (1, 4, 8) x head dim (64, 128) runs 10 programs of at most 8
operations on at most 512 tokens per sequence: appends (batched over the
live sequences), drops of random logical ranges, repositions of random
subsets, forks (pages shared), and decode attention over all live
sequences.  After every operation the Twin checks each key write step-wise
(1 bf16 ulp of the oracle on the bits the kernel read); after each program
every sequence's state is compared with the oracle in full (metadata
bit-exact, keys within the chained bound, values bit-exact) and decoded on
both layers; every sequence is then freed and the pool must be empty.
"""
import numpy as np
import pytest

from agent_kv_cache_gb300 import build
from twin import Twin

pytestmark = pytest.mark.gpu

MAX_TOKENS = 512


def _program(t, rng, step0):
    seqs = [t.create()]
    t.append(seqs, [int(rng.integers(1, 100))])
    step = step0
    for _ in range(int(rng.integers(1, 9))):
        u = rng.random()
        live = [s for s in seqs]
        if u < 0.3:
            k = int(rng.integers(1, 120))
            pick = [s for s in live if t.orc.seqs[t.o[s]].n_logical + k <= MAX_TOKENS]
            if pick:
                t.append(pick, [k] * len(pick))
        elif u < 0.55:
            s = live[int(rng.integers(0, len(live)))]
            n = t.orc.seqs[t.o[s]].n_logical
            ranges = []
            for _ in range(int(rng.integers(1, 4))):
                b = int(rng.integers(0, n))
                ranges.append((b, int(min(n, b + rng.integers(1, 80)))))
            t.drop(s, ranges)
        elif u < 0.75:
            pick = [s for s in live if rng.random() < 0.6] or live[:1]
            t.reposition(pick)
        elif u < 0.85 and len(seqs) < 4:
            seqs.append(t.fork(live[int(rng.integers(0, len(live)))]))
        else:
            t.decode(live, step)
            step += 1
    return seqs, step


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("page", [16, 1])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_tiny_programs(dtype, page, G, D):
    build()
    seed = {"bf16": 1, "fp32": 2}[dtype] * 1000 + page * 100 + G * 10 + D // 64
    hkv = 2
    t = Twin(layers=2, hq=G * hkv, hkv=hkv, head_dim=D, page_size=page, dtype=dtype,
             rope_theta=1e4, max_pages=4 * (MAX_TOKENS // page + 8) * 2,
             max_seqs=6, max_slots=MAX_TOKENS + 64, seed=seed)
    step = 0
    for p in range(10):
        rng = np.random.default_rng([seed, p])
        seqs, step = _program(t, rng, step)
        for s in seqs:
            t.check(s)
        t.append(seqs, [1] * len(seqs))
        t.decode(seqs, step)
        step += 1
        for s in seqs:
            t.free(s)
        assert t.gpu.pool_stats()[1] == 0
    assert t.gpu.sync_errors() == 0
    t.gpu.close()
