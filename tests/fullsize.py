"""Full-size workloads on the GPU checked against the oracle on samples.

The library runs the whole workload (every sequence, every layer, the same
batched calls and therefore the same launch configuration as ``bench.py``).
The oracle follows every sequence's metadata exactly (an instance with no
layers tracks tokens, keep flags, positions and gather maps without storing
any K/V) and the full K/V state of a few sampled sequences on a few sampled
layers, whose keys, values and attention outputs are compared element by
element.  Inputs: ``workloads`` generators only (device copy for the GPU,
numpy for the oracle, bit-identical).
"""
import numpy as np
import torch

from agent_kv_cache_gb300 import Cache
from oracle.akv_oracle import OracleCache
from twin import ATTN_TOL, check_key_step, key_tolerance, key_ulp_fraction
from workloads import device, synth


class FullSize:
    def __init__(self, shape, seed, n_seqs, max_pages, max_slots, sample_seqs, sample_layers,
                 phys_layers=0, chunk=4096):
        self.shape, self.seed = shape, seed
        self.L = shape.layers
        self.phys = phys_layers or shape.layers
        self.width = synth.width_for(shape.dtype)
        self.gpu = Cache(shape.layers, shape.hq, shape.hkv, shape.head_dim, shape.page_size,
                         shape.dtype, max_pages, n_seqs + 2, max_slots, shape.rope_theta,
                         phys_layers=phys_layers)
        mk = lambda layers: OracleCache(shape.hq, shape.hkv, shape.head_dim, shape.rope_theta,
                                        shape.dtype, layers=layers, page_size=shape.page_size)
        self.meta = mk([])
        # sampled layers are physical slabs; each holds the last logical layer
        # written to it (logical layer l lives in slab l % phys)
        self.sample_layers = list(sample_layers)
        self.kv = mk(self.sample_layers)
        self.sample = set(sample_seqs)
        self.chunk = chunk
        self.seqs, self.tags, self.om, self.ok, self.rot = [], {}, {}, {}, {}
        self.t_dtype = torch.bfloat16 if shape.dtype == "bf16" else torch.float32

    def writer_layer(self, slab):
        """Logical layer whose data a slab ends up holding."""
        return slab + self.phys * ((self.L - 1 - slab) // self.phys)

    def create(self, index, tag):
        s = self.gpu.seq_create()
        self.seqs.append(s)
        self.tags[s] = tag
        self.om[s] = self.meta.create()
        if index in self.sample:
            self.ok[s] = self.kv.create()
        self.rot[s] = 1
        return s

    def fork(self, parent, index, tag):
        s = self.gpu.seq_fork(parent)
        self.seqs.append(s)
        self.tags[s] = tag
        self.om[s] = self.meta.fork(self.om[parent])
        if index in self.sample and parent in self.ok:
            self.ok[s] = self.kv.fork(self.ok[parent])
        self.rot[s] = self.rot[parent]
        return s

    def free(self, s):
        self.gpu.seq_free(s)
        self.meta.free(self.om.pop(s))
        if s in self.ok:
            self.kv.free(self.ok.pop(s))
        self.seqs.remove(s)

    def append_tokens(self, seqs, n):
        """Append n tokens to each of seqs (their own streams): the GPU gets
        device-generated chunks, the oracle one host-generated block."""
        sh = self.shape
        L, H, D = sh.layers, sh.hkv, sh.head_dim
        starts = {s: self.meta.seqs[self.om[s]].n_logical for s in seqs}
        if n * len(seqs) <= self.chunk:
            plan = [(list(seqs), 0, n)]
        else:
            plan = [([s], t0, min(self.chunk, n - t0)) for s in seqs
                    for t0 in range(0, n, self.chunk)]
        for group, off, m in plan:
            k = torch.empty((L, m * len(group), H, D), dtype=self.t_dtype, device="cuda")
            v = torch.empty_like(k)
            tags = [self.tags[s] for s in group]
            st = [starts[s] + off for s in group]
            keep = [device.kv_tokens_multi(k, self.seed, tags, synth.KIND_K, range(L), st, m,
                                           H, D, self.width),
                    device.kv_tokens_multi(v, self.seed, tags, synth.KIND_V, range(L), st, m,
                                           H, D, self.width)]
            self.gpu.append(group, [m] * len(group), k, v)
            torch.cuda.synchronize()
            del keep
        layers = [self.writer_layer(p) for p in self.sample_layers]
        for s in seqs:
            h0 = self.meta.seqs[self.om[s]].alive.size
            self.meta.append(self.om[s], np.zeros((0, n, H, D)), np.zeros((0, n, H, D)))
            if s in self.ok:
                kk = synth.kv_tokens(self.seed, self.tags[s], synth.KIND_K, layers, starts[s], n,
                                     H, D, self.width)
                vv = synth.kv_tokens(self.seed, self.tags[s], synth.KIND_V, layers, starts[s], n,
                                     H, D, self.width)
                self.kv.append(self.ok[s], kk, vv)
                # step-wise: the new keys are R(pos) of their raw bits, rounded once
                pos = self.meta.seqs[self.om[s]].pos[h0:h0 + n]
                got = np.stack([self.gpu.read_kv(s, slab, h0, h0 + n)[0]
                                for slab in self.sample_layers], axis=1)
                check_key_step(got, kk.transpose(1, 0, 2, 3), np.zeros_like(pos), pos,
                               self.kv.freq, sh.dtype, "append")

    def drop(self, s, ranges):
        self.gpu.drop(s, ranges)
        self.meta.drop(self.om[s], ranges)
        if s in self.ok:
            self.kv.drop(self.ok[s], ranges)

    def reposition(self, seqs):
        # the key bits the kernel will read, for the sampled sequences, first
        # against the oracle's own state (chained bound)
        before = {}
        for s in seqs:
            if s not in self.ok:
                continue
            st = self.kv.seqs[self.ok[s]]
            src = np.flatnonzero(st.alive)
            k_old = np.stack([self.gpu.read_kv(s, slab)[0] for slab in self.sample_layers])
            ref = st.K[:, src]
            err = np.abs(k_old[:, src] - ref)
            assert not (err > key_tolerance(ref, self.shape.dtype, self.rot[s])).any()
            before[s] = (k_old[:, src], st.pos[src].copy())
        self.gpu.reposition(seqs)
        for s in seqs:
            st = self.meta.seqs[self.om[s]]
            if not (st.alive.all() and np.array_equal(st.pos, np.arange(st.alive.size))):
                self.rot[s] += 1
            self.meta.reposition(self.om[s])
            if s in self.ok:
                self.kv.reposition(self.ok[s])
        # step-wise: survivor j is the key read from its old slot, rotated
        # from its old position to j
        torch.cuda.synchronize()
        for s, (k_src, p_old) in before.items():
            r = p_old.size
            got = np.stack([self.gpu.read_kv(s, slab, 0, r)[0] for slab in self.sample_layers])
            check_key_step(got.transpose(1, 0, 2, 3), k_src.transpose(1, 0, 2, 3), p_old,
                           np.arange(r), self.kv.freq, self.shape.dtype, "reposition")

    # -- checks -------------------------------------------------------------
    def check_metadata(self):
        for s in self.seqs:
            o = self.meta.seqs[self.om[s]]
            info = self.gpu.info(s)
            want = self.meta.info(self.om[s])
            for k in ("n_logical", "n_held", "next_pos", "n_pages", "n_active_pages"):
                assert info[k] == want[k], (s, k, info[k], want[k])
            np.testing.assert_array_equal(self.gpu.keep_mask(s), o.alive)
            np.testing.assert_array_equal(self.gpu.logical(s), o.logical)
            np.testing.assert_array_equal(self.gpu.positions(s), o.pos)
            _, act = self.gpu.page_table(s)
            np.testing.assert_array_equal(act, self.meta.active_pages(self.om[s]))
            if o.last_gather is not None:
                np.testing.assert_array_equal(self.gpu.gather_map(s), o.last_gather)
        assert self.gpu.sync_errors() == 0

    def check_kv(self):
        S = self.shape.page_size
        for s, osid in self.ok.items():
            o = self.kv.seqs[osid]
            n = self.gpu.info(s)["n_held"]
            pages, _ = self.gpu.page_table(s)
            live = np.array([pages[i // S] >= 0 for i in range(n)], dtype=bool)
            for li, slab in enumerate(self.sample_layers):
                k, v = self.gpu.read_kv(s, slab)
                ref = o.K[li][live]
                err = np.abs(k[live] - ref)
                tol = key_tolerance(ref, self.shape.dtype, self.rot[s])
                assert not (err > tol).any(), (s, slab, err[err > tol][:4])
                assert key_ulp_fraction(err, ref, self.shape.dtype, self.rot[s]) >= 0.99
                np.testing.assert_array_equal(v[live], o.V[li][live])

    def decode(self, seqs, step, layers, check_layers):
        """Decode attention for `layers` over all `seqs` (one batched call per
        layer, as in the benchmark); sampled (seq, layer) outputs are checked."""
        sh = self.shape
        worst = 0.0
        q = torch.empty((len(seqs), sh.hq, sh.head_dim), dtype=self.t_dtype, device="cuda")
        for l in layers:
            keep = device.queries(q, self.seed, [self.tags[s] for s in seqs], l, step, sh.hq,
                                  sh.head_dim, self.width)
            out = self.gpu.decode_attention(l, q, seqs).double().cpu().numpy()
            del keep
            if l not in check_layers:
                continue
            slab = l % self.phys
            li = self.sample_layers.index(slab)
            for i, s in enumerate(seqs):
                if s not in self.ok:
                    continue
                qq = synth.query(self.seed, self.tags[s], l, step, sh.hq, sh.head_dim, self.width)
                want = self.kv.attention(li, qq[None], [self.ok[s]])[0]
                err = np.abs(out[i] - want)
                tmax, tmean = ATTN_TOL[sh.dtype]
                assert err.max() <= tmax and err.mean() <= tmean, (s, l, err.max(), err.mean())
                worst = max(worst, float(err.max()))
        return worst

    def close(self):
        self.gpu.close()
        del self.gpu
        torch.cuda.empty_cache()
