"""Drive the CUDA library and the CPU oracle with the same seeded inputs.

Inputs come from ``workloads.synth`` only (values exact in the pool dtype).
The oracle's state is built from those inputs alone and every comparison of
the chained kind below is against that state.  The step-wise key check is
the one place where the oracle's rotation function is applied to key bits
read from the pool: the bits one step starts from, which are first checked
against the oracle's own state (chained bound); almost all of them are
bit-identical to it.

Tolerances (derived from the arithmetic):

* indices, keep masks, positions, gather maps, active page lists: bit-exact;
* V: bit-exact (it is only copied);
* K, step-wise (the bound the method states for Eq. (5)): every key write --
  the rotation of an append, of a reposition, of a prefix fork -- is checked
  against the oracle applied to the exact bits the kernel read
  (``oracle.reposition_key`` from the old position p to the new position q,
  in fp64, rounded to the pool dtype, RNE).  bf16 pools: every element within
  1 bf16 ulp of that value.  fp32 pools: within 4 * 2^-24 * |(x, y)| (one
  rotation in fp32 from a table rounded once from fp64 -- table, product and
  fma roundings, 3 * 2^-24 |(x, y)| -- plus the oracle's own rounding of the
  result).  Both allow, on top, 2^-50 (|p| + |q| + 4) |(x, y)|: a bound on
  the fp64 evaluation error of the rotation angles p f_i and q f_i (f_i <= 1),
  which is what separates the oracle's value from the exact one (about 10^-6
  of a bf16 ulp at typical magnitudes).  A key whose position does not change
  must be bit-identical to what was read; dims past the rotary part too.
* K, chained (the whole history against the oracle's own chain): every
  stored key went through r roundings to the pool dtype (the append plus
  each reposition that moved it), and the two sides start each later
  rotation from inputs that may already differ by 1 ulp per component; a
  rotation preserves the norm of that difference and spreads it over both
  components, so the bound per element is
      ulp(ref) + (r - 1) * sqrt(2) * 2^(1-p) * |(x, y)| + r * 8 * 2^-24 * |(x, y)|
  (p = 8 significant bits for bf16, 24 for fp32; ulp(v) <= 2^(1-p) |v|).
  Every element must meet it, and at least 99% of the elements must lie
  within r ulp of the oracle.  This compounding is not a kernel error: the
  step-wise check pins each step to 1 ulp.
* attention output (fp32): max abs error <= 1e-2 and mean abs error <= 1e-3
  for bf16 pools; 1e-4 / 1e-5 for fp32 pools.
"""
import numpy as np
import torch

from agent_kv_cache_gb300 import Cache
from oracle.akv_oracle import OracleCache, reposition_key, to_pool
from workloads import synth

ATTN_TOL = {"bf16": (1e-2, 1e-3), "fp32": (1e-4, 1e-5)}


def ulp(x, dtype):
    """Spacing of the pool dtype at |x| (x float64)."""
    bits = 8 if dtype == "bf16" else 24
    ax = np.maximum(np.abs(x), 2.0 ** -100)
    return 2.0 ** (np.floor(np.log2(ax)) - (bits - 1))


def _pair_norm(ref, rope_dim=0):
    """|(x, y)| of each element's rotation pair; 0 on dims that never rotate."""
    d = ref.shape[-1]
    r = rope_dim or d
    h = r // 2
    norm = np.sqrt(ref[..., :h] ** 2 + ref[..., h:r] ** 2)
    return np.concatenate([norm, norm, np.zeros(ref.shape[:-1] + (d - r,))], axis=-1)


def key_tolerance(ref, dtype, n_rot, rope_dim=0):
    """Per-element bound of a key that went through n_rot roundings."""
    p = 8 if dtype == "bf16" else 24
    r = max(n_rot, 1)
    norm = _pair_norm(ref, rope_dim)
    return (ulp(ref, dtype) + (r - 1) * np.sqrt(2.0) * 2.0 ** (1 - p) * norm
            + r * 8 * 2.0 ** -24 * norm)


def check_key_step(got, src, p, q, freq, dtype, what=""):
    """Step-wise check of key writes: ``src`` [n, ..., D] are the stored key
    bits a kernel read (fp64 copies of pool values; the raw input for an
    append, with p = 0), ``got`` what it stored, each row rotated from
    position p[n] to q[n] (Eq. 5; Eq. 3 for an append).  ``freq`` holds the
    rotary frequencies (its length is half the rotary width).  Returns the
    largest error in units of the bf16/fp32 bound (<= 1 passes)."""
    got = np.asarray(got, dtype=np.float64)
    src = np.asarray(src, dtype=np.float64)
    p = np.asarray(p, dtype=np.int64)
    q = np.asarray(q, dtype=np.int64)
    if got.shape[0] == 0:
        return 0.0
    shp = (-1,) + (1,) * (src.ndim - 2)
    rw = 2 * len(freq)
    same = p == q
    # unmoved keys and the dims past the rotary part: bit copies
    np.testing.assert_array_equal(got[same], src[same], err_msg=what)
    np.testing.assert_array_equal(got[..., rw:], src[..., rw:], err_msg=what)
    want = to_pool(reposition_key(src, p.reshape(shp), q.reshape(shp), freq), dtype)
    norm = _pair_norm(src, rw)[..., :rw]
    slack = 2.0 ** -50 * (np.abs(p) + np.abs(q) + 4).astype(np.float64).reshape(shp + (1,)) * norm
    if dtype == "bf16":
        tol = ulp(want[..., :rw], dtype) + slack
    else:
        tol = 4 * 2.0 ** -24 * norm + slack
    err = np.abs(got[..., :rw] - want[..., :rw])
    bad = err > tol
    assert not bad.any(), (what, int(bad.sum()), err[bad][:4], want[..., :rw][bad][:4],
                           tol[bad][:4])
    return float((err / np.maximum(tol, 1e-300)).max())


def key_ulp_fraction(err, ref, dtype, n_rot, rope_dim=0):
    """Fraction of elements within n_rot ulp of the oracle."""
    r = max(n_rot, 1)
    ok = err <= r * (ulp(ref, dtype) + 8 * 2.0 ** -24 * _pair_norm(ref, rope_dim))
    return float(ok.mean()) if ok.size else 1.0


class Twin:
    def __init__(self, layers=1, hq=8, hkv=2, head_dim=64, page_size=16, dtype="fp32",
                 rope_theta=1e4, max_pages=256, max_seqs=8, max_slots=2048, seed=1,
                 phys_layers=0, rope_dim=0):
        self.gpu = Cache(layers, hq, hkv, head_dim, page_size, dtype, max_pages, max_seqs,
                         max_slots, rope_theta, phys_layers=phys_layers, rope_dim=rope_dim)
        self.orc = OracleCache(hq, hkv, head_dim, rope_theta, dtype, layers=range(layers),
                               page_size=page_size, rope_dim=rope_dim)
        self.orc.freq_theta = rope_theta
        self.windows = {}
        self.L, self.hq, self.hkv, self.d, self.S = layers, hq, hkv, head_dim, page_size
        self.dtype = dtype
        self.width = synth.width_for(dtype)
        self.seed = seed
        self.o = {}        # gpu seq id -> oracle seq id
        self.tag = {}      # gpu seq id -> input stream tag
        self.rot = {}      # gpu seq id -> rotations a key may have gone through
        self.same_bits = 0  # reposition inputs bit-identical to the oracle's state
        self.all_bits = 0
        self.next_tag = 1
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32

    # -- operations on both sides -----------------------------------------
    def create(self):
        g = self.gpu.seq_create()
        self.o[g] = self.orc.create()
        self.tag[g] = self.next_tag
        self.next_tag += 1
        self.rot[g] = 1
        return g

    def fork(self, parent):
        g = self.gpu.seq_fork(parent)
        self.o[g] = self.orc.fork(self.o[parent])
        self.tag[g] = self.next_tag
        self.next_tag += 1
        self.rot[g] = self.rot[parent]
        return g

    def free(self, g):
        self.gpu.seq_free(g)
        self.orc.free(self.o.pop(g))

    def _kv(self, g, n):
        t0 = self.orc.seqs[self.o[g]].n_logical
        k = synth.kv_tokens(self.seed, self.tag[g], synth.KIND_K, range(self.L), t0, n,
                            self.hkv, self.d, self.width)
        v = synth.kv_tokens(self.seed, self.tag[g], synth.KIND_V, range(self.L), t0, n,
                            self.hkv, self.d, self.width)
        return k, v

    def append(self, seqs, ns, token_ids=None):
        ks, vs = [], []
        for g, n in zip(seqs, ns):
            k, v = self._kv(g, n)
            ks.append(k)
            vs.append(v)
        tok = 0
        for g, n, k, v in zip(seqs, ns, ks, vs):
            ids = None if token_ids is None else token_ids[tok:tok + n]
            self.orc.append(self.o[g], k, v, ids)
            tok += n
        starts = {g: self.gpu.info(g)["n_held"] for g in seqs}
        kt = torch.from_numpy(np.concatenate(ks, axis=1)).to(self.tdtype).cuda().contiguous()
        vt = torch.from_numpy(np.concatenate(vs, axis=1)).to(self.tdtype).cuda().contiguous()
        self.gpu.append(list(seqs), list(ns), kt, vt, token_ids)
        torch.cuda.synchronize()
        # step-wise: each new key is R(pos) of its raw bits, rounded once
        for g, n, k in zip(seqs, ns, ks):
            if n == 0:
                continue
            h0 = starts[g]
            pos = self.orc.seqs[self.o[g]].pos[h0:h0 + n]
            got = self._keys(g)[:, h0:h0 + n]                   # [L][n][hkv][D]
            src = np.asarray(k, dtype=np.float64)
            check_key_step(got.transpose(1, 0, 2, 3), src.transpose(1, 0, 2, 3),
                           np.zeros_like(pos), pos, self.orc.freq, self.dtype, "append")

    def drop(self, g, ranges):
        self.gpu.drop(g, ranges)
        self.orc.drop(self.o[g], ranges)

    def _keys(self, g):
        """Stored keys of every layer, [L][n_held][hkv][D] (fp64 copy)."""
        if self.gpu.info(g)["n_held"] == 0:
            return np.zeros((self.L, 0, self.hkv, self.d))
        return np.stack([self.gpu.read_kv(g, l)[0] for l in range(self.L)])

    def reposition(self, seqs):
        before = {}
        for g in seqs:
            st = self.orc.seqs[self.o[g]]
            k_old = self._keys(g)
            src = np.flatnonzero(st.alive)
            # the bits the kernel will read, against the oracle's own state
            ref = st.K[:, src]
            err = np.abs(k_old[:, src] - ref)
            assert not (err > key_tolerance(ref, self.dtype, self.rot[g],
                                            self.orc.rope_dim)).any()
            self.same_bits += int((err == 0).sum())
            self.all_bits += err.size
            before[g] = (k_old, st.pos.copy(), src)
        self.gpu.reposition(list(seqs))
        for g in seqs:
            st = self.orc.seqs[self.o[g]]
            if not (st.alive.all() and np.array_equal(st.pos, np.arange(st.alive.size))):
                self.rot[g] += 1
            self.orc.reposition(self.o[g])
        # step-wise: survivor j is the key read from its old slot, rotated
        # from its old position to j
        torch.cuda.synchronize()
        for g in seqs:
            k_old, pos_old, src = before[g]
            if src.size == 0:
                continue
            got = self._keys(g)[:, :src.size]
            check_key_step(got.transpose(1, 0, 2, 3), k_old[:, src].transpose(1, 0, 2, 3),
                           pos_old[src], np.arange(src.size), self.orc.freq, self.dtype,
                           "reposition")

    def set_window(self, layer, window):
        self.gpu.set_layer_window(layer, window)
        self.windows[layer] = window

    def decode(self, seqs, step, layers=None):
        """Decode attention for every layer; returns the max/mean abs errors."""
        layers = range(self.L) if layers is None else layers
        worst = (0.0, 0.0)
        for l in layers:
            q = np.stack([synth.query(self.seed, self.tag[g], l, step, self.hq, self.d,
                                      self.width) for g in seqs])
            out = self.gpu.decode_attention(l, torch.from_numpy(q).to(self.tdtype).cuda(),
                                            list(seqs))
            got = out.double().cpu().numpy()
            want = self.orc.attention(l, q, [self.o[g] for g in seqs],
                                      window=self.windows.get(l, 0))
            err = np.abs(got - want)
            worst = (max(worst[0], err.max()), max(worst[1], err.mean()))
            tmax, tmean = ATTN_TOL[self.dtype]
            assert err.max() <= tmax and err.mean() <= tmean, (l, err.max(), err.mean())
        return worst

    def restore(self, program, layer=0):
        """Restore attention of one layer over `program` on the GPU vs the
        oracle's replay; returns (max, mean) abs error."""
        n = sum(op[1] for op in program if op[0] == "append")
        tag = self.next_tag
        self.next_tag += 1
        w = self.width
        q = synth.block(self.seed, tag, synth.KIND_Q, layer, 0, n * self.hq * self.d, w)
        k = synth.block(self.seed, tag, synth.KIND_K, layer, 0, n * self.hkv * self.d, w)
        v = synth.block(self.seed, tag, synth.KIND_V, layer, 0, n * self.hkv * self.d, w)
        q = q.reshape(n, self.hq, self.d)
        k = k.reshape(n, self.hkv, self.d)
        v = v.reshape(n, self.hkv, self.d)
        dev = lambda x: torch.from_numpy(x).to(self.tdtype).cuda().contiguous()
        got = self.gpu.restore_attention(program, layer, dev(q), dev(k), dev(v))
        got = got.double().cpu().numpy()
        o = OracleCache(self.hq, self.hkv, self.d, self.orc.freq_theta, self.dtype, layers=(0,),
                        page_size=self.S, rope_dim=self.orc.rope_dim)
        want, _ = o.replay_attention(program, q[None], k[None], v[None],
                                     window=self.windows.get(layer, 0))
        err = np.abs(got - want[0])
        tmax, tmean = ATTN_TOL[self.dtype]
        assert err.max() <= tmax and err.mean() <= tmean, (err.max(), err.mean())
        assert self.gpu.sync_errors() == 0
        return float(err.max()), float(err.mean())

    def restore_tokens(self, program, layer, tokens):
        """Restore attention of the tokens `tokens` only (GPU) vs the
        oracle's replay of those tokens; the other rows must stay as they
        were (NaN here).  Returns (max, mean) abs error."""
        n = sum(op[1] for op in program if op[0] == "append")
        tag = self.next_tag
        self.next_tag += 1
        w = self.width
        q = synth.block(self.seed, tag, synth.KIND_Q, layer, 0, n * self.hq * self.d, w)
        k = synth.block(self.seed, tag, synth.KIND_K, layer, 0, n * self.hkv * self.d, w)
        v = synth.block(self.seed, tag, synth.KIND_V, layer, 0, n * self.hkv * self.d, w)
        q = q.reshape(n, self.hq, self.d)
        k = k.reshape(n, self.hkv, self.d)
        v = v.reshape(n, self.hkv, self.d)
        dev = lambda x: torch.from_numpy(x).to(self.tdtype).cuda().contiguous()
        out = torch.full((n, self.hq, self.d), float("nan"), dtype=torch.float32, device="cuda")
        self.gpu.restore_attention_tokens(program, layer, dev(q), dev(k), dev(v), list(tokens),
                                          out=out)
        got = out.double().cpu().numpy()
        assert self.gpu.sync_errors() == 0
        rest = np.ones(n, bool)
        rest[list(tokens)] = False
        assert np.isnan(got[rest]).all()
        if not len(tokens):
            return 0.0, 0.0
        o = OracleCache(self.hq, self.hkv, self.d, self.orc.freq_theta, self.dtype, layers=(0,),
                        page_size=self.S, rope_dim=self.orc.rope_dim)
        want, _ = o.replay_attention(program, q[None][:, list(tokens)], k[None], v[None],
                                     window=self.windows.get(layer, 0), only=list(tokens))
        err = np.abs(got[list(tokens)] - want[0])
        tmax, tmean = ATTN_TOL[self.dtype]
        assert err.max() <= tmax and err.mean() <= tmean, (err.max(), err.mean())
        return float(err.max()), float(err.mean())

    # -- comparison --------------------------------------------------------
    def check(self, g, kv=True):
        o = self.orc.seqs[self.o[g]]
        info = self.gpu.info(g)
        want = self.orc.info(self.o[g])
        for k in ("n_logical", "n_held", "next_pos", "n_pages", "n_active_pages"):
            assert info[k] == want[k], (k, info[k], want[k])
        assert info["n_active"] == want["n_alive"]
        n = info["n_held"]
        np.testing.assert_array_equal(self.gpu.keep_mask(g), o.alive)
        np.testing.assert_array_equal(self.gpu.logical(g), o.logical)
        np.testing.assert_array_equal(self.gpu.positions(g), o.pos)
        pages, act = self.gpu.page_table(g)
        np.testing.assert_array_equal(act, self.orc.active_pages(self.o[g]))
        assert len(pages) == -(-n // self.S)
        # every page with an active token is a valid pool page
        for k in act:
            assert 0 <= pages[k] < self.gpu.cfg.max_pages
            assert self.gpu.refcount(int(pages[k])) >= 1
        if o.last_gather is not None:
            np.testing.assert_array_equal(self.gpu.gather_map(g), o.last_gather)
        if kv and n:
            live = np.array([pages[s // self.S] >= 0 for s in range(n)])
            for l in range(self.L):
                k, v = self.gpu.read_kv(g, l)
                ref_k = o.K[l][live]
                tol = key_tolerance(ref_k, self.dtype, self.rot[g], self.orc.rope_dim)
                err = np.abs(k[live] - ref_k)
                bad = err > tol
                assert not bad.any(), (l, err[bad][:5], ref_k[bad][:5], tol[bad][:5])
                frac = key_ulp_fraction(err, ref_k, self.dtype, self.rot[g], self.orc.rope_dim)
                rd = self.orc.rope_dim
                if rd < self.d:      # dims past the rotary part are copied: bit-exact
                    np.testing.assert_array_equal(k[live][..., rd:], ref_k[..., rd:])
                assert frac >= 0.99, (l, frac)
                np.testing.assert_array_equal(v[live], o.V[l][live])
        assert self.gpu.sync_errors() == 0

    def history_equal(self, a, b):
        return self.gpu.history_key(a) == self.gpu.history_key(b)
