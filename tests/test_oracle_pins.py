"""Pins of the CPU oracle to facts fixed outside itself.

Each pin compares the oracle with something it does not compute itself: the
worked examples the pages print (``tests/golden``), closed forms evaluated by
an independent formulation (complex exponentials, explicit matrices and
numpy's own inverse), textbook softmax attention (scipy), brute force on tiny
inputs, and invariants.  ``test_pins_catch_planted_mistakes`` plants
plausible mistakes in the oracle (on the CPU) and checks that some pin fails
for each.
"""
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle.akv_oracle as O
from workloads import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def pin_inv_freq():
    f = O.inv_freq(64, 1.0e4)
    assert f.shape == (32,)
    assert f[0] == 1.0
    # theta^(-2i/D) at i = D/4 is theta^(-1/2) = 0.01 for theta = 1e4
    assert abs(f[16] - 0.01) < 1e-15
    # a geometric sequence with ratio theta^(-2/D)
    np.testing.assert_allclose(f[1:] / f[:-1], 1.0e4 ** (-2.0 / 64), rtol=1e-13)


def pin_rope_complex_form():
    """R(p) is multiplication of z_i = x_i + i x_{i+D/2} by exp(i p f_i)."""
    rng = np.random.default_rng(1)
    for d, theta in ((64, 1.0e4), (128, 5.0e5)):
        f = O.inv_freq(d, theta)
        x = _rand(rng, 7, d)
        pos = np.array([0, 1, 2, 17, 1000, 65535, 131071])
        got = O.rope(x, pos, f)
        z = (x[:, : d // 2] + 1j * x[:, d // 2:]) * np.exp(1j * pos[:, None] * f)
        want = np.concatenate([z.real, z.imag], axis=1)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)
        zi = (x[:, : d // 2] + 1j * x[:, d // 2:]) * np.exp(-1j * pos[:, None] * f)
        np.testing.assert_allclose(O.rope_inverse(x, pos, f),
                                   np.concatenate([zi.real, zi.imag], axis=1),
                                   rtol=0, atol=1e-12)


def _matrix(fn, d, pos, f):
    """Explicit D x D matrix of a linear map, column by column."""
    return fn(np.eye(d), np.full(d, pos), f).T


def pin_rope_matrix_identities():
    """R(p) is orthogonal and R(q) R(p)^-1 = R(q - p) (closed form)."""
    d, theta = 64, 1.0e4
    f = O.inv_freq(d, theta)
    for p, q in ((5, 2), (131071, 13), (40000, 0), (7, 7)):
        rp = _matrix(O.rope, d, p, f)
        rq = _matrix(O.rope, d, q, f)
        np.testing.assert_allclose(rp @ rp.T, np.eye(d), atol=1e-13)
        np.testing.assert_allclose(np.linalg.det(rp), 1.0, atol=1e-12)
        np.testing.assert_allclose(rq @ np.linalg.inv(rp),
                                   _matrix(O.rope, d, q - p, f), atol=1e-12)
        np.testing.assert_allclose(np.linalg.inv(rp),
                                   _matrix(O.rope_inverse, d, p, f), atol=1e-12)
        # Eq. (5) as the oracle evaluates it equals the single rotation by q - p
        x = np.random.default_rng(p).standard_normal((3, d))
        np.testing.assert_allclose(O.reposition_key(x, p, q, f),
                                   O.rope(x, q - p, f), atol=1e-12)


def pin_rope_relative():
    """<R(m) q, R(n) k> depends on m - n only."""
    rng = np.random.default_rng(2)
    f = O.inv_freq(128, 5.0e5)
    q, k = _rand(rng, 128), _rand(rng, 128)
    for m, n in ((10, 3), (1000, 993), (70000, 69993)):
        a = O.rope(q, m, f) @ O.rope(k, n, f)
        b = O.rope(q, m + 12345, f) @ O.rope(k, n + 12345, f)
        c = O.rope(q, m - n, f) @ k
        assert abs(a - b) < 1e-9 and abs(a - c) < 1e-9


# ---------------------------------------------------------------------------
# storage rounding
# ---------------------------------------------------------------------------

def pin_bf16_rounding():
    for _, x, want in _gold("bf16_rounding.json")["cases"]:
        assert O.rne_bf16(np.array([x]))[0] == want, (x, want)
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(200000) * 3).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.rne_bf16(x.astype(np.float64)), want)
    xf = rng.standard_normal(1000)
    np.testing.assert_array_equal(O.to_pool(xf, "fp32"),
                                  xf.astype(np.float32).astype(np.float64))


# ---------------------------------------------------------------------------
# cache operations
# ---------------------------------------------------------------------------

def _tiny_cache(dtype="f64", d=8, hq=4, hkv=2, theta=100.0, page=4):
    return O.OracleCache(hq, hkv, d, theta, dtype, layers=(0,), page_size=page)


def _tokens(rng, c, n):
    return (_rand(rng, 1, n, c.hkv, c.d), _rand(rng, 1, n, c.hkv, c.d))


def pin_fig10_positions():
    """The worked example of Figure 10: positions seen by each query."""
    g = _gold("fig10_positions.json")
    c = _tiny_cache()
    s = c.create()
    name_of = {}
    rng = np.random.default_rng(4)
    for op in g["ops"]:
        st = c.seqs[s]
        if op[0] == "append":
            name_of[st.n_logical] = op[1]
            k, v = _tokens(rng, c, 1)
            c.append(s, k, v)
        elif op[0] == "drop":
            idx = {n: i for i, n in name_of.items()}
            c.drop(s, [(idx[n], idx[n] + 1) for n in op[1]])
        elif op[0] == "repos":
            c.reposition(s)
        elif op[0] == "query":
            st = c.seqs[s]
            seen = {name_of[int(l)]: int(p)
                    for l, p, a in zip(st.logical, st.pos, st.alive) if a}
            assert seen == op[2], (op, seen)
            assert st.next_pos - 1 == op[2][op[1]]


def _replay(c, s, ops, toks):
    name_of = {}
    rng = np.random.default_rng(5)
    for op in ops:
        st = c.seqs[s]
        if op[0] == "append":
            name_of[st.n_logical] = op[1]
            k, v = _tokens(rng, c, 1)
            c.append(s, k, v, token_ids=[toks[op[1]]])
        elif op[0] == "drop":
            idx = {n: i for i, n in name_of.items()}
            c.drop(s, [(idx[n], idx[n] + 1) for n in op[1]])
        else:
            c.reposition(s)
    return name_of


def pin_fig5_histories():
    """Figure 5 / Figure 11: same survivors, different operation sequences."""
    g = _gold("fig5_histories.json")
    c = _tiny_cache()
    hist = {}
    for name, ops in g["paths"].items():
        s = c.create()
        name_of = _replay(c, s, ops, g["tokens"])
        st = c.seqs[s]
        act = [name_of[int(l)] for l, a in zip(st.logical, st.alive) if a]
        assert act == g["final_active"][name], (name, act)
        if name in g.get("final_positions", {}):
            pos = {name_of[int(l)]: int(p) for l, p, a in
                   zip(st.logical, st.pos, st.alive) if a}
            assert pos == g["final_positions"][name]
        hist[name] = c.history(s)
    names = list(hist)
    for i in range(len(names)):
        for j in range(i + 1, len(names)):
            assert hist[names[i]] != hist[names[j]], (names[i], names[j])
    # replaying the same path gives the same history; append n == n appends
    s1, s2 = c.create(), c.create()
    _replay(c, s1, g["paths"]["fig5_2"], g["tokens"])
    _replay(c, s2, g["paths"]["fig5_2"], g["tokens"])
    assert c.history(s1) == c.history(s2)
    a, b = c.create(), c.create()
    rng = np.random.default_rng(6)
    k, v = _tokens(rng, c, 5)
    c.append(a, k, v)
    c.append(b, k[:, :2], v[:, :2])
    c.append(b, k[:, 2:], v[:, 2:])
    assert c.history(a) == c.history(b)


def pin_drop_semantics():
    """Eq. (4): order, values, positions and the next position are unchanged."""
    rng = np.random.default_rng(7)
    c = _tiny_cache(dtype="bf16")
    s = c.create()
    k, v = _tokens(rng, c, 40)
    c.append(s, k, v)
    before = c.seqs[s]
    K0, V0, P0 = before.K.copy(), before.V.copy(), before.pos.copy()
    c.drop(s, [(3, 9), (20, 21), (5, 12), (39, 40), (7, 7)])
    st = c.seqs[s]
    np.testing.assert_array_equal(st.K, K0)
    np.testing.assert_array_equal(st.V, V0)
    np.testing.assert_array_equal(st.pos, P0)
    assert st.next_pos == 40 and st.n_logical == 40
    dead = set(range(3, 12)) | {20, 39}
    assert [i for i in range(40) if not st.alive[i]] == sorted(dead)
    c.drop(s, [(3, 9)])                 # already dropped: no state change
    assert int(st.alive.sum()) == 40 - len(dead)
    for bad in ([(0, 41)], [(-1, 2)], [(5, 4)]):
        with pytest.raises(O.OracleError):
            c.drop(s, bad)


def pin_reposition_positions_and_gather():
    """Survivors move to 0..r-1 in logical order; gather map = brute force."""
    rng = np.random.default_rng(8)
    for trial in range(30):
        c = _tiny_cache(dtype="f64")
        s = c.create()
        n = int(rng.integers(1, 90))
        k, v = _tokens(rng, c, n)
        c.append(s, k, v)
        for _ in range(int(rng.integers(0, 4))):
            b = int(rng.integers(0, n))
            c.drop(s, [(b, int(rng.integers(b, n + 1)))])
        st = c.seqs[s]
        alive = st.alive.copy()
        logical = st.logical.copy()
        V0 = st.V.copy()
        # brute force: walk the keep mask, counting survivors
        brute = []
        for i in range(len(alive)):
            if alive[i]:
                brute.append(i)
        pages = sorted({i // c.page_size for i in brute})
        np.testing.assert_array_equal(c.active_pages(s), pages)
        c.reposition(s)
        st = c.seqs[s]
        r = len(brute)
        np.testing.assert_array_equal(st.last_gather, brute)
        np.testing.assert_array_equal(st.pos, np.arange(r))
        np.testing.assert_array_equal(st.logical, logical[brute])
        np.testing.assert_array_equal(st.V, V0[:, brute])   # V copied, bit-exact
        assert st.next_pos == r and st.alive.all()


def pin_no_drop_unchanged():
    """With nothing dropped a reposition leaves every key bit-identical."""
    rng = np.random.default_rng(9)
    for dtype in ("bf16", "fp32", "f64"):
        c = _tiny_cache(dtype=dtype)
        s = c.create()
        k, v = _tokens(rng, c, 33)
        c.append(s, k, v)
        K0 = c.seqs[s].K.copy()
        c.reposition(s)
        np.testing.assert_array_equal(c.seqs[s].K, K0)
        np.testing.assert_array_equal(c.seqs[s].last_gather, np.arange(33))


def _dense_attention(q, keys, vals, pos_q, pos_k, freq, group):
    """Textbook attention with keys rotated by the complex form, scipy softmax."""
    d = q.shape[-1]

    def rot(x, p):
        z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * np.exp(1j * np.multiply.outer(p, freq))
        return np.concatenate([z.real, z.imag], axis=-1)

    out = np.zeros_like(q)
    for h in range(q.shape[0]):
        qr = rot(q[h], pos_q)
        kr = rot(keys[:, h // group], pos_k)
        w = scipy.special.softmax(kr @ qr / np.sqrt(d))
        out[h] = w @ vals[:, h // group]
    return out


def pin_attention_textbook():
    """No drop: attention equals dense softmax attention (GQA, 1/sqrt(D))."""
    rng = np.random.default_rng(10)
    c = _tiny_cache(dtype="f64", d=16, hq=8, hkv=2, theta=1.0e4)
    s = c.create()
    n = 23
    k, v = _tokens(rng, c, n)
    c.append(s, k, v)
    q = _rand(rng, 1, 8, 16)
    got = c.attention(0, q, [s])[0]
    want = _dense_attention(q[0], k[0], v[0], n - 1, np.arange(n), c.freq, 4)
    np.testing.assert_allclose(got, want, atol=1e-12)


def pin_repositioned_equals_direct():
    """Attention on a repositioned cache == survivors encoded at 0..r-1 directly."""
    rng = np.random.default_rng(11)
    for trial in range(10):
        c = _tiny_cache(dtype="f64", d=16, hq=4, hkv=2, theta=1.0e4)
        a = c.create()
        n = int(rng.integers(20, 120))
        k, v = _tokens(rng, c, n)
        c.append(a, k, v)
        b0 = int(rng.integers(0, n - 5))
        c.drop(a, [(b0, b0 + int(rng.integers(1, 5)))])
        c.drop(a, [(int(rng.integers(0, n)), n - 2)])
        keep = c.seqs[a].alive.copy()
        c.reposition(a)
        kq, vq = _tokens(rng, c, 1)
        c.append(a, kq, vq)
        b = c.create()
        c.append(b, k[:, keep], v[:, keep])
        c.append(b, kq, vq)
        q = _rand(rng, 1, 4, 16)
        np.testing.assert_allclose(c.attention(0, q, [a]), c.attention(0, q, [b]),
                                   atol=1e-10)


def pin_shift_invariance():
    """Shifting the query and all keys by the same offset changes nothing."""
    rng = np.random.default_rng(12)
    c = _tiny_cache(dtype="f64", d=16, hq=4, hkv=2, theta=1.0e4)
    n, shift = 30, 777
    k, v = _tokens(rng, c, n)
    a = c.create()
    c.append(a, k, v)
    b = c.create()
    kp, vp = _tokens(rng, c, shift)
    c.append(b, kp, vp)
    c.drop(b, [(0, shift)])          # positions of what follows start at `shift`
    c.append(b, k, v)
    q = _rand(rng, 1, 4, 16)
    np.testing.assert_allclose(c.attention(0, q, [a]), c.attention(0, q, [b]),
                               atol=1e-10)


def pin_empty_active_set():
    rng = np.random.default_rng(13)
    c = _tiny_cache()
    s = c.create()
    k, v = _tokens(rng, c, 5)
    c.append(s, k, v)
    c.drop(s, [(0, 5)])
    assert np.all(c.attention(0, _rand(rng, 1, 4, 8), [s]) == 0)
    c.reposition(s)
    assert c.info(s)["n_held"] == 0 and c.seqs[s].next_pos == 0


def pin_input_values_exact():
    """Generated inputs are exactly representable in the pool dtype."""
    for w, dt in ((synth.WIDTH_BF16, "bf16"), (synth.WIDTH_FP32, "fp32")):
        x = synth.block(7, 1, synth.KIND_K, 0, 12345, 50000, w).astype(np.float64)
        np.testing.assert_array_equal(O.to_pool(x, dt), x)
        assert abs(x.mean()) < 0.02 and abs(x.var() - 1) < 0.03


def pin_partial_rope():
    """Partial RoPE: the first R dims rotate with frequencies over R (complex
    form), the other D - R dims are untouched; a reposition copies them."""
    rng = np.random.default_rng(14)
    d, r, theta = 128, 64, 1.0e4
    f = O.inv_freq(r, theta)
    assert f.shape == (32,) and abs(f[8] - theta ** -0.25) < 1e-15
    x = _rand(rng, 5, d)
    pos = np.array([0, 3, 100, 4095, 70000])
    got = O.rope(x, pos, f)
    z = (x[:, : r // 2] + 1j * x[:, r // 2: r]) * np.exp(1j * pos[:, None] * f)
    np.testing.assert_allclose(got[:, :r], np.concatenate([z.real, z.imag], axis=1), atol=1e-12)
    np.testing.assert_array_equal(got[:, r:], x[:, r:])
    np.testing.assert_allclose(O.reposition_key(x, 900, 17, f), O.rope(x, 17 - 900, f), atol=1e-12)
    c64 = O.OracleCache(4, 2, d, theta, "f64", layers=(0,), page_size=16, rope_dim=r)
    sid = c64.create()
    k = _rand(rng, 1, 9, 2, d)
    c64.append(sid, k, k)
    ang = np.arange(9)[:, None, None] * (theta ** (-2.0 * np.arange(r // 2) / r))
    z = (k[0, ..., : r // 2] + 1j * k[0, ..., r // 2: r]) * np.exp(1j * ang)
    np.testing.assert_allclose(c64.seqs[sid].K[0, ..., :r],
                               np.concatenate([z.real, z.imag], axis=-1), atol=1e-12)
    c = O.OracleCache(4, 2, d, theta, "bf16", layers=(0,), page_size=16, rope_dim=r)
    sid = c.create()
    k, v = _rand(rng, 1, 40, 2, d), _rand(rng, 1, 40, 2, d)
    c.append(sid, k, v)
    before = c.seqs[sid].K.copy()
    c.drop(sid, [(0, 7)])
    c.reposition(sid)
    np.testing.assert_array_equal(c.seqs[sid].K[..., r:], before[:, 7:, :, r:])


def pin_sliding_window():
    """A window covers positions (p - W, p]: W larger than the sequence is
    full attention; W = 1 reads only the query's own token; with position
    gaps left by a drop the window holds fewer keys; any W equals textbook
    attention over exactly the keys whose positions fall in the window."""
    rng = np.random.default_rng(15)
    c = _tiny_cache(dtype="f64", d=16, hq=4, hkv=2, theta=1.0e4)
    s = c.create()
    n = 60
    k, v = _tokens(rng, c, n)
    c.append(s, k, v)
    q = _rand(rng, 1, 4, 16)
    full = c.attention(0, q, [s])
    np.testing.assert_allclose(c.attention(0, q, [s], window=n + 5), full, atol=1e-14)
    one = c.attention(0, q, [s], window=1)
    for h in range(4):
        np.testing.assert_allclose(one[0, h], v[0, n - 1, h // 2], atol=1e-14)
    c.drop(s, [(30, 55)])                         # gap: positions 30..54 inactive
    for w in (3, 8, 20, 31, 40):
        got = c.attention(0, q, [s], window=w)
        keep = [t for t in range(n) if not (30 <= t < 55) and t > n - 1 - w]
        want = _dense_attention(q[0], k[0][keep], v[0][keep], n - 1, np.array(keep),
                                c.freq, 2)
        np.testing.assert_allclose(got[0], want, atol=1e-12)


def pin_replay_attention():
    """Restore attention: a program of appends alone is plain causal softmax
    attention (textbook, scipy); the Figure 10 program gives each query the
    keys and positions the worked example lists."""
    rng = np.random.default_rng(16)
    c = _tiny_cache(dtype="f64", d=16, hq=4, hkv=2, theta=1.0e4)
    n = 25
    q = _rand(rng, 1, n, 4, 16)
    k, v = _tokens(rng, c, n)
    out, _ = c.replay_attention([("append", 10), ("append", 15)], q, k, v)
    for t in range(n):
        want = _dense_attention(q[0, t], k[0, : t + 1], v[0, : t + 1], t, np.arange(t + 1),
                                c.freq, 2)
        np.testing.assert_allclose(out[0, t], want, atol=1e-12)
    # Figure 10: A B C | drop B, repos | D | drop D | E | repos | F
    g = _gold("fig10_positions.json")
    names = [op[1] for op in g["ops"] if op[0] == "append"]
    idx = {name: i for i, name in enumerate(names)}
    program = []
    for op in g["ops"]:
        if op[0] == "append":
            program.append(("append", 1))
        elif op[0] == "drop":
            program.append(("drop", [(idx[x], idx[x] + 1) for x in op[1]]))
        elif op[0] == "repos":
            program.append(("repos",))
    m = len(names)
    q = _rand(rng, 1, m, 4, 16)
    k, v = _tokens(rng, c, m)
    out, _ = c.replay_attention(program, q, k, v)
    for op in g["ops"]:
        if op[0] != "query":
            continue
        x = idx[op[1]]
        seen = op[2]
        keys = [idx[nm] for nm in seen]
        pos = np.array([seen[nm] for nm in seen])
        want = _dense_attention(q[0, x], k[0][keys], v[0][keys], seen[op[1]], pos, c.freq, 2)
        np.testing.assert_allclose(out[0, x], want, atol=1e-12)


PINS = [pin_inv_freq, pin_partial_rope, pin_sliding_window, pin_replay_attention, pin_rope_complex_form, pin_rope_matrix_identities,
        pin_rope_relative, pin_bf16_rounding, pin_fig10_positions,
        pin_fig5_histories, pin_drop_semantics,
        pin_reposition_positions_and_gather, pin_no_drop_unchanged,
        pin_attention_textbook, pin_repositioned_equals_direct,
        pin_shift_invariance, pin_empty_active_set, pin_input_values_exact]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ---------------------------------------------------------------------------

def _bad_rope_sign(x, pos, freq):
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c + b * s, a * s + b * c], axis=-1)


def _bad_rope_interleaved(x, pos, freq):
    x = np.asarray(x, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def _bad_reposition_forward(k, p, q, freq):
    return O.rope(O.rope(k, p, freq), q, freq)          # R(q) R(p) instead of R(p)^-1


def _bad_scan_inclusive(flags):
    return np.cumsum(np.asarray(flags, dtype=np.int64))


def _bad_freq(head_dim, theta):
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -i / float(head_dim))


def _bad_bf16_truncate(x):
    u = np.ascontiguousarray(x, dtype=np.float64).view(np.uint64).copy()
    u &= ~np.uint64((1 << 45) - 1)
    return u.view(np.float64)


def _mutant_drop_shrinks(self, sid, ranges):
    _orig_drop(self, sid, ranges)
    s = self.seqs[sid]
    s.next_pos = int(s.alive.sum())


def _mutant_attention_no_scale(self, layer_index, q, sids):
    q = np.asarray(q, dtype=np.float64)
    return _orig_attention(self, layer_index, q * np.sqrt(self.d), sids)


def _mutant_gqa_modulo(self, layer_index, q, sids):
    out = np.zeros_like(np.asarray(q, dtype=np.float64))
    for i, sid in enumerate(sids):
        s = self.seqs[sid]
        qr = O.rope(q[i], np.full(self.hq, s.next_pos - 1), self.freq)
        act = np.flatnonzero(s.alive)
        for h in range(self.hq):
            kvh = h % self.hkv
            sc = s.K[layer_index, act, kvh] @ qr[h] / np.sqrt(self.d)
            w = np.exp(sc - sc.max())
            out[i, h] = (w @ s.V[layer_index, act, kvh]) / w.sum()
    return out


def _mutant_query_at_next_pos(self, layer_index, q, sids):
    for sid in sids:
        self.seqs[sid].next_pos += 1
    try:
        return _orig_attention(self, layer_index, q, sids)
    finally:
        for sid in sids:
            self.seqs[sid].next_pos -= 1


def _mutant_history_drops_merged_away(self, sid, ranges):
    _orig_drop(self, sid, ranges)
    log = self.seqs[sid].log
    if log and log[-1][0] == "drop":
        log.pop()


def _mutant_window_counts_tokens(self, layer_index, q, sids, window=0):
    if window <= 0:
        return _orig_attention(self, layer_index, q, sids)
    out = np.zeros(np.asarray(q).shape)
    for i, sid in enumerate(sids):
        s = self.seqs[sid]
        qr = O.rope(q[i], np.full(self.hq, s.next_pos - 1), self.freq)
        act = np.flatnonzero(s.alive)[-window:]       # the last W active tokens
        for h in range(self.hq):
            kvh = h // self.group
            sc = s.K[layer_index, act, kvh] @ qr[h] / np.sqrt(self.d)
            w = np.exp(sc - sc.max())
            out[i, h] = (w @ s.V[layer_index, act, kvh]) / w.sum()
    return out


_orig_drop = O.OracleCache.drop
_orig_attention = O.OracleCache.attention
_orig_init = O.OracleCache.__init__


def _mutant_partial_freq_over_d(self, *a, **kw):
    _orig_init(self, *a, **kw)
    self.freq = O.inv_freq(self.d, 1.0e4)[: self.rope_dim // 2]

MUTANTS = {
    "rope_sign": ("rope", _bad_rope_sign, None),
    "rope_interleaved_pairs": ("rope", _bad_rope_interleaved, None),
    "reposition_forward_rotation": ("reposition_key", _bad_reposition_forward, None),
    "scan_inclusive": (None, None, ("exclusive_scan", staticmethod(_bad_scan_inclusive))),
    "freq_exponent": ("inv_freq", _bad_freq, None),
    "bf16_truncation": ("rne_bf16", _bad_bf16_truncate, None),
    "drop_shrinks_next_pos": (None, None, ("drop", _mutant_drop_shrinks)),
    "attention_unscaled": (None, None, ("attention", _mutant_attention_no_scale)),
    "gqa_head_modulo": (None, None, ("attention", _mutant_gqa_modulo)),
    "query_position_off_by_one": (None, None, ("attention", _mutant_query_at_next_pos)),
    "history_forgets_drop": (None, None, ("drop", _mutant_history_drops_merged_away)),
    "window_counts_tokens": (None, None, ("attention", _mutant_window_counts_tokens)),
    "partial_rope_freq_over_d": (None, None, ("__init__", _mutant_partial_freq_over_d)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, monkeypatch):
    fn_name, fn, method = MUTANTS[name]
    if fn_name:
        monkeypatch.setattr(O, fn_name, fn)
    if method:
        monkeypatch.setattr(O.OracleCache, method[0], method[1])
    failed = []
    for pin in PINS:
        try:
            pin()
        except Exception:  # an assertion, or the mutant breaking outright
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {name}"
