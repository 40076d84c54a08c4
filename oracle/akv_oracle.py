"""Plain, slow fp64 CPU oracle of the active-KV cache operations.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` call it; the library never does, and this
module imports nothing from the library (it takes its inputs from the seeded
generators in ``workloads`` only).

Sources ("Cache Engineering for Agents" paper review = page 1; "[Repo Review]
AKV" = page 2):

* append -- page 1, 3.3 Cache Operations, Eq. (3): the new token's KV is
  concatenated to the active cache in logical order; its key is encoded at
  the next position.
* drop(P) -- page 1, 3.3, Eq. (4): the KV at logical indices P leaves all
  future attention; order, values, positions and the next position of the
  rest are unchanged (page 1, "three operations and position encoding").
* reposition -- page 1, 3.3, Eq. (5): K' = R(q) R(p)^-1 K with p the current
  encoded position and q the target; the r survivors take positions 0..r-1
  in logical order and the next append lands at r; V is not recomputed.
  Page 2, 5.5: the inverse rotation and the new rotation are applied to the
  stored key and the result is stored again; a key whose position does not
  change is copied as it is (no rotation round trip).
* operation sequence -- page 1, 3.4, Eq. (6): the state is the result of the
  operation sequence replayed from empty; m counts operations.
* attention -- plain softmax attention of one query over the active keys
  (the pages' decode reads the active KV only; page 1, A.4.1).
* restore attention -- page 1, 4.2.2, 4.2.3 and A.1.1 (segment-batch
  attention): a restore recomputes every token of an operation program in
  one forward and must give each token the attention it had originally --
  over the keys active when it was appended (including ones dropped later),
  at the positions of that time.  ``replay_attention`` is the definition:
  replay the program, and after each appended token take its query's
  attention over the active cache (the token included).

Readings where the pages are silent or garbled (the display formulas of
Eqs. 3-6 did not survive extraction):

* RoPE is the half-split form: the pairs are (i, i + R/2), i < R/2, with
  frequency f_i = theta^(-2 i / R); R(p) maps (x, y) to
  (x cos(p f_i) - y sin(p f_i), x sin(p f_i) + y cos(p f_i)).  R is the
  rotary width: the full head dim, or the first R dims for partial RoPE,
  whose other dims are not rotated and are copied by a reposition
  ("[Repo Review] AKV", 5.5).
* Sliding-window attention counts positions, not active tokens: with
  position gaps left by a drop, the read range of a query is still the
  window of positions ending at the query ("[Repo Review] AKV", 5.5).
* P is a set of logical (trajectory) indices, assigned at append and never
  renumbered; dropping an index already dropped is a no-op.
* The keys are stored in the pool's dtype: every write of a key (append,
  reposition) rounds the exact fp64 result to that dtype, round to nearest
  even.  Page 1 A.1.3 names a BF16 pool.
* The decode query is rotated to the position of the sequence's last
  appended token (next position - 1); scores are scaled by 1/sqrt(D); query
  head h reads KV head floor(h / (Hq/Hkv)).  With no active key the output
  is zero.
* The history is the operation sequence itself: one record per appended
  token (with its token id, or None), one record per drop carrying the
  sorted, merged, non-empty set of ranges it names (an empty drop is no
  operation), and one record per reposition.

"Held" tokens are the ones that a storage must still hold: everything since
the last reposition, dropped or not.  Their list index is the slot, so the
keep mask, the exclusive-scan gather map and the page list are all defined
over it.

Parity pins live in ``tests/test_oracle_pins.py``; every function here is
pinned there (no function is "parity unpinned").
"""
import bisect
import copy

import numpy as np


# ---------------------------------------------------------------------------
# rotary position embedding
# ---------------------------------------------------------------------------

def inv_freq(rope_dim, theta):
    """f_i = theta^(-2 i / R) for i in [0, R/2), in fp64 (R = rotary dims)."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / float(rope_dim))


def rope(x, pos, freq):
    """R(pos) x on the last axis.

    The rotary part is the first R = 2 len(freq) dims, in half-split pairs
    (i, i + R/2); dims R.. pass through (partial RoPE).  ``x`` is [..., D];
    ``pos`` broadcasts against ``x[..., 0]``.
    """
    x = np.asarray(x, dtype=np.float64)
    h = len(freq)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :h], x[..., h:2 * h]
    return np.concatenate([a * c - b * s, a * s + b * c, x[..., 2 * h:]], axis=-1)


def rope_inverse(x, pos, freq):
    """R(pos)^-1 x = R(pos)^T x."""
    x = np.asarray(x, dtype=np.float64)
    h = len(freq)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :h], x[..., h:2 * h]
    return np.concatenate([a * c + b * s, -a * s + b * c, x[..., 2 * h:]], axis=-1)


def reposition_key(k, p, q, freq):
    """Eq. (5): K' = R(q) R(p)^-1 K, evaluated in that order in fp64."""
    return rope(rope_inverse(k, p, freq), q, freq)


# ---------------------------------------------------------------------------
# storage precision
# ---------------------------------------------------------------------------

def rne_bf16(x):
    """Round fp64 values to the nearest bfloat16, ties to even (as fp64).

    bfloat16 keeps 8 significant bits, so 45 of fp64's 53 are rounded off.
    Finite, normal inputs only (the pool holds moderate values).
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    u = x.view(np.uint64).copy()
    drop = np.uint64(45)
    lsb = (u >> drop) & np.uint64(1)
    with np.errstate(over="ignore"):
        u = u + (np.uint64((1 << 44) - 1) + lsb)
    u &= ~np.uint64((1 << 45) - 1)
    return u.view(np.float64)


def to_pool(x, dtype):
    """Value of ``x`` once stored in a pool of ``dtype`` ('bf16'|'fp32'|'f64')."""
    if dtype == "bf16":
        return rne_bf16(x)
    if dtype == "fp32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if dtype == "f64":
        return np.asarray(x, dtype=np.float64).copy()
    raise ValueError(dtype)


# ---------------------------------------------------------------------------
# cache state
# ---------------------------------------------------------------------------

class OracleError(Exception):
    pass


def _merge_ranges(ranges):
    rs = sorted((int(b), int(e)) for b, e in ranges if int(e) > int(b))
    out = []
    for b, e in rs:
        if out and b <= out[-1][1]:
            out[-1] = (out[-1][0], max(out[-1][1], e))
        else:
            out.append((b, e))
    return tuple(out)


class OracleSeq:
    def __init__(self, n_layers, hkv, d):
        self.logical = np.zeros(0, dtype=np.int64)
        self.alive = np.zeros(0, dtype=bool)
        self.pos = np.zeros(0, dtype=np.int64)
        self.K = np.zeros((n_layers, 0, hkv, d))
        self.V = np.zeros((n_layers, 0, hkv, d))
        self.next_pos = 0
        self.n_logical = 0
        self.log = []
        self.last_gather = None


class OracleCache:
    """Active-KV state of many sequences, for a chosen subset of layers.

    ``layers`` lists the model layers this instance tracks (every layer's
    computation is independent of the others, so a subset is exact for the
    layers it holds).  Arrays passed to ``append`` and ``attention`` carry
    only these layers, in this order.
    """

    def __init__(self, hq, hkv, head_dim, rope_theta, pool_dtype, layers=(0,),
                 page_size=16, rope_dim=0):
        if hq % hkv:
            raise OracleError("hq must be a multiple of hkv")
        self.hq, self.hkv, self.d = hq, hkv, head_dim
        self.group = hq // hkv
        self.layers = list(layers)
        self.rope_dim = rope_dim or head_dim
        self.freq = inv_freq(self.rope_dim, rope_theta)
        self.dtype = pool_dtype
        self.page_size = page_size
        self.seqs = {}
        self._next_id = 0

    # -- sequences ---------------------------------------------------------
    def create(self):
        sid = self._next_id
        self._next_id += 1
        self.seqs[sid] = OracleSeq(len(self.layers), self.hkv, self.d)
        return sid

    def fork(self, parent):
        sid = self._next_id
        self._next_id += 1
        self.seqs[sid] = copy.deepcopy(self.seqs[parent])
        return sid

    def free(self, sid):
        del self.seqs[sid]

    # -- Eq. (3) -------------------------------------------------------------
    def append(self, sid, k_raw, v, token_ids=None):
        """Append n tokens: ``k_raw``, ``v`` are [layers][n][Hkv][D] (pre-RoPE K)."""
        s = self.seqs[sid]
        k_raw = np.asarray(k_raw, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        n = k_raw.shape[1]
        pos = s.next_pos + np.arange(n, dtype=np.int64)
        k_new = to_pool(rope(k_raw, pos[None, :, None], self.freq), self.dtype)
        v_new = to_pool(v, self.dtype)
        s.K = np.concatenate([s.K, k_new], axis=1)
        s.V = np.concatenate([s.V, v_new], axis=1)
        s.logical = np.concatenate(
            [s.logical, s.n_logical + np.arange(n, dtype=np.int64)])
        s.alive = np.concatenate([s.alive, np.ones(n, dtype=bool)])
        s.pos = np.concatenate([s.pos, pos])
        s.next_pos += n
        s.n_logical += n
        for t in range(n):
            s.log.append(("append", None if token_ids is None else int(token_ids[t])))

    # -- Eq. (4) -------------------------------------------------------------
    def drop(self, sid, ranges):
        s = self.seqs[sid]
        for b, e in ranges:
            if b < 0 or e < b or e > s.n_logical:
                raise OracleError(f"bad range [{b}, {e}) for {s.n_logical} tokens")
        canon = _merge_ranges(ranges)
        if not canon:
            return
        for b, e in canon:
            s.alive &= ~((s.logical >= b) & (s.logical < e))
        s.log.append(("drop", canon))

    # -- Eq. (5) -------------------------------------------------------------
    @staticmethod
    def exclusive_scan(flags):
        """Exclusive prefix sum of 0/1 flags: the output slot of each kept item."""
        f = np.asarray(flags, dtype=np.int64)
        return np.cumsum(f) - f

    def reposition(self, sid):
        s = self.seqs[sid]
        dst = self.exclusive_scan(s.alive)
        r = int(s.alive.sum())
        gather = np.zeros(r, dtype=np.int64)
        src = np.flatnonzero(s.alive)
        gather[dst[src]] = src
        q = np.arange(r, dtype=np.int64)
        p = s.pos[gather]
        k_old = s.K[:, gather]
        k_new = to_pool(reposition_key(k_old, p[None, :, None], q[None, :, None],
                                       self.freq), self.dtype)
        same = p == q
        k_new[:, same] = k_old[:, same]
        s.K = k_new
        s.V = s.V[:, gather].copy()
        s.logical = s.logical[gather]
        s.alive = np.ones(r, dtype=bool)
        s.pos = q
        s.next_pos = r
        s.last_gather = gather
        s.log.append(("repos",))

    # -- attention -------------------------------------------------------------
    def attention(self, layer_index, q, sids, window=0):
        """Decode attention for each sequence: ``q`` is [n][Hq][D] (pre-RoPE).

        ``window`` > 0: sliding window over positions -- the query at
        position p reads the active keys whose position lies in (p - window, p]
        (with positions left sparse by a drop, fewer than ``window`` keys).
        """
        q = np.asarray(q, dtype=np.float64)
        out = np.zeros(q.shape, dtype=np.float64)
        for i, sid in enumerate(sids):
            s = self.seqs[sid]
            p = s.next_pos - 1
            qr = rope(q[i], np.full(self.hq, p), self.freq)
            visible = s.alive if window <= 0 else s.alive & (s.pos > p - window)
            act = np.flatnonzero(visible)
            if act.size == 0:
                continue
            for h in range(self.hq):
                kvh = h // self.group
                kk = s.K[layer_index, act, kvh]
                vv = s.V[layer_index, act, kvh]
                sc = kk @ qr[h] / np.sqrt(self.d)
                w = np.exp(sc - sc.max())
                out[i, h] = (w @ vv) / w.sum()
        return out

    # -- restore (segment-batch attention), by replay ------------------------------
    def replay_attention(self, program, q, k_raw, v, window=0, only=None):
        """Attention output of every appended token of ``program``, as it was
        when the token was appended.

        ``program`` is a list of ("append", n) | ("drop", ranges) | ("repos",)
        applied to a fresh sequence; ``q``, ``k_raw``, ``v`` are
        [layers][T][heads][D] for the T appended tokens in order.  Returns
        [layers][T][Hq][D].  The sequence is left in its final state.
        With ``only`` (increasing token indices), just those tokens' outputs
        are computed: ``q`` then holds only their rows, [layers][len(only)],
        and so does the result.
        """
        q = np.asarray(q, dtype=np.float64)
        sid = self.create()
        out = np.zeros(q.shape[:2] + (self.hq, self.d))
        row = {t: i for i, t in enumerate(only)} if only is not None else None
        stops = sorted(row) if row is not None else None
        t = 0
        for op in program:
            if op[0] == "append":
                end = t + op[1]
                while t < end:
                    # append up to the next token whose output is wanted
                    stop = t + 1
                    if stops is not None:
                        j = bisect.bisect_left(stops, t)
                        stop = stops[j] + 1 if j < len(stops) and stops[j] < end else end
                    self.append(sid, k_raw[:, t:stop], v[:, t:stop])
                    t = stop
                    i = t - 1 if row is None else row.get(t - 1)
                    if i is not None:
                        for li in range(len(self.layers)):
                            out[li, i] = self.attention(li, q[li, i:i + 1], [sid], window)[0]
            elif op[0] == "drop":
                self.drop(sid, op[1])
            else:
                self.reposition(sid)
        return out, sid

    # -- introspection ---------------------------------------------------------
    def info(self, sid):
        s = self.seqs[sid]
        return dict(n_logical=s.n_logical, n_held=int(s.alive.size),
                    n_alive=int(s.alive.sum()), next_pos=s.next_pos,
                    n_pages=-(-int(s.alive.size) // self.page_size),
                    n_active_pages=int(self.active_pages(sid).size))

    def active_pages(self, sid):
        """Indices of the pages (of held slots) that hold at least one active token."""
        s = self.seqs[sid]
        return np.unique(np.flatnonzero(s.alive) // self.page_size)

    def history(self, sid):
        return tuple(self.seqs[sid].log)
