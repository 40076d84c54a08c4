"""Plain CPU oracle of history-keyed prefix sharing and drop-aware eviction.

TEST INFRASTRUCTURE ONLY.  The tests call it; the library never does, and
this module imports nothing from the library.

Sources ("Cache Engineering for Agents" paper review = page 1; "[Repo Review]
AKV" = page 2):

* context records -- page 2, 5.4: a cache prefix is compared as a list of
  token records and the event records in front of them, of the kinds TOKEN,
  DELTA and REPOSITION; page 1, 3.4, Eq. (6): the state is the operation
  sequence replayed from empty.
* exact and retrigger matching -- page 1, Appendix A.1.2 (Reposition Scheme):
  a token node T(x, p) carries the token id x and the position p of the key
  as it is stored now; an exact match needs equal token ids, positions and
  operation records; the projection phi removes the stored positions only,
  and a prefix whose projection matches can be reused after its keys are
  rotated to the wanted positions.  The longest valid exact prefix is the
  start; a compatible prefix is taken only when strictly longer (ties keep
  the exact one); the search stops at the first token or operation that
  differs.  Page 1, 4.2.3: same position -> reuse as is, compatible other
  position -> rotate the keys.  Figure 11: the operation records cannot be
  skipped to line up final positions.
* plan of the fork -- page 2, 5.4 (plan of occurrence materialisation):
  per needed token, reuse the stored version, or take a new slot and copy
  (rotating the key); a page handed to another branch is shared only when
  it is unchanged (copy-on-write).
* drop-aware eviction -- page 1, 4.2.2: storage is released only when no
  computation or restore needs it, one request's drop never frees KV that
  another uses, and dropped caches go before caches of finished requests;
  page 2, 5.6: two heaps look at edges that a drop has proven unneeded
  before ordinary leaves, and only the DELTA records of the path in
  question (proven_skip_ranges) may free an ancestor's KV.

Readings (the pages give no algorithm text beyond the above):

* Records of a program: one ("T", id) per appended token, one ("D", ranges)
  per drop with the sorted, merged, non-empty ranges it names (an empty drop
  is no record), one ("R",) per reposition.  Two records are equal when kind
  and contents are equal; phi-equality of record lists is plain equality,
  because positions are not part of a record: they follow from the records
  before it (Eq. 6).
* A published entry is a snapshot of a sequence at the end of its records.
  Its stored key of token t exists when t's slot is still held (t is alive,
  or was dropped after the last reposition) and t's page still holds an
  active token (a page with no active token is released at the drop); the
  key then sits at position = slot.
* A request prefix of n records (0 < n <= common length with the entry) is
  valid when every token active in the request's state after those n
  records has a stored key in the entry; it is exact when, in addition,
  every such key is stored at the position the request's state gives it.
  The positions compared are those of the active tokens (a dropped token is
  never read again).  Ties between entries: the lowest entry id for exact
  matches; fewer rotated keys, then the lowest entry id, for retrigger
  matches.
* Eviction order: entries that another entry extends (its records are a
  prefix of the other's) with a DELTA record after the shared prefix that
  drops a token active at the entry's end are "drop-proven" and go first,
  oldest use first; then leaves (no entry extends them), oldest use first;
  then the remaining ancestors, oldest use first; equal use times go by
  lower id.

Pins: ``tests/test_prefix_pins.py``.
"""


def records(program, token_ids):
    """Context records of an operation program applied to an empty sequence."""
    out = []
    t = 0
    for op in program:
        if op[0] == "append":
            for _ in range(op[1]):
                out.append(("T", int(token_ids[t])))
                t += 1
        elif op[0] == "drop":
            rs = sorted((int(b), int(e)) for b, e in op[1] if e > b)
            merged = []
            for b, e in rs:
                if merged and b <= merged[-1][1]:
                    merged[-1] = (merged[-1][0], max(merged[-1][1], e))
                else:
                    merged.append((b, e))
            if merged:
                out.append(("D", tuple(merged)))
        else:
            out.append(("R",))
    if t != len(token_ids):
        raise ValueError("program appends %d tokens, %d ids given" % (t, len(token_ids)))
    return out


class State:
    """Sequence state after a list of records (Eq. 3-6 replayed):
    per logical token its active flag, its position (== its slot while held)
    and whether its slot is held; plus the next position."""

    def __init__(self, recs):
        self.alive, self.pos, self.held = [], [], []
        self.next_pos = 0
        for r in recs:
            self.apply(r)

    def apply(self, r):
        if r[0] == "T":
            self.alive.append(True)
            self.pos.append(self.next_pos)
            self.held.append(True)
            self.next_pos += 1
        elif r[0] == "D":
            for b, e in r[1]:
                if e > len(self.alive):
                    raise ValueError("drop past the appended tokens")
                for t in range(b, e):
                    self.alive[t] = False
        else:
            j = 0
            for t in range(len(self.alive)):
                self.held[t] = self.alive[t]
                if self.alive[t]:
                    self.pos[t] = j
                    j += 1
            self.next_pos = j

    def stored(self, page_size):
        """Logical token -> position of its stored key, for the tokens whose
        key still exists (slot held, page holding an active token)."""
        live_pages = {self.pos[t] // page_size for t in range(len(self.alive)) if self.alive[t]}
        return {t: self.pos[t] for t in range(len(self.alive))
                if self.held[t] and self.pos[t] // page_size in live_pages}


def common_length(a, b):
    n = 0
    while n < len(a) and n < len(b) and a[n] == b[n]:
        n += 1
    return n


def match(entries, req, page_size):
    """Best reuse of the published ``entries`` ({id: records}) for the
    request records ``req``.  Returns dict(kind in {"none", "exact",
    "retrigger"}, entry, n_records, n_tokens, n_rotated)."""
    best_exact = None      # (n, -id)
    best_valid = None      # (n, -rotated, -id)
    for eid in sorted(entries):
        recs = entries[eid]
        m = common_length(recs, req)
        stored = State(recs).stored(page_size)
        for n in range(1, m + 1):
            st = State(req[:n])
            need = [t for t in range(len(st.alive)) if st.alive[t]]
            if any(t not in stored for t in need):
                continue
            rotated = sum(1 for t in need if stored[t] != st.pos[t])
            if rotated == 0:
                if best_exact is None or (n, -eid) > best_exact:
                    best_exact = (n, -eid)
            cand = (n, -rotated, -eid)
            if best_valid is None or cand > best_valid:
                best_valid = cand
    none = dict(kind="none", entry=-1, n_records=0, n_tokens=0, n_rotated=0)
    if best_valid is None:
        return none
    if best_exact is not None and best_exact[0] >= best_valid[0]:
        n, eid, kind, rot = best_exact[0], -best_exact[1], "exact", 0
    else:
        n, eid, kind, rot = best_valid[0], -best_valid[2], "retrigger", -best_valid[1]
    n_tok = sum(1 for r in req[:n] if r[0] == "T")
    return dict(kind=kind, entry=eid, n_records=n, n_tokens=n_tok, n_rotated=rot)


def fork_plan(entry_recs, req, n, page_size):
    """Materialisation of the request prefix req[:n] from an entry: the new
    sequence's held slots, its active tokens (logical t -> (dst slot,
    src slot in the entry, delta = dst - src)), and per destination page
    whether it is the entry's page (shared, unchanged) or a fresh copy.
    Raises ValueError when the prefix is not valid for the entry."""
    st = State(req[:n])
    stored = State(entry_recs).stored(page_size)
    moves = {}
    for t in range(len(st.alive)):
        if st.alive[t]:
            if t not in stored:
                raise ValueError("token %d has no stored key in the entry" % t)
            moves[t] = (st.pos[t], stored[t], st.pos[t] - stored[t])
    n_pages = -(-st.next_pos // page_size)
    pages = []
    for k in range(n_pages):
        inside = [mv for mv in moves.values() if mv[0] // page_size == k]
        if not inside:
            pages.append("none")
        elif all(dst == src for dst, src, _ in inside):
            pages.append("shared")
        else:
            pages.append("fresh")
    return dict(n_slots=st.next_pos, n_logical=len(st.alive), moves=moves, pages=pages,
                alive=list(st.alive))


def evict_order(entries, last_use):
    """Order in which published entries are evicted (ids)."""
    ids = sorted(entries)
    klass = {}
    for a in ids:
        ra = entries[a]
        ext = [b for b in ids if b != a and len(entries[b]) > len(ra) and entries[b][:len(ra)] == ra]
        if not ext:
            klass[a] = 1
            continue
        st = State(ra)
        active = {t for t in range(len(st.alive)) if st.alive[t]}
        proven = False
        for b in ext:
            for r in entries[b][len(ra):]:
                if r[0] == "D" and any(bb <= t < ee for bb, ee in r[1] for t in active):
                    proven = True
        klass[a] = 0 if proven else 2
    return sorted(ids, key=lambda e: (klass[e], last_use[e], e))
