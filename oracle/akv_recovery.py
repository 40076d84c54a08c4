"""Recovery planning for a restore: which tokens must be recomputed.

TEST INFRASTRUCTURE ONLY.  The tests call it; the library never does, and
this module imports nothing from the library.

Sources ("Cache Engineering for Agents" paper review = page 1; "[Repo Review]
AKV" = page 2):

* page 2, 5.4: a recovery plan closes, backwards, the dependencies of KV that
  later queries have to read but that is missing, and yields the query
  ranges to recompute; ranges in between that are still resident stay in use.
* page 1, 4.2.2 and A.1.1: a restored token's query reads the keys that were
  active when it was appended (tokens dropped later included), so its KV
  depends on exactly those.

Readings (the pages give no formula):

* A token's KV depends on the keys its query read when it was appended: the
  tokens appended before it and not dropped by then.  (A sliding window reads
  a subset of them; the set here is the safe superset for every layer.)
* Recomputing a token needs every key its query read: each one is resident or
  is recomputed as well.
* The tokens whose KV the next step reads ("need") are, unless given, the
  tokens active at the end of the program.
* The plan is the smallest set of tokens that holds every needed missing
  token and, with each token in it, every missing token its query read.
  Resident tokens are never in it.

The program is a list of ("append", n) | ("drop", ranges) | ("repos",), as in
``OracleCache.replay_attention``; ranges are logical [b, e) pairs.
"""


def replay_visibility(program):
    """Replay ``program`` from empty.  Returns (n_tokens, read, active_end):
    read[t] is the set of tokens before t that were active when t was
    appended; active_end the set of tokens active at the end."""
    active = []                   # tokens active now, in logical order
    read = []
    for op in program:
        if op[0] == "append":
            for _ in range(op[1]):
                t = len(read)
                read.append(set(active))
                active.append(t)
        elif op[0] == "drop":
            gone = set()
            for b, e in op[1]:
                if not 0 <= b <= e <= len(read):
                    raise ValueError(f"drop range [{b}, {e}) outside [0, {len(read)})")
                gone.update(range(b, e))
            active = [t for t in active if t not in gone]
        elif op[0] == "repos":
            pass                  # positions change; which tokens are active does not
        else:
            raise ValueError(f"unknown operation {op!r}")
    return len(read), read, set(active)


def plan_recovery(program, missing, need=None):
    """Tokens to recompute, in increasing order, and their maximal runs of
    consecutive tokens ("query segments", [b, e) pairs).

    ``missing``: tokens whose KV is not resident; ``need``: tokens whose KV
    the next step reads (None: the tokens active at the end of ``program``).
    The closure is taken with a work list, one token at a time."""
    n, read, active_end = replay_visibility(program)
    missing = set(missing)
    need = active_end if need is None else set(need)
    if any(not 0 <= t < n for t in missing | need):
        raise ValueError("token index outside the program")
    plan = set(need & missing)
    work = sorted(plan)
    while work:
        t = work.pop()
        for u in read[t]:
            if u in missing and u not in plan:
                plan.add(u)
                work.append(u)
    tokens = sorted(plan)
    segments = []
    for t in tokens:
        if segments and segments[-1][1] == t:
            segments[-1][1] = t + 1
        else:
            segments.append([t, t + 1])
    return tokens, [tuple(s) for s in segments]
