"""Thin ctypes binding of include/akv.h: the same names, argument marshalling only.

Every function raises :class:`AkvError` on a non-zero return code.  Pointers
are plain integers (``tensor.data_ptr()``); host arrays are numpy arrays.  All
computation happens in the CUDA library; if it is not built or cannot be
loaded, :func:`lib` raises -- there is no fallback.
"""
import ctypes
import os

import numpy as np

from . import _build

AKV_OK = 0
AKV_EINVAL = -1
AKV_ERANGE = -2
AKV_ENOSEQ = -3
AKV_ENOPAGES = -4
AKV_ECAPACITY = -5
AKV_ECUDA = -6
AKV_EDEVICE = -7
AKV_NOALLOC_SCRATCH_BYTES = 8 << 20   # the allocation-free decode's device array
AKV_NOALLOC_MAX_SEQS = 256
AKV_DTYPE_BF16 = 0
AKV_DTYPE_FP32 = 1
AKV_DERR_PAGE = 0x1
AKV_DERR_INDEX = 0x2
AKV_DERR_WAIT = 0x4
AKV_DERR_COUNT = 0x8

_NAMES = {AKV_EINVAL: "AKV_EINVAL", AKV_ERANGE: "AKV_ERANGE", AKV_ENOSEQ: "AKV_ENOSEQ",
          AKV_ENOPAGES: "AKV_ENOPAGES", AKV_ECAPACITY: "AKV_ECAPACITY",
          AKV_ECUDA: "AKV_ECUDA", AKV_EDEVICE: "AKV_EDEVICE"}


class AkvError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{_NAMES.get(code, code)}: {msg}")
        self.code = code


class AkvConfig(ctypes.Structure):
    """struct akv_config"""
    _fields_ = [("layers", ctypes.c_int32), ("phys_layers", ctypes.c_int32),
                ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("max_seqs", ctypes.c_int32), ("max_slots", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rope_dim", ctypes.c_int32)]


class AkvOp(ctypes.Structure):
    """struct akv_op"""
    _fields_ = [("kind", ctypes.c_int32), ("count", ctypes.c_int32),
                ("ranges", ctypes.POINTER(ctypes.c_int64))]


AKV_OP_APPEND, AKV_OP_DROP, AKV_OP_REPOS = 0, 1, 2
AKV_MATCH_NONE, AKV_MATCH_EXACT, AKV_MATCH_RETRIGGER = 0, 1, 2
MATCH_KINDS = {AKV_MATCH_NONE: "none", AKV_MATCH_EXACT: "exact", AKV_MATCH_RETRIGGER: "retrigger"}


class AkvPrefixMatch(ctypes.Structure):
    """struct akv_prefix_match_t"""
    _fields_ = [("kind", ctypes.c_int32), ("n_records", ctypes.c_int32),
                ("entry", ctypes.c_int64), ("n_tokens", ctypes.c_int32),
                ("n_rotated", ctypes.c_int32), ("op_index", ctypes.c_int32),
                ("op_tokens", ctypes.c_int32)]

    def as_dict(self):
        return dict(kind=MATCH_KINDS[self.kind], entry=self.entry, n_records=self.n_records,
                    n_tokens=self.n_tokens, n_rotated=self.n_rotated, op_index=self.op_index,
                    op_tokens=self.op_tokens)


class AkvSeqInfo(ctypes.Structure):
    """struct akv_seq_info_t"""
    _fields_ = [("n_logical", ctypes.c_int64), ("n_held", ctypes.c_int64),
                ("n_active", ctypes.c_int64), ("next_pos", ctypes.c_int64),
                ("n_pages", ctypes.c_int32), ("n_active_pages", ctypes.c_int32),
                ("n_owned_pages", ctypes.c_int32), ("n_shared_pages", ctypes.c_int32)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_}


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_PI32 = ctypes.POINTER(ctypes.c_int32)
_PI64 = ctypes.POINTER(ctypes.c_int64)

# name -> (restype, argtypes): the whole exported surface of akv.h
SIGNATURES = {
    "akv_pool_bytes": (ctypes.c_size_t, [ctypes.POINTER(AkvConfig)]),
    "akv_cache_create": (ctypes.c_int, [ctypes.POINTER(AkvConfig), _P, _P, ctypes.c_size_t,
                                        _P, ctypes.POINTER(_P)]),
    "akv_cache_destroy": (ctypes.c_int, [_P]),
    "akv_set_stream": (ctypes.c_int, [_P, _P]),
    "akv_seq_create": (ctypes.c_int, [_P, _PI64]),
    "akv_seq_fork": (ctypes.c_int, [_P, _I64, _PI64]),
    "akv_seq_free": (ctypes.c_int, [_P, _I64]),
    "akv_append": (ctypes.c_int, [_P, _PI64, _PI32, _I32, _P, _P, _PI32]),
    "akv_drop": (ctypes.c_int, [_P, _I64, _PI64, _I32]),
    "akv_reposition": (ctypes.c_int, [_P, _PI64, _I32]),
    "akv_decode_attention": (ctypes.c_int, [_P, _I32, _P, _PI64, _I32, _P]),
    "akv_seq_info": (ctypes.c_int, [_P, _I64, ctypes.POINTER(AkvSeqInfo)]),
    "akv_seq_positions": (ctypes.c_int, [_P, _I64, _PI32]),
    "akv_seq_keep_mask": (ctypes.c_int, [_P, _I64, ctypes.POINTER(ctypes.c_uint8)]),
    "akv_seq_logical": (ctypes.c_int, [_P, _I64, _PI64]),
    "akv_seq_gather_map": (ctypes.c_int, [_P, _I64, _PI32, _PI64]),
    "akv_seq_page_table": (ctypes.c_int, [_P, _I64, _PI32, _PI32, _PI32, _PI32]),
    "akv_seq_host_pages": (ctypes.c_int, [_P, _I64, _PI32, _PI32]),
    "akv_history_key": (ctypes.c_int, [_P, _I64, ctypes.POINTER(ctypes.c_uint64)]),
    "akv_page_refcount": (ctypes.c_int, [_P, _I32, _PI32]),
    "akv_pool_stats": (ctypes.c_int, [_P, _PI32, _PI32]),
    "akv_last_error": (ctypes.c_char_p, [_P]),
    "akv_sync_errors": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "akv_kernel_launches": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint64)]),
    "akv_set_decode_waves": (ctypes.c_int, [_P, _I32]),
    "akv_set_restore_tensor_cores": (ctypes.c_int, [_P, _I32]),
    "akv_set_decode_sharing": (ctypes.c_int, [_P, _I32]),
    "akv_decode_plan_stats": (ctypes.c_int, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32),
                                              ctypes.POINTER(_I32)]),
    "akv_set_layer_window": (ctypes.c_int, [_P, _I32, _I32]),
    "akv_restore_attention": (ctypes.c_int, [_P, ctypes.POINTER(AkvOp), _I32, _I32, _P, _P, _P,
                                             _I32, _P]),
    "akv_restore_attention_tokens": (ctypes.c_int, [_P, ctypes.POINTER(AkvOp), _I32, _I32, _P, _P,
                                                    _P, _I32, _PI32, _I32, _P]),
    "akv_restore_plan_recovery": (ctypes.c_int, [ctypes.POINTER(AkvOp), _I32, _I32,
                                                 ctypes.POINTER(ctypes.c_uint8),
                                                 ctypes.POINTER(ctypes.c_uint8), _PI32, _PI32]),
    "akv_decode_attention_noalloc": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                                                    ctypes.c_double, _P, _P, _P, _I32, _I32,
                                                    _PI32, _PI32, _P, _P, _I32, _P]),
    "akv_set_wait_limit": (ctypes.c_int, [_P, ctypes.c_uint32]),
    "akv_prefix_index_create": (ctypes.c_int, [_I32, ctypes.POINTER(_P)]),
    "akv_prefix_index_destroy": (ctypes.c_int, [_P]),
    "akv_prefix_last_error": (ctypes.c_char_p, [_P]),
    "akv_prefix_insert": (ctypes.c_int, [_P, _I64, ctypes.POINTER(AkvOp), _I32, _PI32, _I32,
                                         _I64]),
    "akv_prefix_remove": (ctypes.c_int, [_P, _I64]),
    "akv_prefix_touch": (ctypes.c_int, [_P, _I64, _I64]),
    "akv_prefix_match": (ctypes.c_int, [_P, ctypes.POINTER(AkvOp), _I32, _PI32, _I32,
                                        ctypes.POINTER(AkvPrefixMatch)]),
    "akv_prefix_evict_order": (ctypes.c_int, [_P, _PI64, _I32, _PI32]),
    "akv_prefix_publish": (ctypes.c_int, [_P, _P, _I64, ctypes.POINTER(AkvOp), _I32, _PI32, _I32,
                                          _PI64]),
    "akv_prefix_fork": (ctypes.c_int, [_P, _P, ctypes.POINTER(AkvOp), _I32, _PI32, _I32,
                                       ctypes.POINTER(AkvPrefixMatch), _PI64]),
    "akv_prefix_evict": (ctypes.c_int, [_P, _P, _I32, _PI32, _PI32]),
}

_lib = None


def lib_path():
    return _build.LIB


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with agent_kv_cache_gb300.build()")
        l = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(rc, cache=None):
    if rc != AKV_OK:
        msg = lib().akv_last_error(cache).decode() if cache else ""
        raise AkvError(rc, msg)


def _arr(a, dtype, ctype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.POINTER(ctype))


def make_config(layers, hq, hkv, head_dim, page_size, dtype, max_pages, max_seqs, max_slots,
                rope_theta, phys_layers=0, rope_dim=0):
    return AkvConfig(layers, phys_layers, hq, hkv, head_dim, page_size,
                     AKV_DTYPE_BF16 if dtype in ("bf16", AKV_DTYPE_BF16) else AKV_DTYPE_FP32,
                     max_pages, max_seqs, max_slots, float(rope_theta), rope_dim)


def akv_pool_bytes(cfg):
    return lib().akv_pool_bytes(ctypes.byref(cfg))


def akv_cache_create(cfg, k_pool, v_pool, pool_bytes, stream=0):
    out = _P()
    _check(lib().akv_cache_create(ctypes.byref(cfg), k_pool, v_pool, pool_bytes, stream or None,
                                  ctypes.byref(out)))
    return out.value


def akv_cache_destroy(cache):
    _check(lib().akv_cache_destroy(cache))


def akv_set_stream(cache, stream):
    _check(lib().akv_set_stream(cache, stream or None), cache)


def akv_seq_create(cache):
    s = ctypes.c_int64()
    _check(lib().akv_seq_create(cache, ctypes.byref(s)), cache)
    return s.value


def akv_seq_fork(cache, parent):
    s = ctypes.c_int64()
    _check(lib().akv_seq_fork(cache, parent, ctypes.byref(s)), cache)
    return s.value


def akv_seq_free(cache, seq):
    _check(lib().akv_seq_free(cache, seq), cache)


def akv_append(cache, seqs, n_tokens, k_raw, v, token_ids=None):
    s, ps = _arr(seqs, np.int64, ctypes.c_int64)
    n, pn = _arr(n_tokens, np.int32, ctypes.c_int32)
    pt = None
    if token_ids is not None:
        t, pt = _arr(token_ids, np.int32, ctypes.c_int32)
    _check(lib().akv_append(cache, ps, pn, len(s), k_raw, v, pt), cache)


def akv_drop(cache, seq, ranges):
    r, pr = _arr(np.asarray(ranges, dtype=np.int64).reshape(-1, 2), np.int64, ctypes.c_int64)
    _check(lib().akv_drop(cache, seq, pr, r.shape[0]), cache)


def akv_reposition(cache, seqs):
    s, ps = _arr(seqs, np.int64, ctypes.c_int64)
    _check(lib().akv_reposition(cache, ps, len(s)), cache)


def akv_decode_attention(cache, layer, q, seqs, out):
    s, ps = _arr(seqs, np.int64, ctypes.c_int64)
    _check(lib().akv_decode_attention(cache, layer, q, ps, len(s), out), cache)


def akv_seq_info(cache, seq):
    info = AkvSeqInfo()
    _check(lib().akv_seq_info(cache, seq, ctypes.byref(info)), cache)
    return info.as_dict()


def akv_seq_positions(cache, seq, n_held):
    out = np.zeros(n_held, dtype=np.int32)
    _check(lib().akv_seq_positions(cache, seq, out.ctypes.data_as(_PI32)), cache)
    return out


def akv_seq_keep_mask(cache, seq, n_held):
    out = np.zeros(n_held, dtype=np.uint8)
    _check(lib().akv_seq_keep_mask(cache, seq, out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))),
           cache)
    return out


def akv_seq_logical(cache, seq, n_held):
    out = np.zeros(n_held, dtype=np.int64)
    _check(lib().akv_seq_logical(cache, seq, out.ctypes.data_as(_PI64)), cache)
    return out


def akv_seq_gather_map(cache, seq):
    n = ctypes.c_int64()
    _check(lib().akv_seq_gather_map(cache, seq, None, ctypes.byref(n)), cache)
    out = np.zeros(n.value, dtype=np.int32)
    _check(lib().akv_seq_gather_map(cache, seq, out.ctypes.data_as(_PI32), ctypes.byref(n)), cache)
    return out


def akv_seq_page_table(cache, seq):
    npg, nact = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().akv_seq_page_table(cache, seq, None, ctypes.byref(npg), None, ctypes.byref(nact)),
           cache)
    pages = np.zeros(npg.value, dtype=np.int32)
    act = np.zeros(nact.value, dtype=np.int32)
    _check(lib().akv_seq_page_table(cache, seq, pages.ctypes.data_as(_PI32), ctypes.byref(npg),
                                    act.ctypes.data_as(_PI32), ctypes.byref(nact)), cache)
    return pages, act


def akv_seq_host_pages(cache, seq):
    """The planner's page table (host state; no wait)."""
    n = ctypes.c_int32()
    _check(lib().akv_seq_host_pages(cache, seq, None, ctypes.byref(n)), cache)
    out = np.zeros(n.value, np.int32)
    _check(lib().akv_seq_host_pages(cache, seq, out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                                    ctypes.byref(n)), cache)
    return out


def akv_history_key(cache, seq):
    k = (ctypes.c_uint64 * 2)()
    _check(lib().akv_history_key(cache, seq, k), cache)
    return (k[0], k[1])


def akv_page_refcount(cache, page):
    r = ctypes.c_int32()
    _check(lib().akv_page_refcount(cache, page, ctypes.byref(r)), cache)
    return r.value


def akv_pool_stats(cache):
    f, u = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().akv_pool_stats(cache, ctypes.byref(f), ctypes.byref(u)), cache)
    return f.value, u.value


def akv_last_error(cache):
    return lib().akv_last_error(cache).decode()


def akv_sync_errors(cache):
    """Returns the device error word (0 = none) and clears it."""
    w = ctypes.c_uint32()
    rc = lib().akv_sync_errors(cache, ctypes.byref(w))
    if rc not in (AKV_OK, AKV_EDEVICE):
        _check(rc, cache)
    return w.value


def make_program(program):
    """Python program [("append", n) | ("drop", ranges) | ("repos",)] -> akv_op array.

    Returns (array, keep-alive list)."""
    keep = []
    arr = (AkvOp * max(1, len(program)))()
    for i, op in enumerate(program):
        if op[0] == "append":
            arr[i] = AkvOp(AKV_OP_APPEND, int(op[1]), None)
        elif op[0] == "drop":
            r = np.ascontiguousarray(np.asarray(op[1], dtype=np.int64).reshape(-1, 2))
            keep.append(r)
            arr[i] = AkvOp(AKV_OP_DROP, r.shape[0], r.ctypes.data_as(_PI64))
        elif op[0] == "repos":
            arr[i] = AkvOp(AKV_OP_REPOS, 0, None)
        else:
            raise ValueError(op)
    return arr, keep


def akv_restore_attention(cache, program, layer, q, k_raw, v, n_tokens, out):
    arr, keep = make_program(program)
    _check(lib().akv_restore_attention(cache, arr, len(program), layer, q, k_raw, v, n_tokens,
                                       out), cache)
    del keep


def akv_restore_attention_tokens(cache, program, layer, q, k_raw, v, n_tokens, tokens, out):
    arr, keep = make_program(program)
    tk, ptk = _arr(tokens, np.int32, ctypes.c_int32)
    _check(lib().akv_restore_attention_tokens(cache, arr, len(program), layer, q, k_raw, v,
                                              n_tokens, ptk, len(tk), out), cache)
    del keep


def akv_restore_plan_recovery(program, n_tokens, missing, need=None):
    """Tokens to recompute (increasing), given per-token missing / need flags
    (need None: the tokens active at the end of the program)."""
    arr, keep = make_program(program)
    u8 = ctypes.POINTER(ctypes.c_uint8)
    m = np.ascontiguousarray(np.asarray(missing, dtype=np.uint8).reshape(-1))
    nd = None if need is None else np.ascontiguousarray(np.asarray(need, dtype=np.uint8).reshape(-1))
    if m.size != n_tokens or (nd is not None and nd.size != n_tokens):
        raise ValueError("missing / need need one flag per token")
    out = np.zeros(max(1, n_tokens), np.int32)
    n = ctypes.c_int32(0)
    _check(lib().akv_restore_plan_recovery(
        arr, len(program), n_tokens, m.ctypes.data_as(u8),
        nd.ctypes.data_as(u8) if nd is not None else None,
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ctypes.byref(n)))
    del keep
    return out[:n.value].tolist()


def akv_set_layer_window(cache, layer, window):
    _check(lib().akv_set_layer_window(cache, layer, window), cache)


def akv_set_decode_waves(cache, waves):
    _check(lib().akv_set_decode_waves(cache, waves), cache)


def akv_set_restore_tensor_cores(cache, enable):
    """0/False: CUDA cores; 1/True: tensor cores, two query tiles per CTA
    (default); 2: tensor cores, one query tile per CTA."""
    _check(lib().akv_set_restore_tensor_cores(cache, int(enable)), cache)


def akv_set_decode_sharing(cache, mode):
    """mode: False/0 off, True/1 automatic, 2..16 the most rows per shared item."""
    _check(lib().akv_set_decode_sharing(cache, int(mode)), cache)


def akv_decode_plan_stats(cache):
    items, shared, members = _I32(), _I32(), _I32()
    _check(lib().akv_decode_plan_stats(cache, ctypes.byref(items), ctypes.byref(shared),
                                       ctypes.byref(members)), cache)
    return {"items": items.value, "shared_items": shared.value, "members": members.value}


def akv_kernel_launches(cache):
    n = ctypes.c_uint64()
    _check(lib().akv_kernel_launches(cache, ctypes.byref(n)), cache)
    return n.value


def akv_decode_attention_noalloc(k_slab, v_slab, max_pages, hq, hkv, head_dim, page_size,
                                 dtype, rope_theta, page_table, active_pages, keep_bits,
                                 row_stride, keep_stride, n_active_pages, n_held, q, out,
                                 stream=0):
    """Decode attention over caller-owned metadata; allocates nothing (see akv.h)."""
    na, pna = _arr(n_active_pages, np.int32, ctypes.c_int32)
    nh, pnh = _arr(n_held, np.int32, ctypes.c_int32)
    dt = {"bf16": AKV_DTYPE_BF16, "fp32": AKV_DTYPE_FP32}.get(dtype, dtype)
    _check(lib().akv_decode_attention_noalloc(
        k_slab, v_slab, max_pages, hq, hkv, head_dim, page_size, dt, float(rope_theta),
        page_table, active_pages, keep_bits, row_stride, keep_stride, pna, pnh, q, out,
        len(na), stream or None))


def akv_set_wait_limit(cache, polls):
    _check(lib().akv_set_wait_limit(cache, polls), cache)


# ---- history-keyed prefix sharing ------------------------------------------

def _icheck(rc, index):
    if rc != AKV_OK:
        raise AkvError(rc, lib().akv_prefix_last_error(index).decode() if index else "")


def _ids(token_ids):
    a = np.ascontiguousarray(np.asarray(token_ids, dtype=np.int32).reshape(-1))
    return a, a.ctypes.data_as(_PI32)


def akv_prefix_index_create(page_size):
    h = _P()
    _check(lib().akv_prefix_index_create(page_size, ctypes.byref(h)))
    return h


def akv_prefix_index_destroy(index):
    _check(lib().akv_prefix_index_destroy(index))


def akv_prefix_insert(index, entry, program, token_ids, use_time=-1):
    arr, keep = make_program(program)
    ids, pid = _ids(token_ids)
    _icheck(lib().akv_prefix_insert(index, entry, arr, len(program), pid, ids.size, use_time), index)
    del keep


def akv_prefix_remove(index, entry):
    _icheck(lib().akv_prefix_remove(index, entry), index)


def akv_prefix_touch(index, entry, use_time=-1):
    _icheck(lib().akv_prefix_touch(index, entry, use_time), index)


def akv_prefix_match(index, program, token_ids):
    arr, keep = make_program(program)
    ids, pid = _ids(token_ids)
    m = AkvPrefixMatch()
    _icheck(lib().akv_prefix_match(index, arr, len(program), pid, ids.size, ctypes.byref(m)), index)
    del keep
    return m.as_dict()


def akv_prefix_evict_order(index, capacity=4096):
    out = (ctypes.c_int64 * max(1, capacity))()
    n = ctypes.c_int32()
    _icheck(lib().akv_prefix_evict_order(index, out, capacity, ctypes.byref(n)), index)
    return [int(out[i]) for i in range(n.value)]


def akv_prefix_publish(cache, index, seq, program, token_ids):
    arr, keep = make_program(program)
    ids, pid = _ids(token_ids)
    e = ctypes.c_int64()
    _check(lib().akv_prefix_publish(cache, index, seq, arr, len(program), pid, ids.size,
                                    ctypes.byref(e)), cache)
    del keep
    return e.value


def akv_prefix_fork(cache, index, program, token_ids):
    arr, keep = make_program(program)
    ids, pid = _ids(token_ids)
    m = AkvPrefixMatch()
    child = ctypes.c_int64()
    _check(lib().akv_prefix_fork(cache, index, arr, len(program), pid, ids.size, ctypes.byref(m),
                                 ctypes.byref(child)), cache)
    del keep
    return child.value, m.as_dict()


def akv_prefix_evict(cache, index, want_pages):
    f, n = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().akv_prefix_evict(cache, index, want_pages, ctypes.byref(f), ctypes.byref(n)), cache)
    return f.value, n.value
