"""Owner of the two device pools plus the cache handle (PyTorch = memory + streams)."""
import numpy as np

from . import abi


class Cache:
    """A cache over K/V pools allocated with torch on the current CUDA device.

    Methods forward to the C ABI with the same names (without the ``akv_``
    prefix); tensors are passed by device pointer.  The pools are exposed as
    ``k_pool`` / ``v_pool`` shaped [phys_layers, max_pages, hkv, page, D].
    """

    def __init__(self, layers, hq, hkv, head_dim, page_size, dtype, max_pages, max_seqs,
                 max_slots, rope_theta, phys_layers=0, stream=None, rope_dim=0):
        import torch
        self.torch = torch
        self.cfg = abi.make_config(layers, hq, hkv, head_dim, page_size, dtype, max_pages,
                                   max_seqs, max_slots, rope_theta, phys_layers, rope_dim)
        self.layers, self.hq, self.hkv, self.d, self.page = layers, hq, hkv, head_dim, page_size
        self.phys = phys_layers or layers
        self.dtype = dtype
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.pool_bytes = abi.akv_pool_bytes(self.cfg)
        if self.pool_bytes == 0:
            raise abi.AkvError(abi.AKV_EINVAL, "invalid configuration")
        shape = (self.phys, max_pages, hkv, page_size, head_dim)
        self.k_pool = torch.empty(shape, dtype=self.tdtype, device="cuda")
        self.v_pool = torch.empty(shape, dtype=self.tdtype, device="cuda")
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.handle = abi.akv_cache_create(self.cfg, self.k_pool.data_ptr(),
                                           self.v_pool.data_ptr(), self.pool_bytes,
                                           self.stream.cuda_stream)

    def close(self):
        if self.handle:
            abi.akv_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- operations ---------------------------------------------------------
    def seq_create(self):
        return abi.akv_seq_create(self.handle)

    def seq_fork(self, parent):
        return abi.akv_seq_fork(self.handle, parent)

    def seq_free(self, seq):
        abi.akv_seq_free(self.handle, seq)

    def append(self, seqs, n_tokens, k_raw, v, token_ids=None):
        """k_raw, v: device tensors [layers, T, hkv, D] in the pool dtype."""
        assert k_raw.is_contiguous() and v.is_contiguous()
        abi.akv_append(self.handle, seqs, n_tokens, k_raw.data_ptr(), v.data_ptr(), token_ids)

    def drop(self, seq, ranges):
        abi.akv_drop(self.handle, seq, ranges)

    def reposition(self, seqs):
        abi.akv_reposition(self.handle, seqs)

    def restore_attention(self, program, layer, q, k_raw, v, out=None):
        """Segment-batch restore attention of one layer: q [T, hq, D],
        k_raw/v [T, hkv, D] device tensors; returns out [T, hq, D] fp32."""
        torch = self.torch
        n = q.shape[0]
        if out is None:
            out = torch.empty((n, self.hq, self.d), dtype=torch.float32, device="cuda")
        assert q.is_contiguous() and k_raw.is_contiguous() and v.is_contiguous()
        abi.akv_restore_attention(self.handle, program, layer, q.data_ptr(), k_raw.data_ptr(),
                                  v.data_ptr(), n, out.data_ptr())
        return out

    def restore_attention_tokens(self, program, layer, q, k_raw, v, tokens, out=None):
        """Restore attention of the tokens `tokens` (increasing) only: rows of
        `out` [T, hq, D] fp32 for those tokens are written, the rest kept;
        q, k_raw, v cover all T tokens of the program."""
        torch = self.torch
        n = q.shape[0]
        if out is None:
            out = torch.zeros((n, self.hq, self.d), dtype=torch.float32, device="cuda")
        assert q.is_contiguous() and k_raw.is_contiguous() and v.is_contiguous()
        abi.akv_restore_attention_tokens(self.handle, program, layer, q.data_ptr(),
                                         k_raw.data_ptr(), v.data_ptr(), n, tokens,
                                         out.data_ptr())
        return out

    @staticmethod
    def plan_recovery(program, n_tokens, missing, need=None):
        """Tokens of `program` to recompute when the tokens flagged in
        `missing` lost their KV (host only; see akv_restore_plan_recovery)."""
        return abi.akv_restore_plan_recovery(program, n_tokens, missing, need)

    # -- history-keyed prefix sharing ----------------------------------------
    def prefix_publish(self, index, seq, program, token_ids):
        """Publish `seq` (whose history is `program` with `token_ids`) into a
        PrefixIndex; returns the entry id (a frozen snapshot sequence)."""
        return abi.akv_prefix_publish(self.handle, index.handle, seq, program, token_ids)

    def prefix_fork(self, index, program, token_ids):
        """Match a request program and materialise the matched prefix as a new
        sequence; returns (child or -1, match dict)."""
        return abi.akv_prefix_fork(self.handle, index.handle, program, token_ids)

    def prefix_evict(self, index, want_pages):
        """Drop-aware eviction; returns (pages freed, entries evicted)."""
        return abi.akv_prefix_evict(self.handle, index.handle, want_pages)

    def set_restore_tensor_cores(self, enable):
        abi.akv_set_restore_tensor_cores(self.handle, enable)

    def set_decode_sharing(self, mode):
        """Rows holding the same pages read them once per decode call: False /
        0 off, True / 1 automatic (default), 2..16 the most rows per item."""
        abi.akv_set_decode_sharing(self.handle, mode)

    def decode_plan_stats(self):
        """Work items of the last decode call: {"items", "shared_items", "members"}."""
        return abi.akv_decode_plan_stats(self.handle)

    def set_layer_window(self, layer, window):
        abi.akv_set_layer_window(self.handle, layer, window)

    def decode_attention(self, layer, q, seqs, out=None):
        """q: device [n, hq, D] pool dtype; returns out [n, hq, D] fp32."""
        torch = self.torch
        if out is None:
            out = torch.empty((len(seqs), self.hq, self.d), dtype=torch.float32, device="cuda")
        assert q.is_contiguous() and out.is_contiguous()
        abi.akv_decode_attention(self.handle, layer, q.data_ptr(), seqs, out.data_ptr())
        return out

    # -- introspection ------------------------------------------------------
    def info(self, seq):
        return abi.akv_seq_info(self.handle, seq)

    def positions(self, seq):
        return abi.akv_seq_positions(self.handle, seq, self.info(seq)["n_held"])

    def keep_mask(self, seq):
        return abi.akv_seq_keep_mask(self.handle, seq, self.info(seq)["n_held"]).astype(bool)

    def logical(self, seq):
        return abi.akv_seq_logical(self.handle, seq, self.info(seq)["n_held"])

    def gather_map(self, seq):
        return abi.akv_seq_gather_map(self.handle, seq)

    def page_table(self, seq):
        return abi.akv_seq_page_table(self.handle, seq)

    def history_key(self, seq):
        return abi.akv_history_key(self.handle, seq)

    def refcount(self, page):
        return abi.akv_page_refcount(self.handle, page)

    def pool_stats(self):
        return abi.akv_pool_stats(self.handle)

    def kernel_launches(self):
        return abi.akv_kernel_launches(self.handle)

    def sync_errors(self):
        return abi.akv_sync_errors(self.handle)

    def read_kv(self, seq, layer, lo=0, hi=None):
        """Held tokens' stored K and V of one layer, [n_held, hkv, D] (host fp64);
        with ``lo`` / ``hi``, only slots [lo, hi).

        Reads the pool through the device page table (test introspection).
        """
        torch = self.torch
        n = self.info(seq)["n_held"]
        pages, _ = self.page_table(seq)
        slots = np.arange(lo, n if hi is None else min(hi, n))
        pid = torch.from_numpy(pages[slots // self.page].astype(np.int64)).cuda()
        off = torch.from_numpy((slots % self.page).astype(np.int64)).cuda()
        slab = layer % self.phys
        k = self.k_pool[slab][pid, :, off]          # [n, hkv, D]
        v = self.v_pool[slab][pid, :, off]
        return (k.double().cpu().numpy(), v.double().cpu().numpy())


class PrefixIndex:
    """Host-only history-keyed prefix index (no GPU needed)."""

    def __init__(self, page_size):
        self.handle = abi.akv_prefix_index_create(page_size)

    def insert(self, entry, program, token_ids, use_time=-1):
        abi.akv_prefix_insert(self.handle, entry, program, token_ids, use_time)

    def remove(self, entry):
        abi.akv_prefix_remove(self.handle, entry)

    def touch(self, entry, use_time=-1):
        abi.akv_prefix_touch(self.handle, entry, use_time)

    def match(self, program, token_ids):
        return abi.akv_prefix_match(self.handle, program, token_ids)

    def evict_order(self):
        return abi.akv_prefix_evict_order(self.handle)

    def close(self):
        if self.handle:
            abi.akv_prefix_index_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
