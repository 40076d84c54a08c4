"""The C-ABI library builds, loads without a GPU and exports every declared symbol."""
import ctypes
import os
import re

import pytest

from agent_kv_cache_gb300 import _build, abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "akv.h")


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:int|size_t|const char\s*\*)\s*(akv_\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return abi.lib()


def test_header_parses():
    names = declared()
    assert len(names) == len(set(names)) >= 20
    assert set(names) == set(abi.SIGNATURES), set(names) ^ set(abi.SIGNATURES)


def test_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_pool_bytes_and_config_validation(lib):
    cfg = abi.make_config(32, 32, 8, 128, 16, "bf16", 1000, 16, 40000, 5e5)
    assert abi.akv_pool_bytes(cfg) == 32 * 1000 * 8 * 16 * 128 * 2
    cfg = abi.make_config(80, 64, 8, 128, 16, "bf16", 10, 4, 1000, 5e5, phys_layers=16)
    assert abi.akv_pool_bytes(cfg) == 16 * 10 * 8 * 16 * 128 * 2
    cfg = abi.make_config(1, 8, 2, 64, 16, "fp32", 40, 1, 600, 1e4)
    assert abi.akv_pool_bytes(cfg) == 40 * 2 * 16 * 64 * 4
    bad = [
        dict(hq=30),            # not a multiple of hkv
        dict(hq=8 * 32),        # group of 32
        dict(head_dim=96),
        dict(page_size=12),
        dict(max_slots=0),
        dict(phys_layers=40),   # more slabs than layers
        dict(rope_theta=0.5),
    ]
    base = dict(layers=32, hq=32, hkv=8, head_dim=128, page_size=16, dtype="bf16",
                max_pages=100, max_seqs=4, max_slots=1000, rope_theta=5e5)
    for b in bad:
        kw = dict(base)
        kw.update(b)
        assert abi.akv_pool_bytes(abi.make_config(**kw)) == 0, b


def test_null_handles_are_rejected(lib):
    assert lib.akv_cache_destroy(None) == abi.AKV_EINVAL
    assert lib.akv_seq_free(None, 1) == abi.AKV_EINVAL
    out = ctypes.c_void_p()
    cfg = abi.make_config(1, 8, 2, 64, 16, "fp32", 40, 1, 600, 1e4)
    # null pools are rejected before any CUDA call
    assert lib.akv_cache_create(ctypes.byref(cfg), None, None, 0, None, ctypes.byref(out)) == abi.AKV_EINVAL


def test_binding_constants_match_the_header():
    text = open(HEADER).read()
    for name in ("AKV_NOALLOC_SCRATCH_BYTES", "AKV_NOALLOC_MAX_SEQS", "AKV_OK", "AKV_EINVAL",
                 "AKV_ECAPACITY"):
        m = re.search(r"#define\s+%s\s+(.+)" % name, text)
        if m is None:
            m = re.search(r"\b%s\s*=\s*([^,\n]+)" % name, text)
        assert m is not None, name
        value = re.sub(r"/\*.*", "", m.group(1)).strip().rstrip(",")
        assert eval(value) == getattr(abi, name), name
