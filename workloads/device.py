"""GPU copy of the seeded generator (workloads/csrc/synth.cu), for full-size inputs.

Produces on the device exactly the values ``workloads.synth`` produces on the
host (the test ``tests/test_gpu_synth.py`` compares them bit for bit).
"""
import ctypes
import os
import subprocess

import numpy as np

from . import synth

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "synth.cu")
LIB = os.path.join(HERE, "_lib", "libakv_synth.so")
_lib = None


def build(force=False):
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    cmd = [nvcc if os.path.exists(nvcc) else "nvcc", "-gencode", "arch=compute_103a,code=sm_103a",
           "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        raise RuntimeError(f"nvcc failed on synth.cu:\n{r.stdout}\n{r.stderr}")
    os.replace(LIB + ".tmp", LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = ctypes.CDLL(LIB)
        _lib.akv_synth_fill.restype = ctypes.c_int
        _lib.akv_synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_void_p]
    return _lib


def fill(out, rows, count, width, stream=None):
    """out: torch tensor (bf16/fp32, cuda); rows: list of (key, start, out_offset)."""
    import torch
    r = torch.tensor(np.array([[np.uint64(k).view(np.int64), s, o] for k, s, o in rows],
                              dtype=np.int64), device=out.device)
    st = (stream or torch.cuda.current_stream()).cuda_stream
    rc = _load().akv_synth_fill(out.data_ptr(), int(out.dtype == torch.bfloat16), r.data_ptr(),
                                len(rows), count, width, st)
    if rc:
        raise RuntimeError(f"akv_synth_fill failed ({rc})")
    return r   # keep alive until the kernel has run


def kv_tokens(out, seed, tag, kind, layers, t0, n, hkv, d, width, stream=None):
    """Fill out [len(layers)][n][hkv][d] with the rows of logical tokens [t0, t0+n)."""
    per = hkv * d
    rows = [(synth.stream_key(seed, tag, kind, l), t0 * per, i * n * per)
            for i, l in enumerate(layers)]
    return fill(out, rows, n * per, width, stream)


def kv_tokens_multi(out, seed, tags, kind, layers, t0s, n, hkv, d, width, stream=None):
    """out [len(layers)][len(tags)*n][hkv][d]: n tokens per tag, tags in order."""
    per = hkv * d
    T = len(tags) * n
    rows = [(synth.stream_key(seed, tag, kind, l), t0 * per, (i * T + j * n) * per)
            for i, l in enumerate(layers) for j, (tag, t0) in enumerate(zip(tags, t0s))]
    return fill(out, rows, n * per, width, stream)


def queries(out, seed, tags, layer, step, hq, d, width, stream=None):
    """out [len(tags)][hq][d]: decode queries of one layer and step."""
    per = hq * d
    rows = [(synth.stream_key(seed, tag, synth.KIND_Q, layer), step * per, j * per)
            for j, tag in enumerate(tags)]
    return fill(out, rows, per, width, stream)
