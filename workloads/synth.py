"""Counter-based synthetic values, identical on the host and on the GPU.

Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the 64-bit finaliser published
with Java's SplittableRandom).  The i-th output of a SplitMix64 stream whose
state starts at ``key`` is ``mix64(key + (i + 1) * GAMMA)`` (mod 2**64), so any
element can be produced independently of the others: that is what makes the
same values cheap to produce on the GPU (``workloads/csrc/synth.cu``) and in
numpy (here) for the oracle.

Values.  A 64-bit output h is cut into three w-bit fields f0, f1, f2 and mapped
to ``(2*(f0+f1+f2) - 3*(2**w - 1)) / 2**w``: a three-term Irwin-Hall sum,
centred, with mean 0 and variance 1 - 4**-w (about N(0,1), bounded by +-3).
Every value is an odd integer over 2**w, so it is exact in the pool dtype:

* w = 6  -> |numerator| <= 189 < 2**8: exact in bfloat16 (8 significant bits);
* w = 21 -> |numerator| <  2**23:      exact in float32.

No rounding happens anywhere in input generation, so host and device agree
bit for bit without sharing any floating-point code.

Streams.  ``stream_key(seed, tag, kind, layer)`` folds the parts into one
64-bit key with the same SplitMix64 step.  ``tag`` names a sequence (or a
branch), ``kind`` one of K, V, Q, and ``layer`` the transformer layer.  For K
and V the element index is ``(logical_token * Hkv + head) * D + d``; for Q it
is ``(decode_step * Hq + head) * D + d``.
"""
import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB

KIND_K = 1
KIND_V = 2
KIND_Q = 3

WIDTH_BF16 = 6
WIDTH_FP32 = 21


def width_for(dtype):
    """Field width that makes every value exact in ``dtype`` ('bf16'/'fp32')."""
    if dtype == "bf16":
        return WIDTH_BF16
    if dtype == "fp32":
        return WIDTH_FP32
    raise ValueError(f"unknown pool dtype {dtype!r}")


def mix64(z):
    """SplitMix64 finaliser on a numpy uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
        z = z ^ (z >> np.uint64(31))
    return z


def _mix64_int(z):
    z &= MASK64
    z = ((z ^ (z >> 30)) * _M1) & MASK64
    z = ((z ^ (z >> 27)) * _M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed, *parts):
    """Fold ``seed`` and integer ``parts`` into one 64-bit stream key."""
    k = int(seed) & MASK64
    for p in parts:
        k = _mix64_int(k + ((int(p) + 1) * GAMMA))
    return k


def block(seed, tag, kind, layer, start, count, width):
    """``count`` consecutive values of stream (seed, tag, kind, layer) from ``start``.

    Returns float32 (every value is exact there, and in bfloat16 when
    ``width == WIDTH_BF16``).
    """
    key = np.uint64(stream_key(seed, tag, kind, layer))
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        h = mix64(key + idx * np.uint64(GAMMA))
    m = np.uint64((1 << width) - 1)
    w = np.uint64(width)
    s = (h & m) + ((h >> w) & m) + ((h >> (w + w)) & m)
    num = 2 * s.astype(np.int64) - 3 * int((1 << width) - 1)
    return (num.astype(np.float64) / float(1 << width)).astype(np.float32)


def kv_tokens(seed, tag, kind, layers, t0, n, hkv, d, width):
    """K or V rows for logical tokens [t0, t0+n) of sequence ``tag``.

    Returns float32 ``[len(layers)][n][hkv][d]``.
    """
    per_tok = hkv * d
    out = np.empty((len(layers), n, hkv, d), dtype=np.float32)
    for i, l in enumerate(layers):
        out[i] = block(seed, tag, kind, l, t0 * per_tok, n * per_tok,
                       width).reshape(n, hkv, d)
    return out


def query(seed, tag, layer, step, hq, d, width):
    """Decode query of sequence ``tag`` at decode step ``step``: ``[hq][d]``."""
    per = hq * d
    return block(seed, tag, KIND_Q, layer, step * per, per, width).reshape(hq, d)
