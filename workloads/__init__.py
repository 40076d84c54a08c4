"""Seeded synthetic inputs for the active-KV cache operations.

This package holds only input generation: counter-based random values and the
shapes of synthetic agent trajectories (which token spans are tool responses,
which of them a rolling-drop policy removes, where reposition happens).  It
contains none of the arithmetic of the method itself; both the CUDA library's
tests/benchmark and the CPU oracle take their inputs from here.
"""
from .synth import (GAMMA, KIND_K, KIND_V, KIND_Q, WIDTH_BF16, WIDTH_FP32,
                    mix64, stream_key, block, width_for)
from . import traces

__all__ = ["GAMMA", "KIND_K", "KIND_V", "KIND_Q", "WIDTH_BF16", "WIDTH_FP32",
           "mix64", "stream_key", "block", "width_for", "traces"]
