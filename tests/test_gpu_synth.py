"""The device input generator reproduces the host generator bit for bit."""
import numpy as np
import pytest
import torch

from workloads import device, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,width", [("bf16", synth.WIDTH_BF16), ("fp32", synth.WIDTH_FP32)])
def test_device_generator_matches_host(dtype, width):
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    layers, n, hkv, d = [0, 3, 7], 37, 2, 64
    out = torch.empty((len(layers), n, hkv, d), dtype=td, device="cuda")
    keep = device.kv_tokens(out, 99, 5, synth.KIND_K, layers, 1000, n, hkv, d, width)
    torch.cuda.synchronize()
    want = synth.kv_tokens(99, 5, synth.KIND_K, layers, 1000, n, hkv, d, width)
    np.testing.assert_array_equal(out.float().cpu().numpy(), want)
    q = torch.empty((3, 8, 64), dtype=td, device="cuda")
    keep = device.queries(q, 99, [4, 5, 6], 2, 11, 8, 64, width)
    torch.cuda.synchronize()
    want = np.stack([synth.query(99, t, 2, 11, 8, 64, width) for t in (4, 5, 6)])
    np.testing.assert_array_equal(q.float().cpu().numpy(), want)
    del keep
