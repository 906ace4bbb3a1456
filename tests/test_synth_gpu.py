"""The device generator reproduces the host generator bit for bit."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("start,n", [(0, 4099), (3 * 2048 * 7168 + 5, 10_000), ((1 << 32) + 1, 777)])
def test_device_matches_host(dtype, start, n):
    t = torch.empty(n, dtype=torch.bfloat16 if dtype == "bf16" else torch.float32, device="cuda")
    synth.fill_device(t, 0, 3, 0.02, start=start)
    torch.cuda.synchronize()
    host = synth.normal(0, 3, (n,), 0.02, dtype, start=start)
    if dtype == "bf16":
        got = t.cpu().view(torch.int16).numpy().view(np.uint16)
    else:
        got = t.cpu().numpy()
    assert (got == host).all()


def test_device_inputs_match_host_slices():
    w = synth.WORKLOADS["mini_deepseek"]
    dev = synth.device_inputs(w)
    torch.cuda.synchronize()
    for name in ("x", "w_router", "w_gate", "w_down"):
        got = dev[name].cpu().view(torch.int16).numpy().view(np.uint16)
        assert (got == synth.host_tensor(w, name)).all(), name
