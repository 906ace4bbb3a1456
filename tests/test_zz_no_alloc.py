"""moe_permute_noalloc: the grouping stage for callers that cannot allocate device memory.

Such callers (code enqueued during CUDA-graph stream capture, plug-ins whose host
framework owns all device memory, allocation-free real-time loops) get the same
grouping as moe_permute while the library keeps the scratch histogram in its own
fixed device array. This file is collected last on purpose: it checks, through the
C ABI, that consecutive calls sharing that array agree exactly with the
workspace-based entry point, whether run alone in a fresh process or after every
other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, cfg_of


def _routing(w, dev, cfg):
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device="cuda")
    gate = torch.empty(w.T, w.top_k, dtype=torch.float32, device="cuda")
    moe.moe_router_topk(cfg, dev["x"], dev["w_router"], dev["bias"], idx, gate)
    return idx


def _outputs(w, cfg, dt):
    R = moe.moe_rows_capacity(cfg)
    return dict(counts=torch.full((w.n_experts,), -1, dtype=torch.int32, device="cuda"),
                offsets=torch.full((w.n_experts + 1,), -1, dtype=torch.int32, device="cuda"),
                dest=torch.full((w.T, w.top_k), -2, dtype=torch.int32, device="cuda"),
                src=torch.full((R,), -3, dtype=torch.int32, device="cuda"),
                xp=torch.zeros(R, w.d_model, dtype=dt, device="cuda"))


def _same(a, b, P):
    assert torch.equal(a["counts"], b["counts"])
    assert torch.equal(a["offsets"], b["offsets"])
    assert torch.equal(a["dest"], b["dest"])
    assert torch.equal(a["src"][:P], b["src"][:P])
    assert torch.equal(a["xp"][:P].view(torch.int16), b["xp"][:P].view(torch.int16))


@pytest.mark.gpu
def test_noalloc_permute_matches_workspace_permute_on_consecutive_calls():
    cases = []
    for name in ("mini_deepseek", "qwen3_30b_a3b"):       # drops + shared expert, then 64 chunks x 128 experts
        w = synth.WORKLOADS[name]
        dev = Inputs(w).device() if name.startswith("mini") else synth.device_inputs(w)
        cases.append((w, cfg_of(w), dev))
    for w, cfg, dev in cases:                              # two calls in a row, different sizes and contents
        idx = _routing(w, dev, cfg)
        ref = _outputs(w, cfg, dev["x"].dtype)
        ws = moe.alloc_workspace(cfg)
        moe.moe_permute(cfg, idx, dev["x"], ref["counts"], ref["offsets"], ref["dest"], ref["src"], ref["xp"], ws)
        got = _outputs(w, cfg, dev["x"].dtype)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = moe.lib().moe_permute_noalloc(ctypes.byref(cfg), idx.data_ptr(), dev["x"].data_ptr(),
                                           got["counts"].data_ptr(), got["offsets"].data_ptr(),
                                           got["dest"].data_ptr(), got["src"].data_ptr(), got["xp"].data_ptr(),
                                           status.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == moe.MOE_OK
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == moe.MOE_OK
        assert status.item() == moe.MOE_OK
        P = int(ref["offsets"][-1].item())
        assert P > 0
        _same(ref, got, P)
    # and once more on the first case: the array still holds the larger call's contents
    w, cfg, dev = cases[0]
    idx = _routing(w, dev, cfg)
    ref = _outputs(w, cfg, dev["x"].dtype)
    moe.moe_permute(cfg, idx, dev["x"], ref["counts"], ref["offsets"], ref["dest"], ref["src"], ref["xp"],
                    moe.alloc_workspace(cfg))
    got = _outputs(w, cfg, dev["x"].dtype)
    moe.moe_permute_noalloc(cfg, idx, dev["x"], got["counts"], got["offsets"], got["dest"], got["src"], got["xp"])
    torch.cuda.synchronize()
    _same(ref, got, int(ref["offsets"][-1].item()))


def test_noalloc_refuses_configurations_beyond_its_array():
    # ceil(65536 / 128) * 256 = 131072 histogram entries > 65536: refused before any launch
    cfg = moe.make_config(T=65536, d_model=128, n_experts=256, top_k=8, d_ff=128)
    p = 0x10000
    rc = moe.lib().moe_permute_noalloc(ctypes.byref(cfg), p, p, p, p, p, p, p, None, None)
    assert rc == moe.MOE_ERR_WORKSPACE
    ok = moe.make_config(T=32768, d_model=128, n_experts=256, top_k=8, d_ff=128)
    assert moe.lib().moe_permute_noalloc(ctypes.byref(ok), None, p, p, p, p, p, p, None, None) == \
        moe.MOE_ERR_INVALID_ARG
