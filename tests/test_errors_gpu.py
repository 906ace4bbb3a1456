"""Failure paths on the GPU, none of which faults or hangs it: out-of-range ids and
corrupt offsets are skipped and recorded, a stalled wait gives up and reports a
status, and the context stays usable afterwards."""
import numpy as np
import pytest
import torch

import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, cfg_of

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    moe.moe_workspace_init(ws)
    moe.moe_selftest_bounded_wait(ws, 20_000_000)        # 20 ms on a barrier nothing completes
    assert moe.moe_get_device_error(ws) == moe.MOE_ERR_TIMEOUT
    moe.moe_clear_device_error(ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    # the context is still healthy: a normal layer runs and reports no error
    w = synth.WORKLOADS["mini_mixtral"]
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    ws2 = moe.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d_model, dtype=torch.bfloat16, device="cuda")
    moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"], dev["w_down"],
                          out, ws2)
    assert moe.moe_get_device_error(ws2) == moe.MOE_OK
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("T", [333, 100])             # multi-chunk kernels; one launch for a single chunk
def test_out_of_range_ids_are_skipped_and_flagged(T):
    w = synth.WORKLOADS["mini_qwen3"].with_(T=T)
    cfg = cfg_of(w)
    dev = Inputs(w).device()
    # distinct experts per token (a random permutation's first k), then the bad entries
    idx = torch.argsort(torch.rand(w.T, w.n_experts, device="cuda"), dim=1)[:, :w.top_k].to(torch.int32)
    idx[5, 3] = w.n_experts + 3
    idx[7, 0] = -1
    idx[9, 2] = idx[9, 1]                                # an expert repeated within a token
    R = moe.moe_rows_capacity(cfg)
    counts = torch.empty(w.n_experts, dtype=torch.int32, device="cuda")
    offsets = torch.empty(w.n_experts + 1, dtype=torch.int32, device="cuda")
    dest = torch.empty(w.T, w.top_k, dtype=torch.int32, device="cuda")
    src = torch.empty(R, dtype=torch.int32, device="cuda")
    xp = torch.empty(R, w.d_model, dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.moe_permute(cfg, idx, dev["x"], counts, offsets, dest, src, xp, ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_ERR_DEVICE_INDEX
    assert dest[5, 3].item() == -1 and dest[7, 0].item() == -1
    d = dest.cpu().numpy()
    assert sorted([d[9, 1], d[9, 2]])[0] == -1 and max(d[9, 1], d[9, 2]) >= 0   # one of the two slots kept
    bad = d < 0
    assert bad.sum() == 3 and bad[5, 3] and bad[7, 0]
    assert (d[~bad] >= 0).all() and int(offsets[-1].item()) == w.T * w.top_k - 3
    rows = torch.from_numpy(d[~bad].astype(np.int64)).cuda()
    toks = torch.from_numpy(np.nonzero(~bad)[0].astype(np.int64)).cuda()
    assert torch.equal(src[rows].long(), toks)                          # each kept row names its token
    assert torch.equal(xp[rows], dev["x"][toks])                        # and holds its x row


def test_corrupt_offsets_are_rejected_on_device():
    w = synth.WORKLOADS["mini_mixtral"]
    cfg = cfg_of(w)
    dev = Inputs(w).device()
    R = moe.moe_rows_capacity(cfg)
    xp = torch.zeros(R, w.d_model, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(moe.moe_grouped_rows(cfg), w.d_model, dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(cfg)
    bad = torch.tensor([0, 50, 40, 600, 600, 600, 600, 600, 10 ** 6], dtype=torch.int32, device="cuda")
    moe.moe_grouped_ffn(cfg, xp, bad, dev["x"], dev["w_gate"], dev["w_up"], dev["w_down"], y, ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_ERR_DEVICE_INDEX
    assert (y == 0).all()        # nothing was written


def test_workspace_too_small_is_refused():
    w = synth.WORKLOADS["mini_mixtral"]
    cfg = cfg_of(w)
    dev = Inputs(w).device()
    ws = torch.empty(moe.moe_workspace_size(cfg) - 256, dtype=torch.uint8, device="cuda")
    out = torch.empty(w.T, w.d_model, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"],
                              dev["w_down"], out, ws)
    assert ei.value.code == moe.MOE_ERR_WORKSPACE
