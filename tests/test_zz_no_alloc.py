"""moe_permute_noalloc: the grouping stage for callers that cannot allocate device memory.

Such callers (code enqueued during CUDA-graph stream capture, plug-ins whose host
framework owns all device memory, allocation-free real-time loops) get the same
grouping as moe_permute; batches of more than one 128-token chunk keep their scratch
histogram in a fixed device array of the library. This file is collected last on
purpose: it checks, through the C ABI, that consecutive calls agree exactly with the
workspace-based entry point and with the oracle's grouping, whether run alone in a
fresh process or after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
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


def _noalloc(cfg, idx, x, got, status):
    rc = moe.lib().moe_permute_noalloc(ctypes.byref(cfg), idx.data_ptr(), x.data_ptr(), got["counts"].data_ptr(),
                                       got["offsets"].data_ptr(), got["dest"].data_ptr(), got["src"].data_ptr(),
                                       got["xp"].data_ptr(), None if status is None else status.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == moe.MOE_OK, moe.status_string(rc)
    torch.cuda.synchronize()


def _same(a, b, P):
    assert torch.equal(a["counts"], b["counts"])
    assert torch.equal(a["offsets"], b["offsets"])
    assert torch.equal(a["dest"], b["dest"])
    assert torch.equal(a["src"][:P], b["src"][:P])
    assert torch.equal(a["xp"][:P].view(torch.int16), b["xp"][:P].view(torch.int16))


def _matches_oracle(w, idx, x, got):
    """counts, offsets, dest_row, src_token and x_perm bit-exact against the oracle's grouping."""
    cap = O.capacity(w.T, w.top_k, w.n_experts, w.capacity_factor)
    disp = O.dispatch(idx.cpu().numpy(), w.n_experts, cap)
    P = int(disp.offsets[-1])
    assert (got["counts"].cpu().numpy() == disp.counts).all()
    assert (got["offsets"].cpu().numpy() == disp.offsets).all()
    assert (got["dest"].cpu().numpy() == disp.dest_row).all()
    assert (got["src"][:P].cpu().numpy() == disp.src_token).all()
    rows = torch.from_numpy(disp.src_token.astype(np.int64)).cuda()
    assert torch.equal(got["xp"][:P].view(torch.int16), x[rows].view(torch.int16))
    return P


def _limit_case():
    """A batch whose histogram fills the array exactly: ceil(32768/128) * 256 = 65536 entries.
    Expert ids are drawn directly (8 distinct of 256 per token, seeded), x is generated."""
    w = synth.Workload("noalloc_limit", T=32768, d_model=128, n_experts=256, top_k=8, d_ff=128)
    rng = np.random.default_rng(7)
    idx = np.argsort(rng.random((w.T, w.n_experts)), axis=1)[:, :w.top_k].astype(np.int32)
    x = synth.host_to_torch(synth.host_tensor(w, "x"), w.dtype).cuda()
    return w, idx, x


@pytest.mark.gpu
def test_noalloc_permute_matches_workspace_permute_on_consecutive_calls():
    cases = []
    for name in ("mini_deepseek", "mini_decode", "qwen3_30b_a3b"):   # drops + shared expert; one chunk; 64 chunks
        w = synth.WORKLOADS[name]
        dev = Inputs(w).device() if name.startswith("mini") else synth.device_inputs(w)
        cases.append((w, cfg_of(w), dev))
    for w, cfg, dev in cases:                              # calls in a row, different sizes and contents
        idx = _routing(w, dev, cfg)
        ref = _outputs(w, cfg, dev["x"].dtype)
        ws = moe.alloc_workspace(cfg)
        moe.moe_permute(cfg, idx, dev["x"], ref["counts"], ref["offsets"], ref["dest"], ref["src"], ref["xp"], ws)
        got = _outputs(w, cfg, dev["x"].dtype)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        _noalloc(cfg, idx, dev["x"], got, status)
        assert moe.moe_get_device_error(ws) == moe.MOE_OK
        assert status.item() == moe.MOE_OK
        P = int(ref["offsets"][-1].item())
        assert P > 0
        _same(ref, got, P)
        assert _matches_oracle(w, idx, dev["x"], got) == P
    # and once more on the first case: the array still holds the larger call's contents
    w, cfg, dev = cases[0]
    idx = _routing(w, dev, cfg)
    got = _outputs(w, cfg, dev["x"].dtype)
    moe.moe_permute_noalloc(cfg, idx, dev["x"], got["counts"], got["offsets"], got["dest"], got["src"], got["xp"])
    torch.cuda.synchronize()
    _matches_oracle(w, idx, dev["x"], got)


@pytest.mark.gpu
def test_noalloc_permute_at_the_array_limit_twice():
    w, idx_np, x = _limit_case()
    cfg = cfg_of(w)
    idx = torch.from_numpy(idx_np).cuda()
    for _ in range(2):                                     # the second call runs over the first one's contents
        got = _outputs(w, cfg, x.dtype)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        _noalloc(cfg, idx, x, got, status)
        assert status.item() == moe.MOE_OK
        assert _matches_oracle(w, idx, x, got) == w.T * w.top_k


@pytest.mark.gpu
@pytest.mark.parametrize("T", [5, 300])                    # single-chunk and multi-chunk grouping
def test_noalloc_flags_an_out_of_range_id(T):
    w = synth.WORKLOADS["mini_qwen3"].with_(T=T)
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    idx = _routing(w, dev, cfg)
    bad = idx.clone()
    bad[T // 2, 1] = w.n_experts                           # one id past the last expert
    got = _outputs(w, cfg, dev["x"].dtype)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _noalloc(cfg, bad, dev["x"], got, status)
    assert status.item() == moe.MOE_ERR_DEVICE_INDEX
    dest = got["dest"].cpu().numpy()
    assert dest[T // 2, 1] == -1                           # the bad pair is skipped ...
    keep = np.ones_like(dest, dtype=bool)
    keep[T // 2, 1] = False
    assert (dest[keep] >= 0).all()                         # ... and every other pair is grouped
    assert int(got["offsets"][-1].item()) == T * w.top_k - 1


def test_noalloc_refuses_configurations_beyond_its_array():
    # ceil(65536 / 128) * 256 = 131072 histogram entries > 65536: refused before any launch
    cfg = moe.make_config(T=65536, d_model=128, n_experts=256, top_k=8, d_ff=128)
    p = 0x10000
    rc = moe.lib().moe_permute_noalloc(ctypes.byref(cfg), p, p, p, p, p, p, p, None, None)
    assert rc == moe.MOE_ERR_WORKSPACE
    ok = moe.make_config(T=32768, d_model=128, n_experts=256, top_k=8, d_ff=128)
    assert moe.lib().moe_permute_noalloc(ctypes.byref(ok), None, p, p, p, p, p, p, None, None) == \
        moe.MOE_ERR_INVALID_ARG
