"""Stage-by-stage parity of the C ABI against the fp64 oracle on the reduced workloads.

Each stage is fed the GPU's own output of the stage before, so a mismatch
points at exactly one kernel. Workloads span several GEMM tiles with ragged
tails (T not a multiple of 128, uneven expert loads, empty experts, capacity
drops, a shared expert, float32 and bf16).
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, assert_close, cfg_of, check_routing, out_tolerance, router_tolerance, to_f64

pytestmark = pytest.mark.gpu

MINI = synth.workloads.MINI


def _router(w, inp, dev, cfg):
    T, k, E = w.T, w.top_k, w.n_experts
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gate = torch.empty(T, k, dtype=torch.float32, device="cuda")
    scores = torch.empty(T, E, dtype=torch.float32, device="cuda")
    moe.moe_router_topk(cfg, dev["x"], dev["w_router"], dev["bias"], idx, gate, scores)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), gate.cpu().numpy().astype(np.float64), scores.cpu().numpy().astype(np.float64), idx, gate


@pytest.mark.parametrize("name", MINI)
def test_router_matches_oracle(name):
    _check_router(synth.WORKLOADS[name])


@pytest.mark.parametrize("edit", [
    dict(T=1, n_experts=1, top_k=1),                        # one token, one expert
    dict(T=130, n_experts=6, top_k=3),                      # E below one 16-column MMA slice
    dict(T=257, n_experts=200, top_k=8, bias_s=1.2),        # E not a multiple of 16 or 32, skewed
    dict(T=64, n_experts=256, top_k=8, score="sigmoid"),    # the widest accumulator
    dict(T=129, n_experts=17, top_k=5, renormalize=False),  # raw softmax gates
    dict(T=40, n_experts=33, top_k=2, score="sigmoid", renormalize=False, bias_s=0.5),
])
def test_router_shapes(edit):
    _check_router(synth.WORKLOADS["mini_qwen3"].with_(**edit))


def _check_router(w, x64=None, wr64=None, bias=None, dev=None):
    if dev is None:
        inp = Inputs(w)
        dev = inp.device()
        x64, wr64, bias = inp.f64["x"], inp.f64["w_router"], inp.bias
    cfg = cfg_of(w)
    idx, gate, scores, _, _ = _router(w, None, dev, cfg)
    ref_scores = O.scores_from_logits(O.router_logits(x64, wr64, bias), w.score)
    tol = router_tolerance(x64, wr64, bias)[:, None]          # [T, 1]: per token
    err = np.abs(scores - ref_scores)
    assert (err <= tol).all(), f"score error {float((err / tol).max()):.2f} x the token's tolerance"
    check_routing(idx, ref_scores, w.top_k)
    ref_gate = O.gates_from_scores(np.take_along_axis(ref_scores, idx.astype(np.int64), axis=1), w.renormalize)
    gerr = np.abs(gate - ref_gate)
    assert (gerr <= tol).all(), f"gate error {float((gerr / tol).max()):.2f} x the token's tolerance"
    if w.renormalize:
        assert np.abs(gate.sum(axis=1) - 1.0).max() <= 1e-5


@pytest.mark.parametrize("name", synth.workloads.FULL + synth.workloads.FULL_EXTRA)
def test_router_full_size(name):
    # the five model-shaped routers on their full batches: scores and gates of every token
    w = synth.WORKLOADS[name]
    raw = {n: synth.host_tensor(w, n) for n in ("x", "w_router")}
    bias = synth.router_bias(w.n_experts, w.bias_s)
    dev = {n: synth.host_to_torch(a, w.dtype).cuda() for n, a in raw.items()}
    dev["bias"] = None if bias is None else torch.from_numpy(bias).cuda()
    _check_router(w, synth.as_f64(raw["x"], w.dtype), synth.as_f64(raw["w_router"], w.dtype), bias, dev)


@pytest.mark.parametrize("name", MINI)
def test_grouping_is_bit_exact(name):
    w = synth.WORKLOADS[name]
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    idx_np, _, _, idx, _ = _router(w, inp, dev, cfg)
    R = moe.moe_rows_capacity(cfg)
    E, T, k = w.n_experts, w.T, w.top_k
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dest = torch.empty(T, k, dtype=torch.int32, device="cuda")
    src = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    xdt = dev["x"].dtype
    x_perm = torch.zeros(R, w.d_model, dtype=xdt, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.moe_permute(cfg, idx, dev["x"], counts, offsets, dest, src, x_perm, ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    ref = O.dispatch(idx_np, E, O.capacity(T, k, E, w.capacity_factor))
    assert (counts.cpu().numpy() == ref.counts).all()
    assert (offsets.cpu().numpy() == ref.offsets).all()
    assert (dest.cpu().numpy() == ref.dest_row).all()
    P = int(ref.offsets[-1])
    assert (src.cpu().numpy()[:P] == ref.src_token).all()
    xp = x_perm[:P].cpu()
    xr = dev["x"].cpu()[torch.from_numpy(ref.src_token.astype(np.int64))]
    assert torch.equal(xp.view(torch.int16) if xdt == torch.bfloat16 else xp.view(torch.int32),
                       xr.view(torch.int16) if xdt == torch.bfloat16 else xr.view(torch.int32))
    if w.capacity_factor > 0:
        assert (dest.cpu().numpy() < 0).sum() == T * k - P


def _grouped(w, inp, dev, cfg):
    idx_np, gate_np, _, idx, gate = _router(w, inp, dev, cfg)
    R = moe.moe_rows_capacity(cfg)
    rows = moe.moe_grouped_rows(cfg)
    E, T, k = w.n_experts, w.T, w.top_k
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dest = torch.empty(T, k, dtype=torch.int32, device="cuda")
    src = torch.empty(R, dtype=torch.int32, device="cuda")
    x_perm = torch.empty(R, w.d_model, dtype=dev["x"].dtype, device="cuda")
    y = torch.full((rows, w.d_model), float("nan"), dtype=dev["x"].dtype, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.moe_permute(cfg, idx, dev["x"], counts, offsets, dest, src, x_perm, ws)
    moe.moe_grouped_ffn(cfg, x_perm, offsets, dev["x"], dev["w_gate"], dev["w_up"], dev["w_down"], y, ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    return dict(idx=idx_np, gate=gate_np, gate_t=gate, offsets=offsets.cpu().numpy(), src=src.cpu().numpy(),
                dest=dest, dest_np=dest.cpu().numpy(), y=y, R=R, ws=ws)


@pytest.mark.parametrize("name", MINI)
def test_grouped_ffn_matches_oracle(name):
    w = synth.WORKLOADS[name]
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    g = _grouped(w, inp, dev, cfg)
    y = to_f64(g["y"])
    off, src, R = g["offsets"], g["src"], g["R"]
    x64 = inp.f64["x"]
    for e in range(w.n_experts):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        ref = O.expert_mlp(x64[src[lo:hi]], *inp.expert(e))
        assert_close(y[lo:hi], ref, out_tolerance(w), f"{name} expert {e}")
    for s in range(w.n_shared):
        ref = O.expert_mlp(x64, *inp.expert(w.n_experts + s))
        assert_close(y[R + s * w.T:R + (s + 1) * w.T], ref, out_tolerance(w), f"{name} shared")


@pytest.mark.parametrize("name", MINI)
def test_combine_matches_oracle(name):
    w = synth.WORKLOADS[name]
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    g = _grouped(w, inp, dev, cfg)
    out = torch.empty(w.T, w.d_model, dtype=dev["x"].dtype, device="cuda")
    moe.moe_combine(cfg, g["y"], g["dest"], g["gate_t"], out, g["ws"])
    assert moe.moe_get_device_error(g["ws"]) == moe.MOE_OK
    y = to_f64(g["y"])
    R = g["R"]
    shared = None
    if w.n_shared:
        shared = sum(y[R + s * w.T:R + (s + 1) * w.T] for s in range(w.n_shared))
    ref = O.combine(g["dest_np"], g["gate"], y[:R], shared, w.d_model)
    # only the final rounding of out (bf16: 2^-9 relative) separates the two
    assert_close(to_f64(out), ref, 4e-3 if w.dtype == "bf16" else 1e-6, f"{name} combine")


def test_router_nan_token_gets_distinct_ids():
    # a token whose logits are all NaN still gets k distinct ids in [0, E); the others are unaffected
    w = synth.WORKLOADS["mini_qwen3"].with_(T=150, n_experts=40, top_k=8)
    inp = Inputs(w)
    dev = inp.device()
    dev["x"][3] = float("nan")
    idx, gate, _, _, _ = _router(w, inp, dev, cfg_of(w))
    row = idx[3]
    assert len(set(row.tolist())) == w.top_k and ((row >= 0) & (row < w.n_experts)).all()
    keep = np.ones(w.T, dtype=bool)
    keep[3] = False
    ref_scores = O.scores_from_logits(O.router_logits(inp.f64["x"], inp.f64["w_router"], inp.bias), w.score)
    check_routing(idx[keep], ref_scores[keep], w.top_k)


@pytest.mark.parametrize("name", MINI)
def test_routing_stats_match_oracle(name):
    w = synth.WORKLOADS[name]
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    ws = moe.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d_model, dtype=dev["x"].dtype, device="cuda")
    counts = torch.empty(w.n_experts, dtype=torch.int32, device="cuda")
    moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"], dev["w_down"],
                          out, ws, counts_out=counts)
    got = moe.routing_stats_to_dict(moe.moe_routing_stats(cfg, counts))
    ref = O.routing_stats(counts.cpu().numpy(), T=w.T, cap=moe.moe_capacity(cfg))
    for key in ("tokens", "pairs", "kept", "dropped", "experts_touched", "max_load", "capacity"):
        assert got[key] == ref[key], key
    for key in ("mean_load", "efficiency"):
        assert abs(got[key] - float(ref[key])) <= 2.0 ** -23 * float(ref[key]), key
