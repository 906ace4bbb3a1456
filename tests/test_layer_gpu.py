"""Whole-layer parity (moe_layer_forward) against the fp64 oracle.

Reduced workloads: every output element is compared. Full-size workloads (the
five model-shaped layers, run exactly as the benchmark runs them, inputs
generated on the device): routing and per-expert counts are compared for every
token; the layer output for every token of the decode batch and the tiny layer,
and for the prefill layers a seeded sample of tokens that includes the first and
last token, tokens of the busiest expert and (with capacity) fully or partly
dropped tokens. The oracle regenerates the same inputs on the host.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import (Inputs, assert_close, cfg_of, check_routing, oracle_gates_for, out_tolerance, to_f64)

pytestmark = pytest.mark.gpu


def _run_layer(w, dev, cfg):
    out = torch.full((w.T, w.d_model), float("nan"), dtype=dev["x"].dtype, device="cuda")
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device="cuda")
    counts = torch.empty(w.n_experts, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"], dev["w_down"],
                          out, ws, topk_idx_out=idx, counts_out=counts)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    return out, idx.cpu().numpy(), counts.cpu().numpy()


def _oracle_on_gpu_routing(w, x64, wr64, bias, experts, gpu_idx, tokens=None):
    ref_scores = O.scores_from_logits(O.router_logits(x64, wr64, bias), w.score)
    swapped = check_routing(gpu_idx, ref_scores, w.top_k)
    gates = oracle_gates_for(gpu_idx, ref_scores, w.renormalize)
    res = O.layer_forward(x64, wr64, bias, experts, top_k=w.top_k, score=w.score, renormalize=w.renormalize,
                          capacity_factor=w.capacity_factor, n_shared=w.n_shared, tokens=tokens,
                          routing=(gpu_idx, gates))
    return res, swapped


@pytest.mark.parametrize("name", synth.workloads.MINI)
def test_layer_reduced(name):
    w = synth.WORKLOADS[name]
    inp = Inputs(w)
    out, idx, counts = _run_layer(w, inp.device(), cfg_of(w))
    res, _ = _oracle_on_gpu_routing(w, inp.f64["x"], inp.f64["w_router"], inp.bias, inp.expert, idx)
    assert (counts == res.disp.counts).all()
    assert_close(to_f64(out), res.out, out_tolerance(w), name)


@pytest.mark.parametrize("name,edit", [
    ("mini_mixtral", dict(T=1)),                                   # a single token
    ("mini_mixtral", dict(T=129)),                                 # one row past a tile
    ("mini_qwen3", dict(top_k=1)),                                 # a single expert per token
    ("mini_decode", dict(T=3, n_experts=8, top_k=8)),              # k = E: every expert, uniform-ish gates
    ("mini_deepseek", dict(capacity_factor=0.05)),                 # cap 1: almost everything dropped
    ("mini_deepseek", dict(capacity_factor=100.0)),                # cap >= T: same as dropless
    ("mini_mixtral", dict(renormalize=False)),
    ("mini_deepseek", dict(score="softmax", n_shared=0)),
    ("tiny_f32", dict(n_shared=1, score="sigmoid", capacity_factor=1.0, T=70)),
])
def test_layer_edge_cases(name, edit):
    w = synth.WORKLOADS[name].with_(**edit)
    inp = Inputs(w)
    out, idx, counts = _run_layer(w, inp.device(), cfg_of(w))
    res, _ = _oracle_on_gpu_routing(w, inp.f64["x"], inp.f64["w_router"], inp.bias, inp.expert, idx)
    assert (counts == res.disp.counts).all()
    assert_close(to_f64(out), res.out, out_tolerance(w), f"{name} {edit}")


def test_layer_empty_experts():
    # a strong bias sends every token to the same few experts: most groups are empty
    w = synth.WORKLOADS["mini_qwen3"].with_(bias_s=8.0, top_k=2)
    inp = Inputs(w)
    out, idx, counts = _run_layer(w, inp.device(), cfg_of(w))
    assert (counts == 0).sum() > w.n_experts // 2
    res, _ = _oracle_on_gpu_routing(w, inp.f64["x"], inp.f64["w_router"], inp.bias, inp.expert, idx)
    assert_close(to_f64(out), res.out, out_tolerance(w), "empty experts")


def test_layer_repeatable():
    w = synth.WORKLOADS["mini_deepseek"]
    dev = Inputs(w).device()
    a, ia, _ = _run_layer(w, dev, cfg_of(w))
    b, ib, _ = _run_layer(w, dev, cfg_of(w))
    assert (ia == ib).all()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name,edit", [
    ("mini_deepseek", dict(T=64, n_experts=256, top_k=8)),        # the most experts
    ("mini_deepseek", dict(T=64, n_experts=149, top_k=6)),        # one past the SM count
    ("mini_qwen3", dict(T=33, n_experts=148, top_k=4)),           # tokens not a multiple of 8
    ("mini_decode", dict(T=1, n_experts=5, top_k=2)),
    ("tiny_f32", dict(T=40, d_model=72, score="sigmoid")),
])
def test_layer_small_batches_repeat_on_one_workspace(name, edit):
    # Decode-sized batches with expert counts around and above the SM count, called three times
    # on one workspace: every call routes and computes identically, and matches the oracle.
    w = synth.WORKLOADS[name].with_(**edit)
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    ws = moe.alloc_workspace(cfg)
    outs, idxs = [], []
    for _ in range(3):
        out = torch.full((w.T, w.d_model), float("nan"), dtype=dev["x"].dtype, device="cuda")
        idx = torch.full((w.T, w.top_k), -1, dtype=torch.int32, device="cuda")
        moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"],
                              dev["w_down"], out, ws, topk_idx_out=idx)
        assert moe.moe_get_device_error(ws) == moe.MOE_OK
        outs.append(out)
        idxs.append(idx.cpu().numpy())
    assert all((i == idxs[0]).all() for i in idxs[1:])
    assert all(torch.equal(o, outs[0]) for o in outs[1:])
    res, _ = _oracle_on_gpu_routing(w, inp.f64["x"], inp.f64["w_router"], inp.bias, inp.expert, idxs[0])
    assert_close(to_f64(outs[0]), res.out, out_tolerance(w), f"{name} {edit}")


# ------------------------------------------------------------- full sizes

def _sample_tokens(w, idx, dest_row, n=32):
    if w.T <= 64:                                   # the decode batch and the tiny layer: every token
        return np.arange(w.T, dtype=np.int64)
    rng = np.random.default_rng(1234)
    toks = {0, w.T - 1}
    toks |= set(rng.choice(w.T, size=min(n, w.T), replace=False).tolist())
    busiest = np.bincount(idx.ravel(), minlength=w.n_experts).argmax()
    toks |= set(np.nonzero((idx == busiest).any(axis=1))[0][-2:].tolist())
    if dest_row is not None:
        dropped = np.nonzero((dest_row < 0).any(axis=1))[0]
        toks |= set(dropped[:2].tolist())
        full = np.nonzero((dest_row < 0).all(axis=1))[0]
        toks |= set(full[:1].tolist())
    return np.array(sorted(toks), dtype=np.int64)


@pytest.mark.parametrize("name", synth.workloads.FULL + synth.workloads.FULL_EXTRA)
def test_layer_full_size_sampled(name):
    w = synth.WORKLOADS[name]
    cfg = cfg_of(w)
    dev = synth.device_inputs(w)
    out, idx, counts = _run_layer(w, dev, cfg)
    x64 = synth.as_f64(synth.host_tensor(w, "x"), w.dtype)
    wr64 = synth.as_f64(synth.host_tensor(w, "w_router"), w.dtype)
    bias = synth.router_bias(w.n_experts, w.bias_s)
    # routing and counts for every token
    ref_scores = O.scores_from_logits(O.router_logits(x64, wr64, bias), w.score)
    check_routing(idx, ref_scores, w.top_k)
    disp = O.dispatch(idx, w.n_experts, O.capacity(w.T, w.top_k, w.n_experts, w.capacity_factor))
    assert (counts == disp.counts).all()
    toks = _sample_tokens(w, idx, disp.dest_row)
    cache = {}

    def experts(g):
        if g not in cache:
            cache.clear()
            cache[g] = tuple(synth.as_f64(a, w.dtype) for a in synth.host_expert(w, g))
        return cache[g]

    res, _ = _oracle_on_gpu_routing(w, x64, wr64, bias, experts, idx, tokens=toks)
    got = to_f64(out[torch.from_numpy(toks).cuda()])
    assert_close(got, res.out, out_tolerance(w), name)
    del dev
    torch.cuda.empty_cache()


# ------------------------------------------------- fused down-projection + combine

@pytest.mark.parametrize("name,edit", [
    ("mini_mixtral", {}),
    ("mini_qwen3", {}),
    ("mini_deepseek", {}),                                         # drops, shared expert (weight one)
    ("mini_decode", {}),
    ("mini_deepseek", dict(capacity_factor=0.05)),                 # almost everything dropped
    ("mini_mixtral", dict(T=1)),
    ("mini_qwen3", dict(top_k=1)),                                 # accumulator larger than the grouped rows
    ("mini_qwen3", dict(bias_s=8.0, top_k=2)),                     # mostly empty experts
])
def test_layer_fused_combine(name, edit, monkeypatch):
    # the down projection adds gate * y into a float32 accumulator in its epilogue, then one
    # rounding pass writes the output: same oracle comparison as the separate combine
    monkeypatch.setenv("MOE_FUSED_COMBINE", "1")
    w = synth.WORKLOADS[name].with_(**edit)
    inp = Inputs(w)
    out, idx, counts = _run_layer(w, inp.device(), cfg_of(w))
    res, _ = _oracle_on_gpu_routing(w, inp.f64["x"], inp.f64["w_router"], inp.bias, inp.expert, idx)
    assert (counts == res.disp.counts).all()
    assert_close(to_f64(out), res.out, out_tolerance(w), f"fused {name} {edit}")


def test_layer_fused_combine_full_size_qwen3(monkeypatch):
    w = synth.WORKLOADS["qwen3_30b_a3b"]
    cfg = cfg_of(w)
    dev = synth.device_inputs(w)
    ref_out, ref_idx, _ = _run_layer(w, dev, cfg)                  # the separate combine
    monkeypatch.setenv("MOE_FUSED_COMBINE", "1")
    out, idx, _ = _run_layer(w, dev, cfg)
    assert (idx == ref_idx).all()
    # both are within 1e-2 of the oracle; against each other they differ by the rounding of y
    # to bf16 (separate path) and the order of the float32 additions
    assert_close(to_f64(out), to_f64(ref_out), 1e-2, "fused vs separate combine")
    del dev
    torch.cuda.empty_cache()


# ------------------------------------------- both contractions in one persistent launch

@pytest.mark.parametrize("name,edit", [
    ("mini_mixtral", {}),
    ("mini_qwen3", {}),
    ("mini_deepseek", {}),                                         # drops, shared expert
    ("mini_decode", {}),
    ("mini_mixtral", dict(T=1)),
    ("mini_qwen3", dict(bias_s=8.0, top_k=2)),                     # mostly empty experts
    ("mini_mixtral", dict(T=1200)),                                # ten-tile experts
    ("mini_deepseek", dict(capacity_factor=0.05)),
])
def test_layer_fused_mlp_is_bit_identical(name, edit, monkeypatch):
    # MOE_FUSED_MLP=1: the gate/up and down tiles in one launch, down tiles of an m-tile started
    # once its h rows are published (the default for single-chunk batches); =0: two launches.
    # Same tiles, same arithmetic: the outputs agree bit for bit, and with the oracle within
    # the usual tolerance
    w = synth.WORKLOADS[name].with_(**edit)
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    monkeypatch.setenv("MOE_FUSED_MLP", "0")                      # two launches
    ref_out, ref_idx, _ = _run_layer(w, dev, cfg)
    monkeypatch.setenv("MOE_FUSED_MLP", "1")
    out, idx, counts = _run_layer(w, dev, cfg)
    assert (idx == ref_idx).all()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    res, _ = _oracle_on_gpu_routing(w, inp.f64["x"], inp.f64["w_router"], inp.bias, inp.expert, idx)
    assert_close(to_f64(out), res.out, out_tolerance(w), f"fused mlp {name} {edit}")


@pytest.mark.parametrize("name", ["mixtral_8x7b", "qwen3_30b_a3b", "deepseek_v3", "decode_qwen3"])
def test_layer_fused_mlp_full_size_bit_identical(name, monkeypatch):
    w = synth.WORKLOADS[name]
    cfg = cfg_of(w)
    dev = synth.device_inputs(w)
    monkeypatch.setenv("MOE_FUSED_MLP", "0")                      # two launches
    ref_out, ref_idx, _ = _run_layer(w, dev, cfg)
    monkeypatch.setenv("MOE_FUSED_MLP", "1")
    for _ in range(2):                                             # twice: the counters restart
        out, idx, _ = _run_layer(w, dev, cfg)
        assert (idx == ref_idx).all()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    del dev
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,edit,force_one_launch", [
    ("mini_decode", {}, False),
    ("mini_decode", dict(T=1), False),
    ("mini_qwen3", dict(T=128), False),                            # one full chunk
    ("mini_qwen3", dict(T=100, capacity_factor=0.05), False),      # tokens with every slot dropped
    ("mini_deepseek", dict(T=128), False),                         # shared expert, drops, sigmoid
    ("mini_mixtral", dict(T=64), False),
    ("mini_qwen3", {}, True),                                      # three chunks, one launch forced
])
def test_layer_mlp_combine_is_bit_identical(name, edit, force_one_launch, monkeypatch):
    # MOE_MLP_COMBINE=1: the one-launch expert MLP combines in its down tiles: each (row, down
    # n-tile) is counted on its token, and the tile that completes a token sums the token's rows
    # in slot order, the arithmetic of the separate combine kernel (=0). Outputs agree bit for
    # bit; tokens that no row reaches get zero rows
    w = synth.WORKLOADS[name].with_(**edit)
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    if force_one_launch:
        monkeypatch.setenv("MOE_FUSED_MLP", "1")
    monkeypatch.setenv("MOE_MLP_COMBINE", "0")
    n_sep = moe.moe_layer_launch_count(cfg)
    ref_out, ref_idx, _ = _run_layer(w, dev, cfg)
    monkeypatch.setenv("MOE_MLP_COMBINE", "1")
    assert moe.moe_layer_launch_count(cfg) == n_sep - 1
    out, idx, _ = _run_layer(w, dev, cfg)
    assert (idx == ref_idx).all()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    res, _ = _oracle_on_gpu_routing(w, inp.f64["x"], inp.f64["w_router"], inp.bias, inp.expert, idx)
    assert_close(to_f64(out), res.out, out_tolerance(w), f"mlp combine {name} {edit}")
