"""W8A8: FP8 (E4M3) expert weights and E4M3 activations on the 8-bit tensor-core path, against
the fp64 oracle's expert_mlp_w8a8 reading (activation rows quantised per row like the weights,
h stored in bf16 and quantised) run on the GPU's routing and the dequantized weights."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, assert_close, cfg_of, check_routing, oracle_gates_for, out_tolerance, to_f64

pytestmark = pytest.mark.gpu


def _quantized(dev):
    """GPU codes and scales of the three weight tensors, checked bit for bit against the oracle's."""
    out = {}
    for name in ("w_gate", "w_up", "w_down"):
        q, s = moe.moe_quantize_fp8_rows(dev[name])
        ref_q, ref_s = O.quantize_fp8_rows(dev[name].float().cpu().numpy())
        assert np.array_equal(q.cpu().numpy(), ref_q), name
        assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32)), name
        out[name] = (q, s, O.dequantize_fp8_rows(ref_q, ref_s))
    return out


def _run(w, dev, qw, cfg):
    ws = moe.alloc_workspace(cfg)
    out = torch.full((w.T, w.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device="cuda")
    moe.moe_layer_forward_w8a8(cfg, dev["x"], dev["w_router"], dev["bias"], *qw["w_gate"][:2], *qw["w_up"][:2],
                               *qw["w_down"][:2], out, ws, topk_idx_out=idx)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    return out, idx.cpu().numpy()


LAYER_CASES = {
    "mini_qwen3": ("mini_qwen3", {}),
    "mini_deepseek": ("mini_deepseek", {}),                        # capacity drops, shared expert
    "mini_mixtral": ("mini_mixtral", {}),
    "mini_decode": ("mini_decode", {}),
    # d_ff of 384: three 128-feature gate/up tiles, a down reduction of three 128-code k-steps
    "f384": ("mini_qwen3", {"d_ff": 384}),
    # ~2400 kept pairs over 8 skewed experts: the largest expert spans ten 128-row tiles
    "many_blocks": ("mini_mixtral", {"T": 1200}),
    "one_token": ("mini_mixtral", {"T": 1}),
    # capacity 2 per expert: fewer grouped rows (96) than tokens (257), most pairs dropped
    "cap_small": ("mini_deepseek", {"capacity_factor": 0.05}),
}


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_layer_w8a8_matches_oracle(name):
    base, over = LAYER_CASES[name]
    w = synth.WORKLOADS[base].with_(**over)
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    qw = _quantized(dev)
    out, gidx = _run(w, dev, qw, cfg)
    x64, wr64 = inp.f64["x"], inp.f64["w_router"]
    scores = O.scores_from_logits(O.router_logits(x64, wr64, inp.bias), w.score)
    check_routing(gidx, scores, w.top_k)
    experts = lambda g: (qw["w_gate"][2][g], qw["w_up"][2][g], qw["w_down"][2][g])
    ref = O.layer_forward(x64, wr64, inp.bias, experts, top_k=w.top_k, score=w.score, renormalize=w.renormalize,
                          capacity_factor=w.capacity_factor, n_shared=w.n_shared, mlp=O.expert_mlp_w8a8,
                          routing=(gidx, oracle_gates_for(gidx, scores, w.renormalize)))
    assert_close(to_f64(out), ref.out, out_tolerance(w), name + " w8a8")


@pytest.mark.parametrize("name,tokens", [("decode_qwen3", None), ("qwen3_30b_a3b", [0, 1000, 4095, 8191])])
def test_layer_w8a8_full_size(name, tokens):
    w = synth.WORKLOADS[name]
    cfg = cfg_of(w)
    dev = synth.device_inputs(w)
    qw = {n: moe.moe_quantize_fp8_rows(dev[n]) for n in ("w_gate", "w_up", "w_down")}
    for n in ("w_gate", "w_up", "w_down"):
        del dev[n]
    out, gidx = _run(w, dev, {n: (*qw[n], None) for n in qw}, cfg)
    x64 = synth.as_f64(synth.host_tensor(w, "x"), w.dtype)
    wr64 = synth.as_f64(synth.host_tensor(w, "w_router"), w.dtype)
    scores = O.scores_from_logits(O.router_logits(x64, wr64, None), w.score)
    check_routing(gidx, scores, w.top_k)
    toks = np.arange(w.T) if tokens is None else np.array(tokens)
    cache = {}

    def experts(g):
        if g not in cache:
            cache.clear()
            raw = synth.host_expert(w, g)
            cache[g] = tuple(O.dequantize_fp8_rows(*O.quantize_fp8_rows(synth.as_f64(a, w.dtype).astype(np.float32)))
                             for a in raw)
        return cache[g]

    ref = O.layer_forward(x64, wr64, None, experts, top_k=w.top_k, score=w.score, tokens=toks,
                          mlp=O.expert_mlp_w8a8, routing=(gidx, oracle_gates_for(gidx, scores, w.renormalize)))
    assert_close(to_f64(out[torch.from_numpy(toks).cuda()]), ref.out, out_tolerance(w), name + " w8a8")


def test_w8a8_differs_from_fp8_by_the_activation_quantisation():
    # the same layer with bf16 activations (FP8 weights only) and with E4M3 activations: the two
    # outputs differ by more than float32 noise and less than E4M3's relative precision
    w = synth.WORKLOADS["mini_qwen3"]
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    qw = _quantized(dev)
    a8, _ = _run(w, dev, qw, cfg)
    ws = moe.alloc_workspace(cfg)
    w8 = torch.empty_like(a8)
    moe.moe_layer_forward_fp8(cfg, dev["x"], dev["w_router"], dev["bias"], *qw["w_gate"][:2], *qw["w_up"][:2],
                              *qw["w_down"][:2], w8, ws)
    rel = float((a8.float() - w8.float()).abs().max() / w8.float().abs().max())
    assert 1e-3 < rel < 8e-2, rel


@pytest.mark.parametrize("edit,dtype", [({"d_model": 384}, torch.bfloat16), ({}, torch.float32)])
def test_w8a8_refuses_shapes_it_does_not_take(edit, dtype):
    # d_model not a multiple of 256, and float32 layers
    w = synth.WORKLOADS["mini_qwen3" if dtype == torch.bfloat16 else "tiny_f32"].with_(**edit)
    cfg = cfg_of(w)
    dev = Inputs(w).device()
    q = {n: moe.moe_quantize_fp8_rows(dev[n].to(torch.bfloat16)) for n in ("w_gate", "w_up", "w_down")}
    ws = moe.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d_model, dtype=dtype, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward_w8a8(cfg, dev["x"], dev["w_router"], dev["bias"], *q["w_gate"], *q["w_up"],
                                   *q["w_down"], out, ws)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("name,edit", [("mini_decode", {}), ("mini_deepseek", {}), ("mini_qwen3", {}),
                                       ("mini_mixtral", {"T": 1200}), ("mini_deepseek", {"capacity_factor": 0.05}),
                                       ("decode_qwen3", {})])
def test_w8a8_one_launch_mlp_is_bit_identical(name, edit, monkeypatch):
    # MOE_FUSED_MLP=1: gate/up tiles, h's per-row quantisation by the tile that completes each
    # 128-row block, and the down tiles in one launch (the default for single-chunk batches);
    # =0: three launches. Same arithmetic: the outputs agree bit for bit.
    w = synth.WORKLOADS[name].with_(**edit)
    dev = synth.device_inputs(w) if not name.startswith("mini") else Inputs(w).device()
    cfg = cfg_of(w)
    qw = {n: moe.moe_quantize_fp8_rows(dev[n]) for n in ("w_gate", "w_up", "w_down")}
    outs = []
    for mode in ("0", "1", "1"):                                 # twice with one launch: counters restart
        monkeypatch.setenv("MOE_FUSED_MLP", mode)
        outs.append(_run(w, dev, {n: (*qw[n], None) for n in qw}, cfg))
    assert all((o[1] == outs[0][1]).all() for o in outs[1:])
    assert all(torch.equal(o[0].view(torch.int16), outs[0][0].view(torch.int16)) for o in outs[1:])
