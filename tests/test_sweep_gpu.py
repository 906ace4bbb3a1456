"""Whole-layer parity over a seeded sweep of layer shapes, against the fp64 oracle.

Each case draws tokens, widths, experts, top-k, shared expert, score function, gate
renormalisation, capacity and router-bias skew from a fixed seed (so the case list is the same
on every run), runs moe_layer_forward, and compares routing, counts and every output element
with the oracle re-run on the GPU's routing. bf16 cases whose shapes the FP8 kernels take are
also run with FP8 weights against the oracle on the dequantized weights, and with FP8 weights
and activations (W8A8) against the oracle's W8A8 reading.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, assert_close, cfg_of, check_routing, oracle_gates_for, out_tolerance, to_f64

pytestmark = pytest.mark.gpu


def _draw_cases(n_bf16=18, n_f32=6, seed=2024):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n_bf16 + n_f32):
        f32 = i >= n_bf16
        E = int(rng.choice([2, 5, 8, 16, 33, 64, 128, 256]))
        k = int(rng.integers(1, min(8, E) + 1))
        step = 4 if f32 else 128
        d = step * int(rng.integers(1, (256 if f32 else 1024) // step + 1))
        F = step * int(rng.integers(1, (256 if f32 else 512) // step + 1))
        T = int(rng.choice([1, 2, 7, 31, 64, 127, 129, 200, 333, 517]))
        cases.append(synth.Workload(
            f"sweep{i}", T=T, d_model=d, n_experts=E, top_k=k, d_ff=F,
            n_shared=int(rng.integers(0, 2)), score=str(rng.choice(["softmax", "sigmoid"])),
            renormalize=bool(rng.random() < 0.8),
            capacity_factor=float(rng.choice([0.0, 0.0, 0.5, 1.0, 1.25, 2.0])),
            bias_s=float(rng.choice([0.0, 0.0, 1.0, 2.5])),
            x_sigma=0.02 if f32 else 1.0, dtype="f32" if f32 else "bf16", seed=1000 + i))
    return cases


CASES = _draw_cases()


def _oracle_on_gpu_routing(w, inp, experts, gpu_idx):
    ref_scores = O.scores_from_logits(O.router_logits(inp.f64["x"], inp.f64["w_router"], inp.bias), w.score)
    check_routing(gpu_idx, ref_scores, w.top_k)
    gates = oracle_gates_for(gpu_idx, ref_scores, w.renormalize)
    return O.layer_forward(inp.f64["x"], inp.f64["w_router"], inp.bias, experts, top_k=w.top_k, score=w.score,
                           renormalize=w.renormalize, capacity_factor=w.capacity_factor, n_shared=w.n_shared,
                           routing=(gpu_idx, gates))


@pytest.mark.parametrize("w", CASES, ids=lambda w: (f"{w.name}-{w.dtype}-T{w.T}-d{w.d_model}-E{w.n_experts}"
                                                      f"-k{w.top_k}-F{w.d_ff}-S{w.n_shared}-{w.score}"
                                                      f"-cf{w.capacity_factor}"))
def test_layer_sweep(w):
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    out = torch.full((w.T, w.d_model), float("nan"), dtype=dev["x"].dtype, device="cuda")
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device="cuda")
    counts = torch.empty(w.n_experts, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"], dev["w_down"],
                          out, ws, topk_idx_out=idx, counts_out=counts)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    gidx = idx.cpu().numpy()
    res = _oracle_on_gpu_routing(w, inp, inp.expert, gidx)
    assert (counts.cpu().numpy() == res.disp.counts).all()
    assert_close(to_f64(out), res.out, out_tolerance(w), w.name)

    if w.dtype != "bf16" or w.d_model % 256 != 0:
        return
    # the same layer with FP8 weights, against the oracle on the dequantized weights
    q = {}
    for n in ("w_gate", "w_up", "w_down"):
        codes, scale = moe.moe_quantize_fp8_rows(dev[n])
        q[n] = (codes, scale, O.dequantize_fp8_rows(codes.cpu().numpy(), scale.cpu().numpy()))
    out8 = torch.full_like(out, float("nan"))
    idx8 = torch.empty_like(idx)
    moe.moe_layer_forward_fp8(cfg, dev["x"], dev["w_router"], dev["bias"], q["w_gate"][0], q["w_gate"][1],
                              q["w_up"][0], q["w_up"][1], q["w_down"][0], q["w_down"][1], out8, ws,
                              topk_idx_out=idx8)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    assert torch.equal(idx8, idx)                      # the router does not see the expert weights
    experts8 = lambda g: (q["w_gate"][2][g], q["w_up"][2][g], q["w_down"][2][g])
    res8 = _oracle_on_gpu_routing(w, inp, experts8, gidx)
    assert_close(to_f64(out8), res8.out, out_tolerance(w), w.name + " fp8")

    # and with E4M3 activations as well (W8A8), against the oracle's W8A8 reading
    outa = torch.full_like(out, float("nan"))
    moe.moe_layer_forward_w8a8(cfg, dev["x"], dev["w_router"], dev["bias"], q["w_gate"][0], q["w_gate"][1],
                               q["w_up"][0], q["w_up"][1], q["w_down"][0], q["w_down"][1], outa, ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    resa = O.layer_forward(inp.f64["x"], inp.f64["w_router"], inp.bias, experts8, top_k=w.top_k, score=w.score,
                           renormalize=w.renormalize, capacity_factor=w.capacity_factor, n_shared=w.n_shared,
                           mlp=O.expert_mlp_w8a8,
                           routing=(gidx, oracle_gates_for(gidx, O.scores_from_logits(
                               O.router_logits(inp.f64["x"], inp.f64["w_router"], inp.bias), w.score),
                               w.renormalize)))
    assert_close(to_f64(outa), resa.out, out_tolerance(w), w.name + " w8a8")
