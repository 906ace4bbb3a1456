"""FP8 (E4M3) expert weights: the quantiser against the oracle's, bit for bit, and layers with
FP8 weights against the fp64 oracle run on the dequantized weights."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, assert_close, cfg_of, check_routing, oracle_gates_for, out_tolerance, to_f64

pytestmark = pytest.mark.gpu


def _bf16_as_f32(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("shape", [(37, 128), (256, 2048), (3, 16)])
def test_quantizer_matches_oracle_bit_for_bit(shape):
    g = torch.Generator().manual_seed(shape[0] * 7 + shape[1])
    w = (torch.randn(shape, generator=g) * 0.02).to(torch.bfloat16)
    w[0] = 0.0                                   # an all-zero row
    w[-1, :5] = torch.tensor([448.0, -3.0e-6, 1.0e-30, -0.0, 7.5]).to(torch.bfloat16)
    wd = w.cuda()
    q, s = moe.moe_quantize_fp8_rows(wd)
    ref_q, ref_s = O.quantize_fp8_rows(_bf16_as_f32(w))
    assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), ref_q)


def _quantized(dev, w):
    """GPU codes and scales of the three weight tensors, checked against the oracle's."""
    out = {}
    for name in ("w_gate", "w_up", "w_down"):
        q, s = moe.moe_quantize_fp8_rows(dev[name])
        ref_q, ref_s = O.quantize_fp8_rows(_bf16_as_f32(dev[name]))
        assert np.array_equal(q.cpu().numpy(), ref_q), name
        assert np.array_equal(s.cpu().numpy().view(np.uint32), ref_s.view(np.uint32)), name
        out[name] = (q, s, O.dequantize_fp8_rows(ref_q, ref_s))
    return out


LAYER_CASES = {
    "mini_qwen3": ("mini_qwen3", {}),
    "mini_deepseek": ("mini_deepseek", {}),
    "mini_mixtral": ("mini_mixtral", {}),
    "mini_decode": ("mini_decode", {}),
    # d_ff of 384: three 128-feature gate/up tiles, a down-GEMM reduction of six 64-wide k-steps
    "f384": ("mini_qwen3", {"d_ff": 384}),
    # ~2400 kept pairs over 8 skewed experts: the largest expert spans ten 128-row tiles, the last ragged
    "many_blocks": ("mini_mixtral", {"T": 1200}),
}


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_layer_fp8_matches_oracle(name):
    base, over = LAYER_CASES[name]
    w = synth.WORKLOADS[base].with_(**over) if over else synth.WORKLOADS[base]
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    qw = _quantized(dev, w)
    ws = moe.alloc_workspace(cfg)
    out = torch.full((w.T, w.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device="cuda")
    moe.moe_layer_forward_fp8(cfg, dev["x"], dev["w_router"], dev["bias"], qw["w_gate"][0], qw["w_gate"][1],
                              qw["w_up"][0], qw["w_up"][1], qw["w_down"][0], qw["w_down"][1], out, ws,
                              topk_idx_out=idx)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    gidx = idx.cpu().numpy()
    x64, wr64 = inp.f64["x"], inp.f64["w_router"]
    scores = O.scores_from_logits(O.router_logits(x64, wr64, inp.bias), w.score)
    check_routing(gidx, scores, w.top_k)
    experts = lambda g: (qw["w_gate"][2][g], qw["w_up"][2][g], qw["w_down"][2][g])
    ref = O.layer_forward(x64, wr64, inp.bias, experts, top_k=w.top_k, score=w.score, renormalize=w.renormalize,
                          capacity_factor=w.capacity_factor, n_shared=w.n_shared,
                          routing=(gidx, oracle_gates_for(gidx, scores, w.renormalize)))
    assert_close(to_f64(out), ref.out, out_tolerance(w), name + " fp8")


def test_grouped_ffn_fp8_stage_matches_oracle():
    w = synth.WORKLOADS["mini_deepseek"]
    inp = Inputs(w)
    dev = inp.device()
    cfg = cfg_of(w)
    qw = _quantized(dev, w)
    E, T, k = w.n_experts, w.T, w.top_k
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gate = torch.empty(T, k, dtype=torch.float32, device="cuda")
    moe.moe_router_topk(cfg, dev["x"], dev["w_router"], dev["bias"], idx, gate)
    R = moe.moe_rows_capacity(cfg)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dest = torch.empty(T, k, dtype=torch.int32, device="cuda")
    src = torch.empty(R, dtype=torch.int32, device="cuda")
    xp = torch.empty(R, w.d_model, dtype=torch.bfloat16, device="cuda")
    y = torch.full((moe.moe_grouped_rows(cfg), w.d_model), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.moe_permute(cfg, idx, dev["x"], counts, offsets, dest, src, xp, ws)
    moe.moe_grouped_ffn_fp8(cfg, xp, offsets, dev["x"], qw["w_gate"][0], qw["w_gate"][1], qw["w_up"][0],
                            qw["w_up"][1], qw["w_down"][0], qw["w_down"][1], y, ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    off, srcn, yn, x64 = offsets.cpu().numpy(), src.cpu().numpy(), to_f64(y), inp.f64["x"]
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            ref = O.expert_mlp(x64[srcn[lo:hi]], qw["w_gate"][2][e], qw["w_up"][2][e], qw["w_down"][2][e])
            assert_close(yn[lo:hi], ref, out_tolerance(w), f"expert {e}")
    ref = O.expert_mlp(x64, qw["w_gate"][2][E], qw["w_up"][2][E], qw["w_down"][2][E])
    assert_close(yn[R:R + T], ref, out_tolerance(w), "shared")


def test_layer_fp8_full_size_decode_sampled():
    w = synth.WORKLOADS["decode_qwen3"]
    cfg = cfg_of(w)
    dev = synth.device_inputs(w)
    q = {n: moe.moe_quantize_fp8_rows(dev[n]) for n in ("w_gate", "w_up", "w_down")}
    ws = moe.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d_model, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device="cuda")
    moe.moe_layer_forward_fp8(cfg, dev["x"], dev["w_router"], dev["bias"], *q["w_gate"], *q["w_up"], *q["w_down"],
                              out, ws, topk_idx_out=idx)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    gidx = idx.cpu().numpy()
    x64 = synth.as_f64(synth.host_tensor(w, "x"), w.dtype)
    wr64 = synth.as_f64(synth.host_tensor(w, "w_router"), w.dtype)
    scores = O.scores_from_logits(O.router_logits(x64, wr64, None), w.score)
    check_routing(gidx, scores, w.top_k)
    toks = np.array([0, 7, 19, w.T - 1])
    cache = {}

    def experts(g):
        if g not in cache:
            raw = synth.host_expert(w, g)
            cache[g] = tuple(O.dequantize_fp8_rows(*O.quantize_fp8_rows(synth.as_f64(a, w.dtype).astype(np.float32)))
                             for a in raw)
        return cache[g]

    ref = O.layer_forward(x64, wr64, None, experts, top_k=w.top_k, score=w.score, tokens=toks,
                          routing=(gidx, oracle_gates_for(gidx, scores, w.renormalize)))
    assert_close(to_f64(out[torch.from_numpy(toks).cuda()]), ref.out, out_tolerance(w), "decode fp8")


def test_fp8_refuses_shapes_it_does_not_take():
    w = synth.WORKLOADS["mini_qwen3"].with_(d_model=384)          # d_model not a multiple of 256
    cfg = cfg_of(w)
    dev = Inputs(w).device()
    q = {n: moe.moe_quantize_fp8_rows(dev[n]) for n in ("w_gate", "w_up", "w_down")}
    ws = moe.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d_model, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward_fp8(cfg, dev["x"], dev["w_router"], dev["bias"], *q["w_gate"], *q["w_up"],
                                  *q["w_down"], out, ws)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED


def test_fp8_refuses_float32_activations():
    w = synth.WORKLOADS["tiny_f32"]
    cfg = cfg_of(w)
    dev = Inputs(w).device()
    q = {n: moe.moe_quantize_fp8_rows(dev[n].to(torch.bfloat16)) for n in ("w_gate", "w_up", "w_down")}
    ws = moe.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d_model, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_layer_forward_fp8(cfg, dev["x"], dev["w_router"], dev["bias"], *q["w_gate"], *q["w_up"],
                                  *q["w_down"], out, ws)
    assert ei.value.code == moe.MOE_ERR_UNSUPPORTED


@pytest.mark.parametrize("T", [256, 32, 8])
@pytest.mark.parametrize("which", ["gate", "up", "down"])
def test_every_e4m3_code_widens_exactly(which, T):
    """Hand-made codes at scale 1 through moe_grouped_ffn_fp8, all tokens in expert 0.

    Token t is the unit vector e_t and the matrices not under test are all-ones or the identity
    (code 0x38 = 1.0), so every output is one decoded code through one SwiGLU:
      gate  y[t,j] = silu(dec(c[j,t]))            (W_up all ones, W_down the identity)
      up    y[t,j] = silu(1) * dec(c[j,t])        (W_gate all ones, W_down the identity)
      down  y[t,j] = bf16(silu(1)) * dec(c[j,t])  (W_gate all ones, W_up the identity)
    with c[j,t] = (j + t) mod 256 sweeping every code but the two NaNs over j for each token (T=256:
    two 128-row tiles; T=32 and T=8: one ragged tile). A wrongly widened code
    (subnormals, -0, the +-448 ends) shows as a relative error of that single output. Bound:
    one bf16 rounding of y (2^-9), the bf16 rounding of h = silu(1) in the down case (8.1e-4)
    and float32 silu; 2^-7 covers them.
    """
    n = 256
    cfg = moe.make_config(T=T, d_model=n, n_experts=2, top_k=1, d_ff=n, n_shared=0, score="softmax",
                          renormalize=True, capacity_factor=0.0, dtype="bf16")
    one, zero = 0x38, 0x00
    ramp = (np.arange(n)[:, None] + np.arange(n)[None, :]) % 256
    ramp = np.where((ramp & 0x7F) == 0x7F, zero, ramp).astype(np.uint8)
    eye = np.where(np.eye(n, dtype=bool), one, zero).astype(np.uint8)
    ones = np.full((n, n), one, np.uint8)
    wg, wu, wd = {"gate": (ramp, ones, eye), "up": (ones, ramp, eye), "down": (ones, eye, ramp)}[which]
    empty = np.zeros((n, n), np.uint8)

    def dev_codes(c):
        return torch.from_numpy(np.stack([c, empty])).cuda()

    scale = torch.ones(2, n, dtype=torch.float32, device="cuda")
    xp = torch.eye(n, dtype=torch.bfloat16, device="cuda")[:T].contiguous()
    offsets = torch.tensor([0, T, T], dtype=torch.int32, device="cuda")
    y = torch.full((moe.moe_grouped_rows(cfg), n), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = moe.alloc_workspace(cfg)
    moe.moe_grouped_ffn_fp8(cfg, xp, offsets, xp, dev_codes(wg), scale, dev_codes(wu), scale, dev_codes(wd),
                            scale, y, ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    got = to_f64(y)
    dec = lambda c: O.e4m3_decode(c).astype(np.float64)
    ref = O.expert_mlp(np.eye(n)[:T], dec(wg), dec(wu), dec(wd))
    assert np.isfinite(got).all()
    bad = np.abs(got - ref) > 2.0 ** -7 * np.abs(ref) + 1e-30
    assert not bad.any(), f"{which}: {int(bad.sum())} outputs off, first at {np.argwhere(bad)[0]}"
