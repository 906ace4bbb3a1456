"""The per-token router tolerance of the GPU parity tests, checked on the CPU.

The tolerance has to hold for any honest float32 evaluation of the router (so it is not
too tight) and has to be small enough that a slip the output comparison would miss is
caught (so it is not too loose). Both are checked here against float32 evaluations of
the same routers: numpy's blocked float32 matmul, and strictly sequential float32
accumulation, the order with the largest rounding drift.
"""
import numpy as np
import pytest

import oracle as O
import synth
from moe_cases import router_tolerance


def _inputs(w, T_max=None):
    x = synth.host_tensor(w, "x")
    wr = synth.host_tensor(w, "w_router")
    if T_max is not None:
        x = x[:T_max]
    return synth.as_f64(x, w.dtype), synth.as_f64(wr, w.dtype), synth.router_bias(w.n_experts, w.bias_s)


def _f32_router(x64, wr64, bias, score, sequential):
    x32, w32 = x64.astype(np.float32), wr64.astype(np.float32)
    if sequential:
        # left-to-right float32 accumulation of the d products
        prod = x32[:, None, :] * w32[None, :, :]               # [T, E, d], each product rounded once
        l = np.zeros(prod.shape[:2], dtype=np.float32)
        for i in range(prod.shape[2]):
            l = (l + prod[:, :, i]).astype(np.float32)
    else:
        l = x32 @ w32.T
    if bias is not None:
        l = (l + bias.astype(np.float32)[None, :]).astype(np.float32)
    if score == "softmax":
        z = np.exp(l - l.max(axis=1, keepdims=True))
        return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return (1.0 / (1.0 + np.exp(-l))).astype(np.float32)


@pytest.mark.parametrize("name", synth.workloads.MINI + ["qwen3_30b_a3b", "deepseek_v3", "decode_qwen3"])
@pytest.mark.parametrize("sequential", [False, True])
def test_float32_routers_stay_within_the_tolerance(name, sequential):
    w = synth.WORKLOADS[name]
    x64, wr64, bias = _inputs(w, T_max=16 if sequential else 512)
    tol = router_tolerance(x64, wr64, bias)[:, None]
    ref = O.scores_from_logits(O.router_logits(x64, wr64, bias), w.score)
    got = _f32_router(x64, wr64, bias, w.score, sequential).astype(np.float64)
    assert (np.abs(got - ref) <= tol).all(), float((np.abs(got - ref) / tol).max())
    idx, _ = O.select_topk(ref, w.top_k)
    g_ref = O.gates_from_scores(np.take_along_axis(ref, idx.astype(np.int64), axis=1), w.renormalize)
    g_got = O.gates_from_scores(np.take_along_axis(got, idx.astype(np.int64), axis=1), w.renormalize)
    assert (np.abs(g_got - g_ref) <= tol).all()


@pytest.mark.parametrize("name", synth.workloads.MINI)
def test_a_gate_slip_of_2e_5_is_caught(name):
    # reduced layers (the ones compared element by element, d_model <= 512): every token's
    # tolerance is below 2e-5, so a gate that is off by 2e-5 (a dropped small bias, a
    # renormalisation over the wrong set) fails the comparison
    w = synth.WORKLOADS[name]
    x64, wr64, bias = _inputs(w)
    assert router_tolerance(x64, wr64, bias).max() < 2e-5


def test_tiny_layer_tolerance_is_the_floor():
    # the float32 tiny layer's logits are about 1e-3: its tolerance is the 1e-6 floor
    w = synth.WORKLOADS["tiny_f32"]
    tol = router_tolerance(*_inputs(w))
    assert tol.max() < 1.05e-6
