"""No call writes outside the buffers it is given.

Every caller-owned output (and the workspace) is placed inside a larger allocation whose
256 bytes before and after it hold a canary byte pattern; after each call the guard bytes must
be unchanged. The buffers are exactly the sizes include/moe.h states: topk_idx/topk_gate [T,k],
scores [T,E], counts [E], offsets [E+1], dest_row [T,k], src_token [R], x_perm [R,d],
y_perm [R + S*T, d], out [T,d], the workspace moe_workspace_size bytes.
"""
import pytest
import torch

import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, cfg_of

pytestmark = pytest.mark.gpu

GUARD = 256          # bytes on each side (keeps every view 256-byte aligned)
CANARY = 0xA5


class Guarded:
    def __init__(self, shape, dtype):
        esize = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD // esize
        n = 1
        for s in shape:
            n *= s
        self.n = n
        self.full = torch.empty(n + 2 * self.g, dtype=dtype, device="cuda")
        self.full.view(torch.uint8).fill_(CANARY)
        self.t = self.full[self.g:self.g + n].view(*shape)

    def intact(self) -> bool:
        raw = self.full.view(torch.uint8)
        lo, hi = raw[:GUARD], raw[GUARD + self.n * self.full.element_size():]
        return bool((lo == CANARY).all()) and bool((hi == CANARY).all()) and hi.numel() == GUARD


def _check_all(bufs, where):
    bad = [name for name, b in bufs.items() if not b.intact()]
    assert not bad, f"{where}: writes outside {bad}"


def _workspace(cfg):
    ws = Guarded((moe.moe_workspace_size(cfg),), torch.uint8)
    moe.moe_workspace_init(ws.t)
    return ws


LAYER_CASES = [
    ("mini_deepseek", {}),                        # capacity drops, shared expert, sigmoid
    ("mini_qwen3", dict(T=129)),                  # one row past a tile
    ("mini_decode", {}),                          # single-chunk grouping
    ("tiny_f32", {}),                             # float32 path
    ("tiny_f32", dict(T=70, n_shared=1, capacity_factor=1.0)),
]


@pytest.mark.parametrize("name,edit", LAYER_CASES, ids=lambda v: str(v))
def test_layer_writes_only_its_outputs(name, edit):
    w = synth.WORKLOADS[name].with_(**edit)
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    dt = dev["x"].dtype
    bufs = {"out": Guarded((w.T, w.d_model), dt), "topk_idx": Guarded((w.T, w.top_k), torch.int32),
            "counts": Guarded((w.n_experts,), torch.int32), "workspace": _workspace(cfg)}
    for _ in range(2):
        moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"],
                              dev["w_down"], bufs["out"].t, bufs["workspace"].t, topk_idx_out=bufs["topk_idx"].t,
                              counts_out=bufs["counts"].t)
        assert moe.moe_get_device_error(bufs["workspace"].t) == moe.MOE_OK
        _check_all(bufs, f"{name} {edit} layer")
    assert bool(torch.isfinite(bufs["out"].t.float()).all())


@pytest.mark.parametrize("name", ["mini_deepseek", "mini_mixtral", "tiny_f32"])
def test_stages_write_only_their_outputs(name):
    w = synth.WORKLOADS[name]
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    dt = dev["x"].dtype
    T, k, E, d = w.T, w.top_k, w.n_experts, w.d_model
    R = moe.moe_rows_capacity(cfg)
    G = moe.moe_grouped_rows(cfg)
    b = {"topk_idx": Guarded((T, k), torch.int32), "topk_gate": Guarded((T, k), torch.float32),
         "scores": Guarded((T, E), torch.float32), "counts": Guarded((E,), torch.int32),
         "offsets": Guarded((E + 1,), torch.int32), "dest_row": Guarded((T, k), torch.int32),
         "src_token": Guarded((R,), torch.int32), "x_perm": Guarded((R, d), dt), "y_perm": Guarded((G, d), dt),
         "out": Guarded((T, d), dt), "workspace": _workspace(cfg)}
    ws = b["workspace"].t
    moe.moe_router_topk(cfg, dev["x"], dev["w_router"], dev["bias"], b["topk_idx"].t, b["topk_gate"].t,
                        b["scores"].t)
    torch.cuda.synchronize()
    _check_all(b, f"{name} router")
    moe.moe_permute(cfg, b["topk_idx"].t, dev["x"], b["counts"].t, b["offsets"].t, b["dest_row"].t,
                    b["src_token"].t, b["x_perm"].t, ws)
    torch.cuda.synchronize()
    _check_all(b, f"{name} permute")
    moe.moe_grouped_ffn(cfg, b["x_perm"].t, b["offsets"].t, dev["x"], dev["w_gate"], dev["w_up"], dev["w_down"],
                        b["y_perm"].t, ws)
    torch.cuda.synchronize()
    _check_all(b, f"{name} grouped ffn")
    moe.moe_combine(cfg, b["y_perm"].t, b["dest_row"].t, b["topk_gate"].t, b["out"].t, ws)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    _check_all(b, f"{name} combine")


def test_fp8_layer_and_quantiser_write_only_their_outputs():
    w = synth.WORKLOADS["mini_qwen3"].with_(T=200)
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    q = {}
    bufs = {}
    for n in ("w_gate", "w_up", "w_down"):
        rows, cols = dev[n].shape[0] * dev[n].shape[1], dev[n].shape[2]
        codes, scale = Guarded(tuple(dev[n].shape), torch.uint8), Guarded((rows,), torch.float32)
        moe.moe_quantize_fp8_rows(dev[n], codes.t, scale.t)
        q[n] = (codes.t, scale.t)
        bufs[n + "_codes"], bufs[n + "_scale"] = codes, scale
    bufs["out"] = Guarded((w.T, w.d_model), torch.bfloat16)
    bufs["workspace"] = _workspace(cfg)
    torch.cuda.synchronize()
    _check_all(bufs, "quantiser")
    moe.moe_layer_forward_fp8(cfg, dev["x"], dev["w_router"], dev["bias"], *q["w_gate"], *q["w_up"], *q["w_down"],
                              bufs["out"].t, bufs["workspace"].t)
    assert moe.moe_get_device_error(bufs["workspace"].t) == moe.MOE_OK
    _check_all(bufs, "fp8 layer")


@pytest.mark.parametrize("name,edit", [("mini_qwen3", {"T": 200}), ("mini_deepseek", {"capacity_factor": 0.05}),
                                       ("mini_decode", {})])
def test_w8a8_layer_writes_only_its_outputs(name, edit):
    # the W8A8 layer keeps its codes and scales inside the workspace (per-token codes in the
    # x_perm region, grouped codes in the y region), also when capacity makes R smaller than T
    w = synth.WORKLOADS[name].with_(**edit)
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    q = {n: moe.moe_quantize_fp8_rows(dev[n]) for n in ("w_gate", "w_up", "w_down")}
    bufs = {"out": Guarded((w.T, w.d_model), torch.bfloat16), "workspace": _workspace(cfg)}
    moe.moe_layer_forward_w8a8(cfg, dev["x"], dev["w_router"], dev["bias"], *q["w_gate"], *q["w_up"], *q["w_down"],
                               bufs["out"].t, bufs["workspace"].t)
    assert moe.moe_get_device_error(bufs["workspace"].t) == moe.MOE_OK
    _check_all(bufs, f"w8a8 layer {name}")


@pytest.mark.parametrize("combine", ["0", "1"])
@pytest.mark.parametrize("name,edit", [("mini_deepseek", {}), ("mini_decode", {}), ("mini_mixtral", {"T": 1200}),
                                       ("mini_qwen3", {"T": 100, "capacity_factor": 0.05})])
def test_fused_mlp_layer_writes_only_its_outputs(name, edit, combine, monkeypatch):
    # the one-launch expert MLP keeps its per-m-tile (and, combining, per-token) counters inside
    # the workspace; combining, it writes the output rows itself
    monkeypatch.setenv("MOE_FUSED_MLP", "1")
    monkeypatch.setenv("MOE_MLP_COMBINE", combine)
    w = synth.WORKLOADS[name].with_(**edit)
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    bufs = {"out": Guarded((w.T, w.d_model), torch.bfloat16), "workspace": _workspace(cfg)}
    moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"], dev["w_down"],
                          bufs["out"].t, bufs["workspace"].t)
    assert moe.moe_get_device_error(bufs["workspace"].t) == moe.MOE_OK
    _check_all(bufs, f"fused mlp layer {name}")


@pytest.mark.parametrize("name,edit", [("mini_decode", {}), ("mini_deepseek", {})])
def test_w8a8_one_launch_layer_writes_only_its_outputs(name, edit, monkeypatch):
    monkeypatch.setenv("MOE_FUSED_MLP", "1")
    w = synth.WORKLOADS[name].with_(**edit)
    dev = Inputs(w).device()
    cfg = cfg_of(w)
    q = {n: moe.moe_quantize_fp8_rows(dev[n]) for n in ("w_gate", "w_up", "w_down")}
    bufs = {"out": Guarded((w.T, w.d_model), torch.bfloat16), "workspace": _workspace(cfg)}
    moe.moe_layer_forward_w8a8(cfg, dev["x"], dev["w_router"], dev["bias"], *q["w_gate"], *q["w_up"], *q["w_down"],
                               bufs["out"].t, bufs["workspace"].t)
    assert moe.moe_get_device_error(bufs["workspace"].t) == moe.MOE_OK
    _check_all(bufs, f"w8a8 one-launch layer {name}")
