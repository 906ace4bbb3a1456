"""moe_layer_forward enqueues no host synchronisation and allocates nothing, so a caller can
capture it into a CUDA graph: a replay must give bit-for-bit the output of an eager call,
also after the inputs change in place between replays."""
import pytest
import torch

import synth
import sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, cfg_of

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["mini_deepseek", "mini_qwen3", "mini_decode"])
def test_layer_replays_from_a_cuda_graph(name):
    w = synth.WORKLOADS[name]
    cfg = cfg_of(w)
    dev = Inputs(w).device()
    ws = moe.alloc_workspace(cfg)
    x = dev["x"].clone()
    args = lambda out: (cfg, x, dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"], dev["w_down"], out, ws)
    eager = torch.empty(w.T, w.d_model, dtype=x.dtype, device="cuda")
    moe.moe_layer_forward(*args(eager))          # eager call first (also warms every launch path)
    torch.cuda.synchronize()

    out = torch.zeros_like(eager)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_layer_forward(*args(out))
    g.replay()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))

    # new activations written in place: the replay routes and computes them afresh
    x.copy_(torch.flip(dev["x"], dims=[0]))
    g.replay()
    moe.moe_layer_forward(*args(eager))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))


def test_timed_layer_records_stage_events_inside_a_graph():
    # the stage events of moe_layer_forward_timed are real event nodes in a captured graph
    w = synth.WORKLOADS["mini_mixtral"]
    cfg = cfg_of(w)
    dev = Inputs(w).device()
    ws = moe.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d_model, dtype=torch.bfloat16, device="cuda")
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    args = (cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"], dev["w_down"], out, ws)
    moe.moe_layer_forward_timed(*args, evs)       # eager: creates the events
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        moe.moe_layer_forward_timed(*args, evs)
    g.replay()
    torch.cuda.synchronize()
    times = [evs[j].elapsed_time(evs[j + 1]) for j in range(5)]
    assert all(t >= 0.0 for t in times) and sum(times) > 0.0
