"""The 2-SM (CTA pair) grouped-GEMM kernels, selected with MOE_GEMM_PAIRS=1, against the fp64
oracle. The selection is read once per process, so the layers run in a child process."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle as O
import synth
from moe_cases import Inputs, out_tolerance

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, sys, numpy as np, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import synth, sparse_expert_mlp_router_b300 as moe
from moe_cases import Inputs, cfg_of
res = {}
for name, edit in json.loads(sys.argv[2]):
    w = synth.WORKLOADS[name].with_(**edit)
    dev = Inputs(w).device(); cfg = cfg_of(w); ws = moe.alloc_workspace(cfg)
    out = torch.empty(w.T, w.d_model, dtype=dev["x"].dtype, device="cuda")
    idx = torch.empty(w.T, w.top_k, dtype=torch.int32, device="cuda")
    moe.moe_layer_forward(cfg, dev["x"], dev["w_router"], dev["bias"], dev["w_gate"], dev["w_up"], dev["w_down"],
                          out, ws, topk_idx_out=idx)
    status = moe.moe_get_device_error(ws)
    res[name + json.dumps(edit)] = dict(status=status, out=out.float().cpu().numpy().tolist(),
                                        idx=idx.cpu().numpy().tolist())
print(json.dumps(res))
"""

CASES = [("mini_qwen3", {}), ("mini_deepseek", {}), ("mini_qwen3", {"T": 700, "bias_s": 1.5}),
         ("mini_mixtral", {"d_model": 512, "d_ff": 512, "T": 600})]


def test_pair_kernels_match_oracle():
    env = dict(os.environ, MOE_GEMM_PAIRS="1")
    p = subprocess.run([sys.executable, "-c", CHILD, ROOT, json.dumps(CASES)], env=env, capture_output=True,
                       text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    res = json.loads(p.stdout.strip().splitlines()[-1])
    for name, edit in CASES:
        r = res[name + json.dumps(edit)]
        assert r["status"] == 0
        w = synth.WORKLOADS[name].with_(**edit)
        inp = Inputs(w)
        gidx = np.array(r["idx"], dtype=np.int32)
        x64, wr64 = inp.f64["x"], inp.f64["w_router"]
        scores = O.scores_from_logits(O.router_logits(x64, wr64, inp.bias), w.score)
        gates = O.gates_from_scores(np.take_along_axis(scores, gidx.astype(np.int64), axis=1), w.renormalize)
        ref = O.layer_forward(x64, wr64, inp.bias, inp.expert, top_k=w.top_k, score=w.score,
                              renormalize=w.renormalize, capacity_factor=w.capacity_factor, n_shared=w.n_shared,
                              routing=(gidx, gates)).out
        got = np.array(r["out"], dtype=np.float64)
        err = np.abs(got - ref).max() / np.abs(ref).max()
        assert err <= out_tolerance(w), (name, edit, err)
