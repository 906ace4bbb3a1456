"""Shared helpers of the GPU parity tests: inputs, the oracle side, and the comparison rules.

Comparison rules (GPU vs the fp64 oracle on the same seeded inputs):
  * expert ids: identical, except that a token may swap experts whose oracle
    scores differ by less than 1e-6 at the top-k boundary (or inside the
    ranking); the swapped selection must still be a valid top-k within 1e-6;
  * counts, offsets, dest_row, src_token, x_perm: bit-exact against the
    oracle's grouping of the GPU's ids;
  * layer / MLP outputs: max-abs error <= 1e-2 * max|ref| (bf16 layers, float32
    accumulation) or <= 1e-4 * max|ref| (float32 layers);
  * scores and gates: per token, see router_tolerance().
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import synth
import sparse_expert_mlp_router_b300 as moe

TIE = 1e-6


def cfg_of(w: synth.Workload) -> moe.MoeConfig:
    return moe.make_config(T=w.T, d_model=w.d_model, n_experts=w.n_experts, top_k=w.top_k, d_ff=w.d_ff,
                           n_shared=w.n_shared, score=w.score, renormalize=w.renormalize,
                           capacity_factor=w.capacity_factor, dtype=w.dtype)


def out_tolerance(w: synth.Workload) -> float:
    return 1e-2 if w.dtype == "bf16" else 1e-4


# Margin over the random-walk scale of float32 summation rounding (see router_tolerance).
ROUND_MARGIN = 8.0


def router_tolerance(x64: np.ndarray, wr64: np.ndarray, bias) -> np.ndarray:
    """Per-token absolute tolerance [T] of float32 scores and gates against the fp64 oracle.

    A logit is a float32 sum of the d products x_i * w_i (exact for bf16 inputs, each
    rounded once for float32 inputs), plus the bias. Each rounding of a partial sum errs by
    at most 2^-24 of it; the partial sums of d terms of random sign wander like a random
    walk, so the accumulated error has the scale 2^-24 * sqrt(d) * ||x (.) w||_2 (the 2-norm
    of the products, the random walk's step size times sqrt(d)), whatever order or grouping
    (tensor-core k-blocks, split reductions) the sum takes. The tolerance of a logit is
    ROUND_MARGIN times that scale for the token's largest such norm over the experts, plus
    two roundings of the biased logit. A softmax or sigmoid score, and a renormalised gate,
    moves by at most twice the largest logit error (d s_j = s_j (d l_j - sum_i s_i d l_i)
    for softmax; gates g_j = s_j / sum s are s_j times a common factor), and the score
    function's own float32 evaluation adds a few ulps of values at most 1: the 1e-6 floor.
    """
    x64 = np.asarray(x64, dtype=np.float64)
    wr64 = np.asarray(wr64, dtype=np.float64)
    d = x64.shape[1]
    p2 = np.sqrt((x64 * x64) @ (wr64 * wr64).T)               # [T, E] ||x_t (.) w_e||_2
    l = x64 @ wr64.T
    b = np.zeros(wr64.shape[0]) if bias is None else np.abs(np.asarray(bias, dtype=np.float64))
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float64)[None, :]
    dl = 2.0 ** -24 * (ROUND_MARGIN * math.sqrt(d) * p2.max(axis=1) + 2.0 * (np.abs(l) + b[None, :]).max(axis=1))
    return 1e-6 + 2.0 * dl


class Inputs:
    """Whole host-generated inputs of a (small) workload, as stored bits and as exact float64."""

    def __init__(self, w: synth.Workload):
        self.w = w
        self.raw = {n: synth.host_tensor(w, n) for n in ("x", "w_router", "w_gate", "w_up", "w_down")}
        self.f64 = {n: synth.as_f64(a, w.dtype) for n, a in self.raw.items()}
        self.bias = synth.router_bias(w.n_experts, w.bias_s)

    def expert(self, g):
        return self.f64["w_gate"][g], self.f64["w_up"][g], self.f64["w_down"][g]

    def device(self):
        t = {n: synth.host_to_torch(a, self.w.dtype).cuda() for n, a in self.raw.items()}
        t["bias"] = None if self.bias is None else torch.from_numpy(self.bias).cuda()
        return t


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_routing(gpu_idx: np.ndarray, ref_scores: np.ndarray, k: int) -> np.ndarray:
    """Assert the GPU's ids are the oracle's top-k up to near-ties; return the tokens that swapped."""
    T, E = ref_scores.shape
    ref_idx, _ = O.select_topk(ref_scores, k)
    assert gpu_idx.shape == (T, k)
    assert ((gpu_idx >= 0) & (gpu_idx < E)).all(), "expert id out of range"
    swapped = np.nonzero((gpu_idx != ref_idx).any(axis=1))[0]
    for t in swapped:
        row = gpu_idx[t]
        assert len(set(row.tolist())) == k, f"token {t}: repeated expert {row}"
        s = ref_scores[t]
        chosen = s[row]
        others = np.delete(s, row)
        # a valid top-k up to TIE: nothing left out beats anything chosen by more than TIE
        if others.size:
            assert others.max() <= chosen.min() + TIE, (t, row, ref_idx[t], chosen, others.max())
        # rank order up to TIE
        assert (chosen[:-1] >= chosen[1:] - TIE).all(), (t, row, chosen)
    return swapped


def oracle_gates_for(ids: np.ndarray, ref_scores: np.ndarray, renormalize: bool) -> np.ndarray:
    sel = np.take_along_axis(ref_scores, ids.astype(np.int64), axis=1)
    return O.gates_from_scores(sel, renormalize)


def assert_close(got: np.ndarray, ref: np.ndarray, rel_to_max: float, what: str) -> float:
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    assert err <= rel_to_max * max(scale, 1e-30), f"{what}: max-abs error {err:.3e} > {rel_to_max:g} x {scale:.3e}"
    return err / max(scale, 1e-30)
