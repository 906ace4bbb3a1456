"""Plain fp64 CPU oracle of one Mixture-of-Experts FFN layer (forward pass).

TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline may use this module; the CUDA path never does. It is deliberately
slow and literal: every stage follows the definition on the source pages, in
float64, with numpy's matmul as the only library primitive and no blocking,
fusion or reordering beyond what the definition states.

Source pages (cited by the short names used below):
  [ST]  shubhamtatvamasi.com/llm-inference/moe, "Mixture of Experts"
  [KG]  klaylearn.com/glossary/mixture-of-experts, "Mixture of Experts" (glossary)
  [KL]  klaylearn.com/inference-engineering/l/mixture-of-experts, lesson 06.05
  [TB]  techbonafide.com, "Mixture of Experts (MoE) explained: why AI models
        don't use every parameter at once"
  [SA]  shipai.vats.cc/learn/advanced-concepts/mixture-of-experts, "Mixture of
        Experts (MoE)"

What the layer computes (the plainest reading of the pages):
  1. logits l[t,e] = x[t] . W_r[e] (+ b[e])          [ST "The router"; Q&A "How does a top-k router work?"]
  2. scores s = softmax over all E experts, or sigmoid per expert
                                                     [ST "The router"; SA "How routing works"]
  3. keep the k highest scores per token, ties to the lower expert index
                                                     [ST "The router"; TB "How Does Routing Work"]
  4. gates g_j = s_j / sum of the selected s (renormalised to sum to one)
                                                     [ST "The router" and its Q&A]
  5. group the (token, expert) pairs by destination expert; with a capacity
     factor cf each expert keeps at most ceil(cf * T * k / E) tokens and the
     overflow skips that expert (the token only goes on through the residual connection)
                                                     [KG definition; ST "Load imbalance"; ST Q&A on capacity factor]
  6. each kept pair runs its expert's MLP; the MLP form is not fixed by the
     pages (each expert is only called an ordinary feed-forward block, TB "Experts as
     Specialized Subnetworks"); this layer uses SwiGLU without biases:
        y = W_down (silu(W_gate x) * (W_up x)),  silu(z) = z / (1 + exp(-z))
  7. out[t] = sum over the token's kept slots j of g_j * y_j, plus every shared
     expert's MLP of x[t] with weight one           [ST "The router" (shared experts); KG definition]
The residual add is outside the layer: a token whose every routed pair was
dropped gets only its shared-expert part (zero when there is none).
With FP8 (E4M3) weights the expert MLP runs on the dequantized weights; with FP8
activations as well (W8A8, a mode beyond the pages) it is expert_mlp_w8a8.

Readings where the pages are silent (each the plainest one):
  * tie-break of equal scores: the lower expert index wins; slot order is the
    rank order (highest score first);
  * softmax is taken over all E logits before selection, then the selected
    scores are renormalised (for softmax this equals a softmax over the
    selected logits);
  * which tokens overflow a full expert: tokens are admitted in ascending
    token index, so the highest-index tokens are dropped;
  * the capacity factor is the binary32 number the caller passes; the
    ceiling is taken of its exact rational value times T*k/E;
  * dropped pairs are not compensated: the remaining gates are not
    renormalised again;
  * a router bias, when present, is added to the logits before the score
    function, so it moves both the selection and the gates.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from fractions import Fraction
from typing import Callable, Optional, Sequence

import numpy as np

__all__ = [
    "router_logits", "scores_from_logits", "select_topk", "gates_from_scores", "route",
    "capacity", "dispatch", "silu", "expert_mlp", "combine", "layer_forward", "LayerResult",
    "flops_per_token", "weight_bytes", "experts_touched_expected", "experts_touched",
    "routing_stats", "e4m3_decode", "e4m3_encode", "quantize_fp8_rows", "dequantize_fp8_rows",
    "bf16_round", "expert_mlp_w8a8",
]


# ---------------------------------------------------------------------------
# 1-4: routing

def router_logits(x: np.ndarray, w_router: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    """l = x W_r^T (+ b): one logit per expert from one small linear layer [ST "The router"]."""
    l = np.asarray(x, dtype=np.float64) @ np.asarray(w_router, dtype=np.float64).T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float64)[None, :]
    return l


def scores_from_logits(logits: np.ndarray, score: str) -> np.ndarray:
    """Softmax over all experts (max-subtracted), or the sigmoid variant [ST "The router"]."""
    l = np.asarray(logits, dtype=np.float64)
    if score == "softmax":
        z = np.exp(l - l.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    if score == "sigmoid":
        with np.errstate(over="ignore"):
            return 1.0 / (1.0 + np.exp(-l))
    raise ValueError(score)


def select_topk(scores: np.ndarray, k: int):
    """The k highest scores per token, in rank order; equal scores go to the lower index.

    A stable sort of -s keeps equal scores in ascending expert order.
    Returns (idx [T,k] int32, selected scores [T,k] float64).
    """
    s = np.asarray(scores, dtype=np.float64)
    order = np.argsort(-s, axis=1, kind="stable")[:, :k]
    return order.astype(np.int32), np.take_along_axis(s, order, axis=1)


def gates_from_scores(s_sel: np.ndarray, renormalize: bool = True) -> np.ndarray:
    """Selected gate values renormalised to sum to one [ST "The router"; Q&A top-k router]."""
    if not renormalize:
        return np.array(s_sel, dtype=np.float64)
    return s_sel / s_sel.sum(axis=1, keepdims=True)


def route(x, w_router, bias, k: int, score: str, renormalize: bool = True):
    """Stages 1-4. Returns (idx [T,k] int32, gate [T,k] f64, scores [T,E] f64)."""
    s = scores_from_logits(router_logits(x, w_router, bias), score)
    idx, s_sel = select_topk(s, k)
    return idx, gates_from_scores(s_sel, renormalize), s


# ---------------------------------------------------------------------------
# 5: capacity and the permutation by destination expert

def capacity(T: int, k: int, E: int, capacity_factor: float) -> Optional[int]:
    """Per-expert limit ceil(cf * T*k/E) on the exact value of binary32 cf; None = dropless.

    [ST "Load imbalance": at most capacity factor x ideal tokens; ST Q&A on
    capacity factor: "factor x (T.k/E)".]
    """
    cf = float(np.float32(capacity_factor))
    if cf <= 0.0:
        return None
    return math.ceil(Fraction(cf) * T * k / E)


@dataclass
class Dispatch:
    counts: np.ndarray     # [E]   pairs routed to each expert, before capacity
    kept: np.ndarray       # [E]   pairs each expert keeps
    offsets: np.ndarray    # [E+1] exclusive scan of kept; offsets[E] = kept pairs P'
    dest_row: np.ndarray   # [T,k] row of pair (t,j) in the grouped buffer, -1 if dropped
    src_token: np.ndarray  # [P']  token of each grouped row


def dispatch(idx: np.ndarray, n_experts: int, cap: Optional[int]) -> Dispatch:
    """Group the (token, slot) pairs by expert, admitting tokens in ascending index.

    "Permuting tokens by destination expert" [KG definition]; overflow beyond
    the capacity skips the expert [ST "Load imbalance"].
    """
    T, k = idx.shape
    per_expert: list[list[tuple[int, int]]] = [[] for _ in range(n_experts)]
    seen = np.zeros(n_experts, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if cap is None or seen[e] < cap:
                per_expert[e].append((t, j))
            seen[e] += 1
    counts = seen.astype(np.int32)
    kept = np.array([len(p) for p in per_expert], dtype=np.int32)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(kept)
    dest_row = np.full((T, k), -1, dtype=np.int32)
    src_token = np.zeros(int(offsets[-1]), dtype=np.int32)
    for e in range(n_experts):
        for r, (t, j) in enumerate(per_expert[e]):
            dest_row[t, j] = offsets[e] + r
            src_token[offsets[e] + r] = t
    return Dispatch(counts, kept, offsets, dest_row, src_token)


# ---------------------------------------------------------------------------
# 6: the expert MLP

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_mlp(xrows: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """SwiGLU MLP of each row: W_down (silu(W_gate x) * (W_up x)).

    xrows [n,d]; w_gate, w_up [F,d]; w_down [d,F]; returns [n,d] float64.
    """
    xr = np.asarray(xrows, dtype=np.float64)
    g = xr @ np.asarray(w_gate, dtype=np.float64).T
    u = xr @ np.asarray(w_up, dtype=np.float64).T
    return (silu(g) * u) @ np.asarray(w_down, dtype=np.float64).T


# ---------------------------------------------------------------------------
# 7: combine

def combine(dest_row: np.ndarray, gate: np.ndarray, y_rows: np.ndarray,
            shared: Optional[np.ndarray], d_model: int) -> np.ndarray:
    """out[t] = sum over kept slots of gate * expert output, plus the shared part.

    [ST Q&A "How does a top-k router work?": gate-weighted sum; ST "The router":
    shared experts, which all tokens pass through.] Dropped slots add nothing.
    """
    T, k = dest_row.shape
    out = np.zeros((T, d_model), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            r = int(dest_row[t, j])
            if r >= 0:
                out[t] += gate[t, j] * y_rows[r]
    if shared is not None:
        out += shared
    return out


# ---------------------------------------------------------------------------
# whole layer

@dataclass
class LayerResult:
    idx: np.ndarray
    gate: np.ndarray
    scores: np.ndarray
    disp: Dispatch
    cap: Optional[int]
    tokens: np.ndarray          # the token ids whose outputs are in `out`
    out: np.ndarray             # [len(tokens), d] float64


ExpertFn = Callable[[int], Sequence[np.ndarray]]


def layer_forward(x: np.ndarray, w_router: np.ndarray, bias: Optional[np.ndarray], experts: ExpertFn,
                  *, top_k: int, score: str = "softmax", renormalize: bool = True,
                  capacity_factor: float = 0.0, n_shared: int = 0,
                  tokens: Optional[np.ndarray] = None,
                  routing: Optional[tuple] = None,
                  mlp: Callable = None) -> LayerResult:
    """The MoE FFN layer for all tokens, or only the outputs of `tokens`.

    x [T,d] and w_router [E,d] are float64 (exact copies of the stored
    values). experts(g) returns expert g's (W_gate [F,d], W_up [F,d],
    W_down [d,F]) in float64; g = E .. E+S-1 are the shared experts. Routing
    and capacity always cover all T tokens (admission depends on the whole
    batch); only the MLP and combine are restricted to `tokens`.
    `routing` = (idx, gate) replaces stages 1-4 (scores then come back None).
    `mlp` replaces the expert MLP (expert_mlp_w8a8 for FP8 activations).
    """
    mlp = expert_mlp if mlp is None else mlp
    x = np.asarray(x, dtype=np.float64)
    T, d = x.shape
    E = w_router.shape[0]
    if routing is None:
        idx, gate, s = route(x, w_router, bias, top_k, score, renormalize)
    else:
        idx, gate = routing
        idx = np.asarray(idx, dtype=np.int32)
        gate = np.asarray(gate, dtype=np.float64)
        s = None
    cap = capacity(T, top_k, E, capacity_factor)
    disp = dispatch(idx, E, cap)
    tok = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    want = np.zeros(T, dtype=bool)
    want[tok] = True

    y_rows = np.zeros((int(disp.offsets[-1]), d), dtype=np.float64)
    for e in range(E):
        rows = np.arange(disp.offsets[e], disp.offsets[e + 1])
        rows = rows[want[disp.src_token[rows]]]
        if rows.size == 0:
            continue
        wg, wu, wd = experts(e)
        y_rows[rows] = mlp(x[disp.src_token[rows]], wg, wu, wd)

    shared = None
    if n_shared > 0:
        shared = np.zeros((T, d), dtype=np.float64)
        for s_i in range(n_shared):
            wg, wu, wd = experts(E + s_i)
            shared[tok] += mlp(x[tok], wg, wu, wd)
    out = combine(disp.dest_row, gate, y_rows, shared, d)[tok]
    return LayerResult(idx, gate, s, disp, cap, tok, out)


# ---------------------------------------------------------------------------
# accounting rules the pages state

def flops_per_token(active_params: float) -> float:
    """FLOPs per token = 2 x active parameters [ST "Memory vs compute, quantified", table]."""
    return 2.0 * active_params


def weight_bytes(total_params: float, bytes_per_param: float) -> float:
    """Resident weight memory = total parameters x bytes per parameter [ST same table]."""
    return total_params * bytes_per_param


def experts_touched_expected(E: int, k: int, batch: int) -> float:
    """Expected experts read per step under uniform routing: E (1 - (1 - k/E)^batch).

    [ST "Memory vs compute, quantified": the touched fraction is about
    1 - (1 - k/E)^batch.] Exact for tokens that each pick a uniformly random
    k-subset independently: each expert is missed by one token with
    probability 1 - k/E.
    """
    return E * (1.0 - (1.0 - k / E) ** batch)


def experts_touched(idx: np.ndarray, E: int) -> int:
    """Number of distinct experts a routing reads."""
    return int(np.unique(np.asarray(idx).ravel()).size) if np.asarray(idx).size else 0


def routing_stats(counts, T: int, cap: Optional[int]) -> dict:
    """Load report of one batch from the per-expert counts (pairs routed before capacity).

    [ST "Load imbalance": per-expert load, drops under a capacity limit, and, for dropless
    serving, the share of expert compute that is useful while all wait for the busiest
    expert -- read here as mean load / max load; ST "Memory vs compute, quantified":
    the experts a batch touches.] kept[e] = min(counts[e], cap); exact fractions for the
    mean load and the efficiency (1 when nothing is kept).
    """
    c = np.maximum(np.asarray(counts, dtype=np.int64), 0)
    cap_v = T if cap is None else int(cap)
    kept = np.minimum(c, cap_v)
    E = c.size
    K = int(kept.sum())
    M = int(kept.max()) if E else 0
    mean = Fraction(K, E)
    return {"tokens": int(T), "pairs": int(c.sum()), "kept": K, "dropped": int(c.sum()) - K,
            "experts_touched": int((kept > 0).sum()), "max_load": M, "capacity": cap_v,
            "mean_load": mean, "efficiency": (mean / M) if M > 0 else Fraction(1)}


# ---------------------------------------------------------------------------
# FP8 (E4M3) expert weights
#
# [ST "Memory vs compute, quantified": the 671B model's weights are about 671 GB in FP8.]
# The pages name the format only; the encoding is the OCP 8-bit floating point E4M3 format:
# 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 holds the
# subnormals m/8 * 2^-6; exponent 15 with mantissa 7 is NaN (no infinities); the largest
# finite magnitude is 1.75 * 2^8 = 448. A weight row is stored as codes with one float32
# scale: W[r][c] = scale[r] * value(code[r][c]).

def e4m3_decode(codes) -> np.ndarray:
    """Exact float64 values of E4M3 codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(v) -> np.ndarray:
    """E4M3 code of each value: round to the nearest representable magnitude, ties to the even
    mantissa code, magnitudes above 448 saturated to 448, the sign bit copied from the input
    (so a negative value that rounds to zero gives negative zero, 0x80), NaN to 0x7F."""
    x = np.asarray(v, dtype=np.float64)
    codes = np.arange(0x7F, dtype=np.int64)                  # all non-negative finite codes
    vals = e4m3_decode(codes)                                # increasing
    mag = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(vals, mag, side="left"), 1, len(vals) - 1)
    lo = hi - 1
    d_lo = mag - vals[lo]
    d_hi = vals[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    code = np.where(pick_hi, codes[hi], codes[lo])
    code = np.where(mag == vals[hi], codes[hi], code)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def quantize_fp8_rows(w) -> tuple:
    """Per-row E4M3 quantisation of float32-representable weights, in the arithmetic the codes
    are defined with: scale = float32(max|w_row|) / float32(448) and code = E4M3 of
    float32(w) / scale, both divisions rounded once to float32 (code 0 for an all-zero row).
    Returns (codes uint8 [.., cols], scale float32 [..])."""
    w32 = np.asarray(w, dtype=np.float32)
    mx = np.max(np.abs(w32), axis=-1)
    scale = (mx / np.float32(448.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    v = (w32 / safe[..., None]).astype(np.float32)
    v = np.where(scale[..., None] > 0, v, np.float32(0.0))
    return e4m3_encode(v), scale


def dequantize_fp8_rows(codes, scale) -> np.ndarray:
    """scale[r] * value(code[r][c]) in float64 (exact)."""
    return np.asarray(scale, dtype=np.float64)[..., None] * e4m3_decode(codes)


# ---------------------------------------------------------------------------
# FP8 activations as well (W8A8)
#
# A reading beyond what the pages fix. The pages put the weights in FP8 (the 671B model in
# ~671 GB) and say nothing of the activations; this mode also stores the activations that
# enter each expert contraction in E4M3, quantised per row exactly as the weights are (one
# float32 scale per row, scale = max|row| / 448, code = E4M3 of value / scale): the expert's
# input rows before the gate/up products, and the intermediate h = silu(g) * u -- which is
# stored in bf16 between the two contractions -- before the down product. Products and sums
# are then exact in the quantised values. It changes the layer's numbers by the activations'
# quantisation error (about 2^-4 of an element at most), so it is compared with this
# function, not with the bf16-activation layer.

def bf16_round(v) -> np.ndarray:
    """Values rounded to float32, then to bfloat16 with round-to-nearest-even (float64 out):
    how a float32 result is stored in bf16."""
    u = np.ascontiguousarray(np.asarray(v, dtype=np.float64).astype(np.float32)).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def expert_mlp_w8a8(xrows: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """The SwiGLU expert MLP with E4M3 activations: x rows quantised per row, gate and up
    products of the quantised rows, h = silu(g) * u stored in bf16 and quantised per row,
    down product of the quantised h. Same shapes as expert_mlp."""
    qx, sx = quantize_fp8_rows(np.asarray(xrows, dtype=np.float64))
    xq = dequantize_fp8_rows(qx, sx)
    g = xq @ np.asarray(w_gate, dtype=np.float64).T
    u = xq @ np.asarray(w_up, dtype=np.float64).T
    h = bf16_round(silu(g) * u)
    qh, sh = quantize_fp8_rows(h)
    return dequantize_fp8_rows(qh, sh) @ np.asarray(w_down, dtype=np.float64).T
