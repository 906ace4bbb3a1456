"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than its own formulas:
hand-worked cases with closed-form answers, brute-force enumeration on tiny
inputs, structural invariants (gates sum to one, counts sum to T*k minus
drops, k = E with uniform gates gives the mean of the experts, E = 1 gives a
dense MLP), and the figures the pages print (tests/golden/). A plausible slip
in the oracle (a wrong sign, a dropped term, a transposed operand, floor for
ceil, an unstable permutation) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as O
import synth
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _sig(z):
    return 1.0 / (1.0 + math.exp(-z))


# ---------------------------------------------------------------- routing ---

def test_hand_softmax_top2():
    # logits (3, 1, 2, 0), k = 2 -> experts (0, 2); gates e^3/(e^3+e^2), e^2/(e^3+e^2)
    x = np.array([[1.0]])
    w = np.array([[3.0], [1.0], [2.0], [0.0]])
    idx, gate, s = O.route(x, w, None, 2, "softmax")
    assert idx.tolist() == [[0, 2]]
    assert gate[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), abs=1e-15)
    assert gate[0, 1] == pytest.approx(1.0 / (1.0 + math.e), abs=1e-15)
    z = sum(math.exp(v) for v in (3, 1, 2, 0))
    assert s[0].tolist() == pytest.approx([math.exp(v) / z for v in (3, 1, 2, 0)], abs=1e-15)


def test_hand_sigmoid_top2_with_bias():
    # logits x.W = (0, 2, -1, 1); bias (0, 0, 3, 0) -> (0, 2, 2, 1): tie between 1 and 2 goes to 1
    x = np.array([[1.0]])
    w = np.array([[0.0], [2.0], [-1.0], [1.0]])
    b = np.array([0.0, 0.0, 3.0, 0.0])
    idx, gate, _ = O.route(x, w, b, 2, "sigmoid")
    assert idx.tolist() == [[1, 2]]
    assert gate[0].tolist() == pytest.approx([0.5, 0.5], abs=1e-15)
    idx, gate, _ = O.route(x, w, None, 3, "sigmoid")
    assert idx.tolist() == [[1, 3, 0]]
    tot = _sig(2) + _sig(1) + _sig(0)
    assert gate[0].tolist() == pytest.approx([_sig(2) / tot, _sig(1) / tot, 0.5 / tot], abs=1e-15)


def test_no_renormalize_keeps_raw_scores():
    x = np.array([[1.0]])
    w = np.array([[0.0], [2.0], [-1.0], [1.0]])
    _, gate, _ = O.route(x, w, None, 2, "sigmoid", renormalize=False)
    assert gate[0].tolist() == pytest.approx([_sig(2), _sig(1)], abs=1e-15)


def test_softmax_survives_large_logits():
    x = np.array([[1.0]])
    w = np.array([[800.0], [799.0], [0.0]])
    idx, gate, s = O.route(x, w, None, 2, "softmax")
    assert np.isfinite(s).all()
    assert idx.tolist() == [[0, 1]]
    assert gate[0, 0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), abs=1e-15)


def test_ties_go_to_lower_index():
    s = np.array([[0.2, 0.3, 0.3, 0.1, 0.3]])
    idx, sel = O.select_topk(s, 3)
    assert idx.tolist() == [[1, 2, 4]]
    idx, _ = O.select_topk(s, 2)
    assert idx.tolist() == [[1, 2]]


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
@pytest.mark.parametrize("k", [1, 2, 3])
def test_bruteforce_routing(score, k):
    rng = _rng(k)
    T, d, E = 16, 5, 6
    x = rng.standard_normal((T, d))
    w = rng.standard_normal((E, d))
    b = rng.standard_normal(E) * 0.5
    idx, gate, s = O.route(x, w, b, k, score)
    for t in range(T):
        # scores recomputed independently with scalar math
        logit = [sum(x[t, i] * w[e, i] for i in range(d)) + b[e] for e in range(E)]
        if score == "softmax":
            m = max(logit)
            z = [math.exp(v - m) for v in logit]
            ref = [v / sum(z) for v in z]
        else:
            ref = [_sig(v) for v in logit]
        assert s[t].tolist() == pytest.approx(ref, rel=1e-12, abs=1e-15)
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(ref[e] for e in c))
        assert sorted(idx[t].tolist()) == sorted(best)
        assert len(set(idx[t].tolist())) == k
        # slot order is rank order
        assert all(ref[idx[t, j]] >= ref[idx[t, j + 1]] for j in range(k - 1))
        assert sum(gate[t]) == pytest.approx(1.0, abs=1e-12)
        assert all(0.0 < g <= 1.0 for g in gate[t])
        if score == "softmax":
            # renormalised softmax == softmax over the selected logits
            sel = [logit[e] for e in idx[t]]
            zs = [math.exp(v - max(sel)) for v in sel]
            assert gate[t].tolist() == pytest.approx([v / sum(zs) for v in zs], rel=1e-12)


# --------------------------------------------------- capacity / dispatch ---

def test_capacity_formula():
    assert O.capacity(4096, 8, 256, 1.25) == 160          # the DeepSeek-V3-shaped workload
    assert O.capacity(10, 1, 4, 1.0) == 3                 # ceil(2.5), not floor
    assert O.capacity(8, 2, 4, 1.0) == 4                  # exact integer stays
    assert O.capacity(6, 1, 2, 0.5) == 2
    assert O.capacity(100, 2, 8, 0.0) is None             # dropless
    assert O.capacity(100, 2, 8, -1.0) is None
    # binary32 0.8 is slightly above 4/5, so ceil(0.8f * 5 / 2) = 3, not 2
    assert O.capacity(5, 1, 2, 0.8) == 3


def test_dispatch_hand_drop_highest_index():
    # 6 tokens, 2 experts, k = 1, cap = 2: tokens 0,1,2 -> expert 0; 3,4,5 -> expert 1
    idx = np.array([[0], [0], [0], [1], [1], [1]], dtype=np.int32)
    cap = O.capacity(6, 1, 2, 0.5)
    dsp = O.dispatch(idx, 2, cap)
    assert dsp.counts.tolist() == [3, 3]
    assert dsp.kept.tolist() == [2, 2]
    assert dsp.offsets.tolist() == [0, 2, 4]
    assert dsp.dest_row[:, 0].tolist() == [0, 1, -1, 2, 3, -1]
    assert dsp.src_token.tolist() == [0, 1, 3, 4]


def test_dispatch_one_over_capacity():
    # one expert gets cap + 1 tokens: exactly its highest-index token is dropped
    T, k, E = 12, 2, 4
    idx = np.array([[t % 2, 2 + (t % 2)] for t in range(T)], dtype=np.int32)
    idx[7] = [0, 2]          # expert 0 now has tokens 0,2,4,6,7,8,10 = 7 = cap + 1
    cap = O.capacity(T, k, E, 1.0)
    assert cap == 6
    dsp = O.dispatch(idx, E, cap)
    assert dsp.counts[0] == 7 and dsp.kept[0] == 6
    assert dsp.dest_row[10, 0] == -1
    assert (np.delete(dsp.dest_row[:, 0], 10) >= 0).all()


@pytest.mark.parametrize("cf", [0.0, 0.5, 1.0, 1.25, 100.0])
def test_dispatch_invariants(cf):
    rng = _rng(3)
    T, k, E = 97, 3, 7
    w = rng.random(E) ** 3                 # skewed expert preference
    idx = np.array([rng.choice(E, size=k, replace=False, p=w / w.sum()) for _ in range(T)], dtype=np.int32)
    cap = O.capacity(T, k, E, cf)
    dsp = O.dispatch(idx, E, cap)
    assert dsp.counts.sum() == T * k
    assert dsp.counts.tolist() == [int((idx == e).sum()) for e in range(E)]
    drops = int((dsp.dest_row < 0).sum())
    assert dsp.kept.sum() == T * k - drops == dsp.offsets[-1]
    assert (np.diff(dsp.offsets) >= 0).all() and dsp.offsets[0] == 0
    if cap is not None:
        assert (dsp.kept == np.minimum(dsp.counts, cap)).all()
    else:
        assert drops == 0
    for t in range(T):
        for j in range(k):
            r = dsp.dest_row[t, j]
            if r >= 0:
                assert dsp.src_token[r] == t
                e = idx[t, j]
                assert dsp.offsets[e] <= r < dsp.offsets[e + 1]
    for e in range(E):    # rows of an expert in ascending token order; its kept tokens are the lowest
        toks = dsp.src_token[dsp.offsets[e]:dsp.offsets[e + 1]].tolist()
        assert toks == sorted(toks)
        allt = [t for t in range(T) if e in idx[t]]
        assert toks == allt[:len(toks)]
    if cf == 100.0:        # cap >= T: identical to dropless
        ref = O.dispatch(idx, E, None)
        assert (ref.dest_row == dsp.dest_row).all()


# ----------------------------------------------------------- expert MLP ---

def test_silu_values():
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert O.silu(np.array([1.0]))[0] == pytest.approx(1.0 / (1.0 + math.exp(-1.0)), abs=1e-16)
    assert O.silu(np.array([math.log(3.0)]))[0] == pytest.approx(0.75 * math.log(3.0), abs=1e-15)
    assert O.silu(np.array([50.0]))[0] == pytest.approx(50.0, rel=1e-15)
    assert O.silu(np.array([-800.0]))[0] == 0.0


def test_mlp_closed_form_scalar():
    # d = F = 1: y = w_d * silu(w_g x) * (w_u x); sigmoid(ln 3) = 3/4
    y = O.expert_mlp(np.array([[1.0]]), np.array([[math.log(3.0)]]), np.array([[2.0]]), np.array([[4.0]]))
    assert y[0, 0] == pytest.approx(6.0 * math.log(3.0), abs=1e-14)
    # gate and up are not interchangeable
    y2 = O.expert_mlp(np.array([[1.0]]), np.array([[2.0]]), np.array([[math.log(3.0)]]), np.array([[4.0]]))
    assert abs(y2[0, 0] - y[0, 0]) > 0.1


def _textbook_mlp(xv, wg, wu, wd):
    """Scalar-loop SwiGLU: out_c = sum_f wd[c,f] * silu(sum_i wg[f,i] x_i) * (sum_i wu[f,i] x_i)."""
    F, d = wg.shape
    h = []
    for f in range(F):
        g = sum(wg[f, i] * xv[i] for i in range(d))
        u = sum(wu[f, i] * xv[i] for i in range(d))
        h.append(g * _sig(g) * u)
    return np.array([sum(wd[c, f] * h[f] for f in range(F)) for c in range(d)])


def _experts(rng, G, F, d, scale=0.5):
    ws = [(rng.standard_normal((F, d)) * scale, rng.standard_normal((F, d)) * scale,
           rng.standard_normal((d, F)) * scale) for _ in range(G)]
    return ws, (lambda g: ws[g])


def test_single_expert_is_dense_mlp():
    rng = _rng(5)
    T, d, F = 4, 5, 7
    x = rng.standard_normal((T, d))
    ws, fn = _experts(rng, 1, F, d)
    res = O.layer_forward(x, rng.standard_normal((1, d)), None, fn, top_k=1)
    assert (res.gate == 1.0).all()
    for t in range(T):
        assert res.out[t] == pytest.approx(_textbook_mlp(x[t], *ws[0]), rel=1e-12, abs=1e-14)


@pytest.mark.parametrize("score", ["softmax", "sigmoid"])
def test_k_equals_E_uniform_gates_gives_mean(score):
    rng = _rng(6)
    T, d, F, E = 3, 4, 6, 5
    x = rng.standard_normal((T, d))
    ws, fn = _experts(rng, E, F, d)
    res = O.layer_forward(x, np.zeros((E, d)), None, fn, top_k=E, score=score)
    assert res.gate == pytest.approx(np.full((T, E), 1.0 / E), abs=1e-15)
    for t in range(T):
        mean = sum(_textbook_mlp(x[t], *ws[e]) for e in range(E)) / E
        assert res.out[t] == pytest.approx(mean, rel=1e-12, abs=1e-14)


def test_shared_expert_added_with_weight_one():
    rng = _rng(7)
    T, d, F, E = 3, 4, 6, 3
    x = rng.standard_normal((T, d))
    ws, fn = _experts(rng, E + 1, F, d)
    wr = rng.standard_normal((E, d))
    with_s = O.layer_forward(x, wr, None, fn, top_k=2, n_shared=1)
    without = O.layer_forward(x, wr, None, fn, top_k=2, n_shared=0)
    for t in range(T):
        assert with_s.out[t] - without.out[t] == pytest.approx(_textbook_mlp(x[t], *ws[E]), rel=1e-12, abs=1e-14)


def test_combine_hand():
    dest = np.array([[1, -1], [0, 2]], dtype=np.int32)
    gate = np.array([[0.25, 0.75], [0.5, 0.5]])
    y = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]])
    out = O.combine(dest, gate, y, None, 2)
    assert out.tolist() == [[2.5, 5.0], [50.5, 101.0]]
    out = O.combine(dest, gate, y, np.ones((2, 2)), 2)
    assert out.tolist() == [[3.5, 6.0], [51.5, 102.0]]


def test_fully_dropped_token_gets_shared_part_only():
    rng = _rng(8)
    T, d, F, E, k = 6, 4, 5, 2, 1
    x = rng.standard_normal((T, d))
    ws, fn = _experts(rng, E + 1, F, d)
    wr = np.zeros((E, d))
    b = np.array([1.0, 0.0])               # every token prefers expert 0
    res = O.layer_forward(x, wr, b, fn, top_k=k, capacity_factor=0.5, n_shared=1)
    assert res.cap == 2
    dropped = [t for t in range(T) if (res.disp.dest_row[t] < 0).all()]
    assert dropped == [2, 3, 4, 5]
    for t in range(T):
        shared = _textbook_mlp(x[t], *ws[E])
        routed = 0 if t in dropped else _textbook_mlp(x[t], *ws[0])
        assert res.out[t] == pytest.approx(routed + shared, rel=1e-12, abs=1e-14)
    res0 = O.layer_forward(x, wr, b, fn, top_k=k, capacity_factor=0.5, n_shared=0)
    assert (res0.out[dropped] == 0.0).all()


def test_permuting_tokens_permutes_outputs_when_dropless():
    rng = _rng(9)
    T, d, F, E = 11, 6, 5, 4
    x = rng.standard_normal((T, d))
    ws, fn = _experts(rng, E, F, d)
    wr = rng.standard_normal((E, d))
    perm = rng.permutation(T)
    a = O.layer_forward(x, wr, None, fn, top_k=2)
    b = O.layer_forward(x[perm], wr, None, fn, top_k=2)
    assert b.out == pytest.approx(a.out[perm], rel=1e-12, abs=1e-14)


def test_routed_part_is_linear_in_down_projection():
    rng = _rng(10)
    T, d, F, E = 5, 4, 6, 3
    x = rng.standard_normal((T, d))
    ws, fn = _experts(rng, E + 1, F, d)
    wr = rng.standard_normal((E, d))
    c = 3.0
    scaled = [(g, u, dn * c) if i < E else (g, u, dn) for i, (g, u, dn) in enumerate(ws)]
    a = O.layer_forward(x, wr, None, fn, top_k=2, n_shared=1)
    b = O.layer_forward(x, wr, None, lambda g: scaled[g], top_k=2, n_shared=1)
    shared = np.array([_textbook_mlp(x[t], *ws[E]) for t in range(T)])
    assert b.out - shared == pytest.approx(c * (a.out - shared), rel=1e-11, abs=1e-13)


def test_token_subset_matches_full_layer():
    rng = _rng(11)
    T, d, F, E = 20, 6, 5, 5
    x = rng.standard_normal((T, d))
    ws, fn = _experts(rng, E + 1, F, d)
    wr = rng.standard_normal((E, d))
    full = O.layer_forward(x, wr, None, fn, top_k=2, capacity_factor=1.0, n_shared=1)
    sub = O.layer_forward(x, wr, None, fn, top_k=2, capacity_factor=1.0, n_shared=1, tokens=np.array([3, 17, 0]))
    assert sub.out == pytest.approx(full.out[[3, 17, 0]], rel=1e-14, abs=1e-15)


# ------------------------------------------------------------ accounting ---

def test_experts_touched_formula_matches_random_routing():
    rng = _rng(12)
    E, k, batch, trials = 128, 8, 32, 400
    touched = [O.experts_touched(np.array([rng.choice(E, size=k, replace=False) for _ in range(batch)]), E)
               for _ in range(trials)]
    expect = O.experts_touched_expected(E, k, batch)
    assert expect == pytest.approx(111.771, abs=0.001)   # 128 (1 - (15/16)^32)
    sd = np.std(touched) / math.sqrt(trials)
    assert abs(np.mean(touched) - expect) < 5 * sd + 0.05
    assert O.experts_touched_expected(E, k, 1) == pytest.approx(k)     # batch 1 reads k experts
    assert O.experts_touched_expected(E, k, 10_000) == pytest.approx(E)


def test_memory_and_flops_table_from_page():
    rows = []
    with open(os.path.join(GOLDEN, "memory_compute_table.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([v.strip() for v in line.split(",")])
    assert len(rows) == 4
    for name, total, active, bpp, gb, gflop, tol in rows:
        assert O.weight_bytes(float(total), float(bpp)) / 1e9 == pytest.approx(float(gb), rel=float(tol)), name
        assert O.flops_per_token(float(active)) / 1e9 == pytest.approx(float(gflop), rel=float(tol)), name


# ------------------------------------------------------------- telemetry ---

def test_routing_stats_hand_case():
    # counts (5, 0, 3, 2) with capacity 3: kept (3, 0, 3, 2) -> 8 kept, 2 dropped, 3 experts
    # touched, busiest 3, mean 2, useful share 2/3
    st = O.routing_stats([5, 0, 3, 2], T=5, cap=3)
    assert (st["pairs"], st["kept"], st["dropped"], st["experts_touched"], st["max_load"]) == (10, 8, 2, 3, 3)
    assert st["mean_load"] == 2 and st["efficiency"] == pytest.approx(2 / 3, abs=0)


def test_routing_stats_balanced_and_empty():
    assert O.routing_stats([4, 4, 4, 4], T=8, cap=None)["efficiency"] == 1
    empty = O.routing_stats([0, 0, 0], T=1, cap=2)
    assert empty["kept"] == 0 and empty["efficiency"] == 1 and empty["experts_touched"] == 0


def test_routing_stats_agree_with_dispatch():
    rng = _rng(7)
    T, E, k = 200, 16, 4
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    cap = O.capacity(T, k, E, 1.0)
    d = O.dispatch(idx, E, cap)
    st = O.routing_stats(d.counts, T=T, cap=cap)
    assert st["pairs"] == T * k and st["kept"] == int(d.offsets[-1]) == int(d.kept.sum())
    assert st["dropped"] == int((d.dest_row < 0).sum())
    assert st["experts_touched"] == O.experts_touched(idx[d.dest_row >= 0], E)
    assert st["max_load"] <= cap


# ------------------------------------------------------------ FP8 weights ---

def test_e4m3_codes_from_the_format():
    vals = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF]) and np.isfinite(np.delete(vals, [0x7F, 0xFF])).all()
    assert vals[0x7E] == 448.0 and vals[0x01] == 2.0 ** -9 and vals[0x08] == 2.0 ** -6 and vals[0x38] == 1.0
    assert vals[0x80] == 0.0 and np.signbit(vals[0x80]) and vals[0xC0] == -2.0
    finite = [c for c in range(256) if c not in (0x7F, 0xFF)]
    assert (O.e4m3_encode(vals[finite]) == np.array(finite, dtype=np.uint8)).all()      # round trip


def test_e4m3_rounding_ties_and_saturation():
    vals = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2                     # exact midpoints between neighbours
    got = O.e4m3_encode(mids)
    want = np.where(np.arange(0x7E) % 2 == 0, np.arange(0x7E), np.arange(1, 0x7F))
    assert (got == want).all()                            # ties go to the even code
    assert (O.e4m3_encode(mids * (1 + 1e-9)) == np.arange(1, 0x7F)).all()
    assert O.e4m3_encode([1e6, -1e6, 449.0])[0] == 0x7E and O.e4m3_encode([-1e6])[0] == 0xFE
    assert O.e4m3_encode([-1e-30])[0] == 0x80 and np.isnan(O.e4m3_decode(O.e4m3_encode([np.nan])))[0]


def test_quantize_rows_error_bound_and_scale():
    rng = _rng(3)
    w = (rng.standard_normal((40, 96)) * 0.02).astype(np.float32)
    w[5] = 0.0
    q, s = O.quantize_fp8_rows(w)
    assert s.dtype == np.float32 and s[5] == 0 and (q[5] == 0).all()
    deq = O.dequantize_fp8_rows(q, s)
    rows = np.arange(40) != 5
    # the largest magnitude of a row lands on +-448 (within the float32 rounding of the scale)
    top = np.abs(w[rows]).argmax(axis=1)
    assert np.all(np.abs(O.e4m3_decode(q[rows][np.arange(39), top])) == 448.0)
    # every element within half a mantissa step (2^-4 relative) or half the subnormal step
    err = np.abs(deq[rows] - w[rows].astype(np.float64))
    bound = np.maximum(np.abs(w[rows]) * 2.0 ** -4, s[rows, None] * 2.0 ** -10) * (1 + 1e-6)
    assert (err <= bound).all()


# --------------------------------------------------------- FP8 activations ---

def test_bf16_round_matches_the_format():
    # hand values: exact ones stay, a tie rounds to the even mantissa, just above a tie rounds up
    one = 1.0
    assert O.bf16_round([one, -2.5, 0.0])[0] == 1.0
    assert O.bf16_round([1.0 + 2.0 ** -8])[0] == 1.0                       # tie -> even (1.0)
    assert O.bf16_round([1.0 + 3 * 2.0 ** -8])[0] == 1.0 + 2.0 ** -6       # tie -> even (1 + 2^-6)
    assert O.bf16_round([1.0 + 2.0 ** -8 + 2.0 ** -20])[0] == 1.0 + 2.0 ** -7
    # and torch's float32 -> bfloat16 conversion (round to nearest even) on random values
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(4096) * np.exp(rng.uniform(-20, 20, 4096))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(O.bf16_round(v), ref)


def test_w8a8_mlp_one_element_closed_form():
    # d = F = 1: a one-element row quantises to +-448 times its scale, i.e. to itself up to the
    # float32 rounding of the scale, so the W8A8 MLP is c * bf16(silu(a x) * b x)
    for x0, a, b, c in [(0.75, 1.5, -2.0, 0.5), (-3.0, 0.25, 0.125, -1.0), (1e-3, 40.0, 2.0, 3.0)]:
        y = O.expert_mlp_w8a8(np.array([[x0]]), np.array([[a]]), np.array([[b]]), np.array([[c]]))[0, 0]
        z = a * x0
        h = O.bf16_round([z / (1.0 + math.exp(-z)) * (b * x0)])[0]
        assert y == pytest.approx(c * h, rel=1e-6)


def test_w8a8_mlp_error_is_the_activation_quantisation_error():
    # random bf16-like rows through a 256 -> 128 -> 256 expert: the W8A8 output differs from the
    # exact MLP by E4M3's relative precision (3 mantissa bits: at most 2^-4 of an element,
    # about 2^-4 / sqrt(3) in rms), so the relative max error sits between 0.1 % and 8 %:
    # no quantisation (error 0) or a dropped or doubled scale (error ~100 %) fall outside
    rng = np.random.default_rng(11)
    d, F = 256, 128
    x = O.bf16_round(rng.standard_normal((64, d)))
    wg, wu = (O.bf16_round(rng.standard_normal((F, d)) * 0.05) for _ in range(2))
    wd = O.bf16_round(rng.standard_normal((d, F)) * 0.05)
    exact = O.expert_mlp(x, wg, wu, wd)
    got = O.expert_mlp_w8a8(x, wg, wu, wd)
    rel = np.abs(got - exact).max() / np.abs(exact).max()
    assert 1e-3 < rel < 8e-2, rel
    # scaling an input row by a power of two changes only its scale, by the same power of two:
    # the quantised rows scale exactly
    q1, s1 = O.quantize_fp8_rows(x)
    q2, s2 = O.quantize_fp8_rows(x * 8.0)
    assert np.array_equal(q1, q2) and np.array_equal(s2, s1 * np.float32(8.0))


def test_layer_forward_takes_the_w8a8_mlp():
    # the layer with the W8A8 MLP equals the same routing and combine over expert_mlp_w8a8
    w = synth.WORKLOADS["mini_qwen3"].with_(T=40, n_experts=8, top_k=2, d_model=128, d_ff=128)
    x = synth.as_f64(synth.host_tensor(w, "x"), w.dtype)
    wr = synth.as_f64(synth.host_tensor(w, "w_router"), w.dtype)
    ex = {g: tuple(synth.as_f64(a, w.dtype) for a in synth.host_expert(w, g)) for g in range(w.n_experts)}
    res = O.layer_forward(x, wr, None, ex.__getitem__, top_k=2, mlp=O.expert_mlp_w8a8)
    plain = O.layer_forward(x, wr, None, ex.__getitem__, top_k=2)
    assert (res.idx == plain.idx).all()
    for t in (0, 17, 39):
        want = sum(res.gate[t, j] * O.expert_mlp_w8a8(x[t:t + 1], *ex[int(res.idx[t, j])])[0] for j in range(2))
        assert np.allclose(res.out[t], want, rtol=0, atol=1e-12)
    rel = np.abs(res.out - plain.out).max() / np.abs(plain.out).max()
    assert 1e-4 < rel < 8e-2
