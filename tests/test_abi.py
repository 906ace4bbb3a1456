"""The C ABI without a GPU: libmoe.so loads, exports what include/moe.h declares, and
its host-side logic (validation, capacity, workspace sizing) behaves as documented.
No call here launches a kernel."""
import ctypes
import os
import re

import pytest

import oracle as O
import sparse_expert_mlp_router_b300 as moe
from sparse_expert_mlp_router_b300.build import LIB_PATH

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    assert os.path.exists(LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    declared = _declared_symbols()
    assert len(declared) >= 16
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(moe.EXPORTS)


def _cfg(**kw):
    base = dict(T=4096, d_model=7168, n_experts=256, top_k=8, d_ff=2048, n_shared=1, score="sigmoid",
                capacity_factor=1.25, dtype="bf16")
    base.update(kw)
    return moe.make_config(**base)


def test_status_strings():
    for code in range(7):
        assert moe.status_string(code).startswith("MOE_")
    assert "unknown" in moe.status_string(99)


def test_config_validation():
    assert moe.moe_check_config(_cfg()) == moe.MOE_OK
    assert moe.moe_check_config(_cfg(top_k=9, n_experts=8)) == moe.MOE_ERR_INVALID_ARG   # k > E
    assert moe.moe_check_config(_cfg(T=0)) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_check_config(_cfg(d_model=100)) == moe.MOE_ERR_UNSUPPORTED          # bf16 needs d % 128
    assert moe.moe_check_config(_cfg(d_model=100, d_ff=100, dtype="f32")) == moe.MOE_OK
    assert moe.moe_check_config(_cfg(n_experts=512)) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_check_config(_cfg(top_k=9, n_experts=16)) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_check_config(_cfg(n_shared=2)) == moe.MOE_ERR_UNSUPPORTED
    assert moe.moe_check_config(_cfg(capacity_factor=float("nan"))) == moe.MOE_ERR_INVALID_ARG
    assert moe.lib().moe_check_config(None) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_workspace_size(_cfg(T=0)) == 0


@pytest.mark.parametrize("T,k,E,cf", [
    (4096, 8, 256, 1.25), (10, 1, 4, 1.0), (5, 1, 2, 0.8), (6, 1, 2, 0.5), (333, 8, 32, 1.1),
    (257, 6, 48, 1.25), (1, 1, 1, 0.001), (100, 2, 8, 0.0), (100, 2, 8, -3.0), (7, 3, 5, 1e30),
    (8192, 8, 128, 0.3), (999, 7, 13, 2.0 / 3.0),
])
def test_capacity_is_exact_ceiling(T, k, E, cf):
    ref = O.capacity(T, k, E, cf)
    ref = T if ref is None else min(ref, T)
    c = moe.make_config(T=T, d_model=128, n_experts=E, top_k=k, d_ff=128, capacity_factor=cf)
    assert moe.moe_capacity(c) == ref
    assert moe.moe_rows_capacity(c) == min(T * k, E * ref)


def test_workspace_grows_with_rows():
    small = moe.moe_workspace_size(_cfg(capacity_factor=0.5))
    big = moe.moe_workspace_size(_cfg(capacity_factor=0.0))
    assert 0 < small < big
    c = _cfg()
    assert moe.moe_grouped_rows(c) == moe.moe_rows_capacity(c) + 4096
    assert moe.moe_workspace_size(c) % 256 == 0


def test_host_validation_rejects_before_any_launch():
    c = _cfg()
    L = moe.lib()
    # null data pointers: rejected on the host, nothing is enqueued
    assert L.moe_router_topk(ctypes.byref(c), None, None, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_layer_forward(ctypes.byref(c), None, None, None, None, None, None, None, None, None, None, 0,
                               None) == moe.MOE_ERR_INVALID_ARG
    # misaligned pointers
    p = 0x10000
    assert L.moe_router_topk(ctypes.byref(c), p + 2, p, None, p, p, None, None) == moe.MOE_ERR_INVALID_ARG
    # workspace too small / misaligned
    assert L.moe_permute(ctypes.byref(c), p, p, p, p, p, p, p, p, 256, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_permute(ctypes.byref(c), p, p, p, p, p, p, p, p + 16, 1 << 40, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_combine(ctypes.byref(c), p, p, p, p, p, 16, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_selftest_bounded_wait(None, 0, 10, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_init(p + 8, 4096, None) == moe.MOE_ERR_INVALID_ARG
    # unsupported configuration reaches no launch either
    bad = _cfg(d_model=100)
    assert L.moe_grouped_ffn(ctypes.byref(bad), p, p, p, p, p, p, p, p, 1 << 40, None) == moe.MOE_ERR_UNSUPPORTED


def test_timed_variant_rejects_bad_event_count():
    c = _cfg()
    p = 0x10000
    L = moe.lib()
    ev = (ctypes.c_void_p * 7)()
    n = moe.moe_workspace_size(c)
    assert L.moe_layer_forward_timed(ctypes.byref(c), p, p, None, p, p, p, p, None, None, p, n, ev, 7,
                                     None) == moe.MOE_ERR_INVALID_ARG


def test_fp8_quantiser_and_stats_validation_before_any_launch():
    L = moe.lib()
    p = 0x10000
    c = _cfg()                                   # d_model 7168, d_ff 2048: shapes the FP8 kernels take
    n = moe.moe_workspace_size(c)
    ok = (p, p, p, p, p, p)                      # codes / scales of W_g, W_u, W_d

    def layer(cfg, w8):
        return L.moe_layer_forward_fp8(ctypes.byref(cfg), p, p, None, *w8, p, None, None, p, n, None)

    def ffn(cfg, w8):
        return L.moe_grouped_ffn_fp8(ctypes.byref(cfg), p, p, p, *w8, p, p, n, None)

    for call in (layer, ffn):
        assert call(c, (p, None, p, p, p, p)) == moe.MOE_ERR_INVALID_ARG          # a missing scale
        assert call(c, (p + 8, p, p, p, p, p)) == moe.MOE_ERR_INVALID_ARG         # codes not 16-byte aligned
        assert call(c, (p, p + 2, p, p, p, p)) == moe.MOE_ERR_INVALID_ARG         # scales not 4-byte aligned
        assert call(_cfg(d_model=384), ok) == moe.MOE_ERR_UNSUPPORTED             # d_model not a multiple of 256
        assert call(_cfg(d_ff=200), ok) == moe.MOE_ERR_UNSUPPORTED                # d_ff not a multiple of 128
        assert call(_cfg(dtype="f32", d_model=256, d_ff=128), ok) == moe.MOE_ERR_UNSUPPORTED   # float32 layers
    assert L.moe_quantize_fp8_rows(p, 4, 24, p, p, None) == moe.MOE_ERR_INVALID_ARG   # row not 16 codes wide
    assert L.moe_quantize_fp8_rows(p, 0, 32, p, p, None) == moe.MOE_ERR_INVALID_ARG   # no rows
    assert L.moe_quantize_fp8_rows(p + 8, 4, 32, p, p, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_quantize_fp8_rows(p, 4, 32, p, p + 1, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_routing_stats(ctypes.byref(c), None, p, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_routing_stats(ctypes.byref(c), p + 2, p, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_routing_stats(ctypes.byref(_cfg(top_k=300)), p, p, None) == moe.MOE_ERR_INVALID_ARG


def test_launch_count_follows_the_grouping_path(monkeypatch):
    # router, grouping (one kernel with the row copy for a single 128-token chunk, else
    # histogram, scan, scatter and the row copy), the expert MLP (one persistent launch of both
    # contractions for a single chunk of a bf16 layer, else two) and the combine
    monkeypatch.delenv("MOE_FUSED_MLP", raising=False)
    monkeypatch.delenv("MOE_MLP_COMBINE", raising=False)
    assert moe.moe_layer_mlp_fused(_cfg(T=128)) == 1
    assert moe.moe_layer_launch_count(_cfg(T=128)) == 1 + 1 + 1 + 1
    monkeypatch.setenv("MOE_MLP_COMBINE", "1")                    # the combine inside the one launch
    assert moe.moe_layer_launch_count(_cfg(T=128)) == 1 + 1 + 1 + 0
    assert moe.moe_layer_launch_count(_cfg(T=129)) == 1 + 4 + 2 + 1   # two MLP launches: no effect
    monkeypatch.delenv("MOE_MLP_COMBINE")
    assert moe.moe_layer_mlp_fused(_cfg(T=129)) == 0
    assert moe.moe_layer_launch_count(_cfg(T=129)) == 1 + 4 + 2 + 1
    assert moe.moe_layer_launch_count(_cfg(top_k=300)) == -1
    assert moe.moe_layer_mlp_fused(_cfg(top_k=300)) == -1
    # the environment forces either way (read at every call); float32 layers always take two
    monkeypatch.setenv("MOE_FUSED_MLP", "0")
    assert moe.moe_layer_mlp_fused(_cfg(T=128)) == 0
    assert moe.moe_layer_launch_count(_cfg(T=128)) == 1 + 1 + 2 + 1
    monkeypatch.setenv("MOE_FUSED_MLP", "1")
    assert moe.moe_layer_mlp_fused(_cfg(T=129)) == 1
    assert moe.moe_layer_mlp_fused(_cfg(T=128, dtype="f32")) == 0
    # per weight format: FP8 weights keep two expert launches; W8A8 three (gate/up, h's
    # quantiser, down), and for multi-chunk batches a per-token quantiser before the code-row copy
    monkeypatch.delenv("MOE_FUSED_MLP", raising=False)
    assert moe.moe_layer_launch_count_weights(_cfg(T=128), "bf16") == 1 + 1 + 1 + 1
    assert moe.moe_layer_launch_count_weights(_cfg(T=128), "fp8") == 1 + 1 + 2 + 1
    assert moe.moe_layer_launch_count_weights(_cfg(T=128), "w8a8") == 1 + 1 + 3 + 1
    assert moe.moe_layer_mlp_fused_weights(_cfg(T=128), "bf16") == 1
    assert moe.moe_layer_mlp_fused_weights(_cfg(T=128), "fp8") == 0
    assert moe.moe_layer_mlp_fused_weights(_cfg(T=128), "w8a8") == 0
    assert moe.moe_layer_mlp_fused_weights(_cfg(T=128, d_model=384), "w8a8") == -1
    assert moe.moe_layer_launch_count_weights(_cfg(T=129), "fp8") == 1 + 4 + 2 + 1
    assert moe.moe_layer_launch_count_weights(_cfg(T=129), "w8a8") == 1 + 5 + 3 + 1
    assert moe.moe_layer_launch_count_weights(_cfg(T=129, d_model=384), "w8a8") == -1   # FP8 kernels need d % 256
    # W8A8 as one launch only on request (it measured slower than three)
    monkeypatch.setenv("MOE_FUSED_MLP", "1")
    assert moe.moe_layer_mlp_fused_weights(_cfg(T=128), "w8a8") == 1
    assert moe.moe_layer_launch_count_weights(_cfg(T=128), "w8a8") == 1 + 1 + 1 + 1
    assert moe.moe_layer_launch_count_weights(_cfg(T=129), "w8a8") == 1 + 5 + 1 + 1



def test_float32_layers_read_routed_rows_through_src_token(monkeypatch):
    # a float32 layer's expert MLP reads x through src_token: no grouped copy of x in its
    # permute stage (router, grouping, two MLP kernels, combine)
    monkeypatch.delenv("MOE_FUSED_MLP", raising=False)
    tiny = dict(d_model=64, n_experts=8, top_k=2, d_ff=128, n_shared=0, score="softmax", capacity_factor=0.0,
                dtype="f32")
    assert moe.moe_layer_launch_count(_cfg(T=64, **tiny)) == 1 + 1 + 2 + 1
    assert moe.moe_layer_launch_count(_cfg(T=129, **tiny)) == 1 + 3 + 2 + 1
