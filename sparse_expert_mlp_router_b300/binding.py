"""ctypes binding of libmoe.so: same names as the C ABI (include/moe.h), argument marshalling only.

Tensors are torch tensors on the GPU; every call passes their data pointers and
the current CUDA stream to the library, checks the returned status and raises
MoeError on failure. No computation happens here.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .build import LIB_PATH

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, \
    MOE_ERR_DEVICE_INDEX = range(7)
MOE_F32, MOE_BF16 = 0, 1
MOE_SOFTMAX, MOE_SIGMOID = 0, 1

# Every symbol include/moe.h declares.
EXPORTS = [
    "moe_status_string", "moe_check_config", "moe_capacity", "moe_rows_capacity", "moe_grouped_rows",
    "moe_workspace_size", "moe_workspace_init", "moe_router_topk", "moe_permute", "moe_grouped_ffn",
    "moe_combine", "moe_layer_forward", "moe_layer_forward_timed", "moe_get_device_error",
    "moe_clear_device_error", "moe_selftest_bounded_wait", "moe_layer_launch_count", "moe_layer_mlp_fused",
    "moe_layer_launch_count_weights", "moe_layer_mlp_fused_weights",
    "moe_permute_noalloc", "moe_routing_stats", "moe_quantize_fp8_rows", "moe_grouped_ffn_fp8",
    "moe_layer_forward_fp8", "moe_layer_forward_fp8_timed", "moe_layer_forward_w8a8", "moe_layer_forward_w8a8_timed",
]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


class MoeRoutingStats(ctypes.Structure):
    _fields_ = [
        ("tokens", ctypes.c_int32), ("pairs", ctypes.c_int32), ("kept", ctypes.c_int32),
        ("dropped", ctypes.c_int32), ("experts_touched", ctypes.c_int32), ("max_load", ctypes.c_int32),
        ("capacity", ctypes.c_int32), ("mean_load", ctypes.c_float), ("efficiency", ctypes.c_float),
    ]
    FIELDS = [n for n, _ in _fields_]


class MoeConfig(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
        ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("n_shared", ctypes.c_int32),
        ("score", ctypes.c_int32), ("renormalize", ctypes.c_int32), ("capacity_factor", ctypes.c_float),
        ("dtype", ctypes.c_int32),
    ]

    def __repr__(self):
        return "MoeConfig(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


def make_config(T: int, d_model: int, n_experts: int, top_k: int, d_ff: int, n_shared: int = 0,
                score: str = "softmax", renormalize: bool = True, capacity_factor: float = 0.0,
                dtype: str = "bf16") -> MoeConfig:
    return MoeConfig(T, d_model, n_experts, top_k, d_ff, n_shared,
                     MOE_SOFTMAX if score == "softmax" else MOE_SIGMOID, 1 if renormalize else 0,
                     float(capacity_factor), MOE_BF16 if dtype == "bf16" else MOE_F32)


_lib = None
_vp = ctypes.c_void_p
_cfgp = ctypes.POINTER(MoeConfig)


def lib() -> ctypes.CDLL:
    """The loaded libmoe.so. Raises if the library has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmoe.so is not built ({LIB_PATH}); run `python -m sparse_expert_mlp_router_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        i32, i64, sz, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint64
        sig = {
            "moe_status_string": ([i32], ctypes.c_char_p),
            "moe_check_config": ([_cfgp], i32),
            "moe_capacity": ([_cfgp], i32),
            "moe_rows_capacity": ([_cfgp], i64),
            "moe_grouped_rows": ([_cfgp], i64),
            "moe_workspace_size": ([_cfgp], sz),
            "moe_workspace_init": ([_vp, sz, _vp], i32),
            "moe_router_topk": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], i32),
            "moe_permute": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, sz, _vp], i32),
            "moe_grouped_ffn": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, sz, _vp], i32),
            "moe_combine": ([_cfgp, _vp, _vp, _vp, _vp, _vp, sz, _vp], i32),
            "moe_layer_forward": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, sz, _vp], i32),
            "moe_layer_forward_timed": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, sz,
                                         ctypes.POINTER(_vp), i32, _vp], i32),
            "moe_get_device_error": ([_vp, _vp], i32),
            "moe_clear_device_error": ([_vp, _vp], i32),
            "moe_selftest_bounded_wait": ([_vp, sz, u64, _vp], i32),
            "moe_layer_launch_count": ([_cfgp], i32),
            "moe_layer_mlp_fused": ([_cfgp], i32),
            "moe_layer_launch_count_weights": ([_cfgp, i32], i32),
            "moe_layer_mlp_fused_weights": ([_cfgp, i32], i32),
            "moe_permute_noalloc": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp], i32),
            "moe_routing_stats": ([_cfgp, _vp, _vp, _vp], i32),
            "moe_quantize_fp8_rows": ([_vp, i64, i32, _vp, _vp, _vp], i32),
            "moe_grouped_ffn_fp8": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, sz, _vp], i32),
            "moe_layer_forward_fp8": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, sz,
                                       _vp], i32),
            "moe_layer_forward_fp8_timed": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                             _vp, sz, ctypes.POINTER(_vp), i32, _vp], i32),
            "moe_layer_forward_w8a8": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, sz,
                                        _vp], i32),
            "moe_layer_forward_w8a8_timed": ([_cfgp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                              _vp, sz, ctypes.POINTER(_vp), i32, _vp], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(code: int, where: str) -> None:
    if code != MOE_OK:
        raise MoeError(code, where)


# ------------------------------------------------------------------ queries

def moe_check_config(cfg: MoeConfig) -> int:
    return lib().moe_check_config(ctypes.byref(cfg))


def moe_capacity(cfg: MoeConfig) -> int:
    return lib().moe_capacity(ctypes.byref(cfg))


def moe_rows_capacity(cfg: MoeConfig) -> int:
    return lib().moe_rows_capacity(ctypes.byref(cfg))


def moe_grouped_rows(cfg: MoeConfig) -> int:
    return lib().moe_grouped_rows(ctypes.byref(cfg))


def moe_workspace_size(cfg: MoeConfig) -> int:
    return lib().moe_workspace_size(ctypes.byref(cfg))


def moe_layer_launch_count(cfg: MoeConfig) -> int:
    return lib().moe_layer_launch_count(ctypes.byref(cfg))


def moe_layer_mlp_fused(cfg: MoeConfig) -> int:
    return lib().moe_layer_mlp_fused(ctypes.byref(cfg))


WEIGHTS_MODE = {"bf16": 0, "f32": 0, "fp8": 1, "w8a8": 2}


def moe_layer_launch_count_weights(cfg: MoeConfig, weights: str) -> int:
    return lib().moe_layer_launch_count_weights(ctypes.byref(cfg), WEIGHTS_MODE[weights])


def moe_layer_mlp_fused_weights(cfg: MoeConfig, weights: str) -> int:
    return lib().moe_layer_mlp_fused_weights(ctypes.byref(cfg), WEIGHTS_MODE[weights])


# -------------------------------------------------------------- workspace

def alloc_workspace(cfg: MoeConfig, device="cuda"):
    """A zero-status workspace of moe_workspace_size(cfg) bytes (torch uint8 tensor)."""
    import torch
    n = moe_workspace_size(cfg)
    if n == 0:
        raise MoeError(moe_check_config(cfg) or MOE_ERR_INVALID_ARG, "moe_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    moe_workspace_init(ws)
    return ws


def moe_workspace_init(ws, stream=None) -> None:
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


def moe_get_device_error(ws, stream=None) -> int:
    return lib().moe_get_device_error(_ptr(ws), _stream(stream))


def moe_clear_device_error(ws, stream=None) -> None:
    _check(lib().moe_clear_device_error(_ptr(ws), _stream(stream)), "moe_clear_device_error")


def moe_selftest_bounded_wait(ws, limit_ns: int, stream=None) -> None:
    _check(lib().moe_selftest_bounded_wait(_ptr(ws), ws.numel(), int(limit_ns), _stream(stream)),
           "moe_selftest_bounded_wait")


# ------------------------------------------------------------------ stages

def moe_router_topk(cfg, x, w_router, bias, topk_idx, topk_gate, scores=None, stream=None) -> None:
    _check(lib().moe_router_topk(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(topk_idx),
                                 _ptr(topk_gate), _ptr(scores), _stream(stream)), "moe_router_topk")


def moe_permute(cfg, topk_idx, x, counts, offsets, dest_row, src_token, x_perm, ws, stream=None) -> None:
    _check(lib().moe_permute(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets),
                             _ptr(dest_row), _ptr(src_token), _ptr(x_perm), _ptr(ws), ws.numel(),
                             _stream(stream)), "moe_permute")


def moe_permute_noalloc(cfg, topk_idx, x, counts, offsets, dest_row, src_token, x_perm, status=None,
                        stream=None) -> None:
    """moe_permute without a workspace, for callers that cannot allocate device memory (see moe.h)."""
    _check(lib().moe_permute_noalloc(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(counts), _ptr(offsets),
                                     _ptr(dest_row), _ptr(src_token), _ptr(x_perm), _ptr(status),
                                     _stream(stream)), "moe_permute_noalloc")


def moe_grouped_ffn(cfg, x_perm, offsets, x, w_gate, w_up, w_down, y_perm, ws, stream=None) -> None:
    _check(lib().moe_grouped_ffn(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(x), _ptr(w_gate),
                                 _ptr(w_up), _ptr(w_down), _ptr(y_perm), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_ffn")


def moe_combine(cfg, y_perm, dest_row, topk_gate, out, ws, stream=None) -> None:
    _check(lib().moe_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(dest_row), _ptr(topk_gate), _ptr(out),
                             _ptr(ws), ws.numel(), _stream(stream)), "moe_combine")


def moe_layer_forward(cfg, x, w_router, bias, w_gate, w_up, w_down, out, ws, topk_idx_out=None,
                      counts_out=None, stream=None) -> None:
    _check(lib().moe_layer_forward(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_gate),
                                   _ptr(w_up), _ptr(w_down), _ptr(out), _ptr(topk_idx_out), _ptr(counts_out),
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_layer_forward")


def moe_layer_forward_timed(cfg, x, w_router, bias, w_gate, w_up, w_down, out, ws, events,
                            topk_idx_out=None, counts_out=None, stream=None) -> None:
    """events: up to 6 torch.cuda.Event(enable_timing=True) recorded at the stage boundaries."""
    for e in events:
        if e.cuda_event == 0:        # torch creates the CUDA event on its first record
            e.record()
    handles = (_vp * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_layer_forward_timed(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w_gate),
                                         _ptr(w_up), _ptr(w_down), _ptr(out), _ptr(topk_idx_out),
                                         _ptr(counts_out), _ptr(ws), ws.numel(), handles, len(events),
                                         _stream(stream)), "moe_layer_forward_timed")


def moe_routing_stats(cfg, counts, stats=None, stream=None):
    """Routing telemetry from per-expert counts (see include/moe.h). `stats`: a device buffer of
    at least sizeof(moe_routing_stats_t) bytes (a uint8 tensor), or None to allocate one.
    Returns the buffer; read it with routing_stats_to_dict()."""
    import torch
    if stats is None:
        stats = torch.zeros(ctypes.sizeof(MoeRoutingStats), dtype=torch.uint8, device=counts.device)
    _check(lib().moe_routing_stats(ctypes.byref(cfg), _ptr(counts), _ptr(stats), _stream(stream)),
           "moe_routing_stats")
    return stats


def routing_stats_to_dict(stats) -> dict:
    """Host copy of a moe_routing_stats_t device buffer as a dict (synchronises)."""
    raw = bytes(stats.cpu().numpy().tobytes())[:ctypes.sizeof(MoeRoutingStats)]
    st = MoeRoutingStats.from_buffer_copy(raw)
    return {n: getattr(st, n) for n in MoeRoutingStats.FIELDS}


# ------------------------------------------------------------- FP8 weights

def moe_quantize_fp8_rows(w, wq=None, scale=None, stream=None):
    """E4M3 codes and per-row float32 scales of a bf16 matrix (any leading shape; rows are the
    product of all but the last dimension). Returns (wq uint8, scale float32)."""
    import torch
    rows = w.numel() // w.shape[-1]
    if wq is None:
        wq = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    if scale is None:
        scale = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
    _check(lib().moe_quantize_fp8_rows(_ptr(w), rows, w.shape[-1], _ptr(wq), _ptr(scale), _stream(stream)),
           "moe_quantize_fp8_rows")
    return wq, scale


def moe_grouped_ffn_fp8(cfg, x_perm, offsets, x, wg_q, wg_s, wu_q, wu_s, wd_q, wd_s, y_perm, ws, stream=None) -> None:
    _check(lib().moe_grouped_ffn_fp8(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(x), _ptr(wg_q),
                                     _ptr(wg_s), _ptr(wu_q), _ptr(wu_s), _ptr(wd_q), _ptr(wd_s), _ptr(y_perm),
                                     _ptr(ws), ws.numel(), _stream(stream)), "moe_grouped_ffn_fp8")


def moe_layer_forward_fp8(cfg, x, w_router, bias, wg_q, wg_s, wu_q, wu_s, wd_q, wd_s, out, ws, topk_idx_out=None,
                          counts_out=None, stream=None) -> None:
    _check(lib().moe_layer_forward_fp8(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(wg_q),
                                       _ptr(wg_s), _ptr(wu_q), _ptr(wu_s), _ptr(wd_q), _ptr(wd_s), _ptr(out),
                                       _ptr(topk_idx_out), _ptr(counts_out), _ptr(ws), ws.numel(),
                                       _stream(stream)), "moe_layer_forward_fp8")


def moe_layer_forward_fp8_timed(cfg, x, w_router, bias, wg_q, wg_s, wu_q, wu_s, wd_q, wd_s, out, ws, events,
                                topk_idx_out=None, counts_out=None, stream=None) -> None:
    for e in events:
        if e.cuda_event == 0:
            e.record()
    handles = (_vp * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_layer_forward_fp8_timed(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(wg_q),
                                             _ptr(wg_s), _ptr(wu_q), _ptr(wu_s), _ptr(wd_q), _ptr(wd_s), _ptr(out),
                                             _ptr(topk_idx_out), _ptr(counts_out), _ptr(ws), ws.numel(), handles,
                                             len(events), _stream(stream)), "moe_layer_forward_fp8_timed")


def moe_layer_forward_w8a8(cfg, x, w_router, bias, wg_q, wg_s, wu_q, wu_s, wd_q, wd_s, out, ws, topk_idx_out=None,
                           counts_out=None, stream=None) -> None:
    _check(lib().moe_layer_forward_w8a8(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(wg_q),
                                        _ptr(wg_s), _ptr(wu_q), _ptr(wu_s), _ptr(wd_q), _ptr(wd_s), _ptr(out),
                                        _ptr(topk_idx_out), _ptr(counts_out), _ptr(ws), ws.numel(),
                                        _stream(stream)), "moe_layer_forward_w8a8")


def moe_layer_forward_w8a8_timed(cfg, x, w_router, bias, wg_q, wg_s, wu_q, wu_s, wd_q, wd_s, out, ws, events,
                                 topk_idx_out=None, counts_out=None, stream=None) -> None:
    for e in events:
        if e.cuda_event == 0:
            e.record()
    handles = (_vp * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_layer_forward_w8a8_timed(ctypes.byref(cfg), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(wg_q),
                                              _ptr(wg_s), _ptr(wu_q), _ptr(wu_s), _ptr(wd_q), _ptr(wd_s), _ptr(out),
                                              _ptr(topk_idx_out), _ptr(counts_out), _ptr(ws), ws.numel(), handles,
                                              len(events), _stream(stream)), "moe_layer_forward_w8a8_timed")
