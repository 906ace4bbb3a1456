"""Seeded synthetic inputs for the MoE FFN layer.

This package is the one module both sides of a parity check draw from: the
CUDA path (through the device filler in ``gen_device.cu``) and the CPU oracle
(through the host filler in ``gen_host.c`` or the pure-numpy restatement
below). It holds no MoE arithmetic: only the counter-based generator, the
router-bias recipe that synthesises skewed expert loads, and the workload
shapes.

Generator definition: see the header of ``gen_host.c``. In short, element i of
stream (seed, tensor_id) is an Irwin-Hall(4) sum of four 16-bit fields of the
(i+1)-th SplitMix64 output, centred, multiplied once in binary32 by a scale
that gives standard deviation sigma, and (for bf16 tensors) rounded to
bfloat16 with round-to-nearest-even.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

from .workloads import WORKLOADS, Workload, TENSOR_ID  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBDIR = os.path.join(_HERE, "lib")
HOST_LIB = os.path.join(_LIBDIR, "libsynth_host.so")
DEVICE_LIB = os.path.join(_LIBDIR, "libsynth_device.so")

_M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_KEYMUL = 0xD1B54A32D192ED03

# standard deviation of c = 2*S - 262140, S a sum of four uniform 16-bit fields
_C_STD = 2.0 * math.sqrt((65536.0 ** 2 - 1.0) / 3.0)


def scale_for(sigma: float) -> np.float32:
    """The binary32 multiplier that turns the centred integer into N(0, sigma^2)."""
    return np.float32(sigma / _C_STD)


def _mix64_int(z: int) -> int:
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    return _mix64_int(seed * _GOLDEN + tensor_id * _KEYMUL)


def _mix64_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def centred_numpy(seed: int, tensor_id: int, start: int, n: int) -> np.ndarray:
    """The centred integers c(start..start+n) in pure numpy (int32)."""
    key = np.uint64(stream_key(seed, tensor_id))
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        b = _mix64_np(key + i * np.uint64(_GOLDEN))
    m = np.uint64(0xFFFF)
    s = (b & m) + ((b >> np.uint64(16)) & m) + ((b >> np.uint64(32)) & m) + ((b >> np.uint64(48)) & m)
    return (2 * s.astype(np.int64) - 262140).astype(np.int32)


def bf16_bits_from_f32(v: np.ndarray) -> np.ndarray:
    """Round binary32 values to bfloat16 (RNE); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_numpy(seed: int, tensor_id: int, start: int, n: int, sigma: float, dtype: str) -> np.ndarray:
    """Pure-numpy restatement of the generator (slow; used to check the C one)."""
    v = centred_numpy(seed, tensor_id, start, n).astype(np.float32) * scale_for(sigma)
    v = v.astype(np.float32)
    return bf16_bits_from_f32(v) if dtype == "bf16" else v


# --------------------------------------------------------------------------
# host library (C + OpenMP)

def build_host(force: bool = False) -> str:
    os.makedirs(_LIBDIR, exist_ok=True)
    src = os.path.join(_HERE, "gen_host.c")
    if force or not os.path.exists(HOST_LIB) or os.path.getmtime(HOST_LIB) < os.path.getmtime(src):
        tmp = HOST_LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp])
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_device(force: bool = False) -> str:
    os.makedirs(_LIBDIR, exist_ok=True)
    src = os.path.join(_HERE, "gen_device.cu")
    if force or not os.path.exists(DEVICE_LIB) or os.path.getmtime(DEVICE_LIB) < os.path.getmtime(src):
        tmp = DEVICE_LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", "-O3", "-shared", "-Xcompiler", "-fPIC", "-std=c++17",
                               "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
                               src, "-o", tmp])
        os.replace(tmp, DEVICE_LIB)
    return DEVICE_LIB


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            build_host()
        lib = ctypes.CDLL(HOST_LIB)
        u64 = ctypes.c_uint64
        lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, ctypes.c_float, ctypes.c_void_p]
        lib.synth_normal_bf16.argtypes = [u64, u64, u64, u64, ctypes.c_float, ctypes.c_void_p]
        lib.synth_stream_key.argtypes = [u64, u64]
        lib.synth_stream_key.restype = u64
        _host = lib
    return _host


def normal(seed: int, tensor_id: int, shape, sigma: float, dtype: str, start: int = 0) -> np.ndarray:
    """Host-generated tensor of the given shape: float32 values, or bf16 bit patterns (uint16)."""
    n = int(np.prod(shape)) if len(shape) else 1
    lib = _host_lib()
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        lib.synth_normal_bf16(seed, tensor_id, start, n, float(scale_for(sigma)), out.ctypes.data)
    elif dtype == "f32":
        out = np.empty(n, dtype=np.float32)
        lib.synth_normal_f32(seed, tensor_id, start, n, float(scale_for(sigma)), out.ctypes.data)
    else:
        raise ValueError(dtype)
    return out.reshape(shape)


def as_f64(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 view of generated values (bf16 bit patterns or float32)."""
    if dtype == "bf16":
        return bf16_bits_to_f32(arr).astype(np.float64)
    return np.asarray(arr, dtype=np.float32).astype(np.float64)


def router_bias(n_experts: int, s: float) -> np.ndarray | None:
    """Per-expert router bias b_e = -s * ln(e + 1) (binary32), or None when s == 0.

    Added to the router logits it scales expert e's softmax weight by
    (e+1)^-s, a Zipf(s) skew over experts; it is how skewed traffic is
    synthesised here, not a learned quantity.
    """
    if s == 0:
        return None
    return np.array([np.float32(-s * math.log(e + 1.0)) for e in range(n_experts)], dtype=np.float32)


# --------------------------------------------------------------------------
# device filler

def _device_lib():
    global _dev
    if _dev is None:
        if not os.path.exists(DEVICE_LIB):
            raise RuntimeError(f"synth device library missing: {DEVICE_LIB} (run __graft_entry__.build())")
        lib = ctypes.CDLL(DEVICE_LIB)
        lib.synth_fill_device.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                          ctypes.c_uint64, ctypes.c_float, ctypes.c_int, ctypes.c_void_p]
        lib.synth_fill_device.restype = ctypes.c_int
        _dev = lib
    return _dev


def fill_device(tensor, seed: int, tensor_id: int, sigma: float, start: int = 0) -> None:
    """Fill a contiguous torch CUDA tensor (float32 or bfloat16) in place on the current stream."""
    import torch
    assert tensor.is_cuda and tensor.is_contiguous()
    if tensor.dtype == torch.bfloat16:
        dt = 1
    elif tensor.dtype == torch.float32:
        dt = 0
    else:
        raise TypeError(tensor.dtype)
    rc = _device_lib().synth_fill_device(tensor.data_ptr(), tensor.numel(), seed, tensor_id, start,
                                         float(scale_for(sigma)), dt,
                                         torch.cuda.current_stream(tensor.device).cuda_stream)
    if rc != 0:
        raise RuntimeError(f"synth_fill_device failed with cudaError {rc}")


# --------------------------------------------------------------------------
# whole-workload helpers

def shapes(w: Workload) -> dict:
    G = w.n_experts + w.n_shared
    return {
        "x": (w.T, w.d_model),
        "w_router": (w.n_experts, w.d_model),
        "w_gate": (G, w.d_ff, w.d_model),
        "w_up": (G, w.d_ff, w.d_model),
        "w_down": (G, w.d_model, w.d_ff),
    }


def host_tensor(w: Workload, name: str) -> np.ndarray:
    """One whole input tensor generated on the host (bf16 bit patterns or float32)."""
    sigma = w.x_sigma if name == "x" else w.w_sigma
    return normal(w.seed, TENSOR_ID[name], shapes(w)[name], sigma, w.dtype)


def host_expert(w: Workload, g: int):
    """Expert g's (W_gate [F,d], W_up [F,d], W_down [d,F]) generated on the host.

    Expert g's slab starts at element g*F*d of each weight stream, so this
    reproduces the slices of the whole tensors without materialising them.
    """
    F, d = w.d_ff, w.d_model
    out = []
    for name, shp in (("w_gate", (F, d)), ("w_up", (F, d)), ("w_down", (d, F))):
        out.append(normal(w.seed, TENSOR_ID[name], shp, w.w_sigma, w.dtype, start=g * F * d))
    return tuple(out)


def device_inputs(w: Workload, device="cuda"):
    """All inputs of a workload generated directly in device memory (torch tensors)."""
    import torch
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    t = {}
    for name, shp in shapes(w).items():
        t[name] = torch.empty(shp, dtype=dt, device=device)
        fill_device(t[name], w.seed, TENSOR_ID[name], w.x_sigma if name == "x" else w.w_sigma)
    b = router_bias(w.n_experts, w.bias_s)
    t["bias"] = None if b is None else torch.from_numpy(b).to(device)
    return t


def host_to_torch(arr: np.ndarray, dtype: str):
    """Wrap generated host data as a CPU torch tensor of the workload dtype (no copy of values)."""
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
