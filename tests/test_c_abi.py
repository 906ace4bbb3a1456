"""A plain C program (tests/c_abi/layer_forward.c) as a client of libmoe.so.

CPU: it compiles against include/moe.h and links against the built library and the CUDA
runtime alone (no Python, no torch). GPU: its layer output, top-k ids and counts equal,
bit for bit, those of the same call made through the Python binding on the same inputs.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import sparse_expert_mlp_router_b300 as moe
from sparse_expert_mlp_router_b300.build import LIB_PATH

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "layer_forward.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
T, D, E, K, F = 64, 256, 8, 2, 256


def _compile(out_dir) -> str:
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(LIB_PATH):
        pytest.skip("libmoe.so is not built")
    lib_dir = os.path.dirname(LIB_PATH)
    exe = os.path.join(str(out_dir), "layer_forward")
    cmd = [cc, "-O2", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), SRC, "-o", exe, "-L", lib_dir, "-lmoe",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-Wl,-rpath," + lib_dir,
           "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _hash_values(seed: int, n: int, scale_log2: int) -> np.ndarray:
    """The C program's inputs: the same integer hash, the same exact float32 steps."""
    with np.errstate(over="ignore"):
        h = np.arange(n, dtype=np.uint32) * np.uint32(2654435761) ^ np.uint32(seed)
        h ^= h >> np.uint32(15)
        h *= np.uint32(0x2C1B3C6D)
        h ^= h >> np.uint32(12)
        h *= np.uint32(0x297A2D39)
        h ^= h >> np.uint32(15)
    u = (h >> np.uint32(8)).astype(np.float32) * np.float32(1.0 / 16777216.0)
    return (u * np.float32(2.0) - np.float32(1.0)) / np.float32(2 ** scale_log2)


def test_c_client_compiles_and_links(tmp_path):
    exe = _compile(tmp_path)
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_c_client_matches_the_binding(tmp_path):
    import torch

    exe = _compile(tmp_path)
    out_file = os.path.join(str(tmp_path), "out.bin")
    r = subprocess.run([exe, out_file], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    raw = np.fromfile(out_file, dtype=np.uint8)
    n_out, n_idx = T * D * 2, T * K * 4
    assert raw.size == n_out + n_idx + E * 4
    c_out = raw[:n_out].view(np.uint16).reshape(T, D)
    c_idx = raw[n_out:n_out + n_idx].view(np.int32).reshape(T, K)
    c_counts = raw[n_out + n_idx:].view(np.int32)

    def tensor(seed, shape, scale_log2):
        v = _hash_values(seed, int(np.prod(shape)), scale_log2).reshape(shape)
        return torch.from_numpy(v).to(torch.bfloat16).cuda()

    x = tensor(1, (T, D), 0)
    w_router = tensor(2, (E, D), 4)
    w_gate = tensor(3, (E, F, D), 4)
    w_up = tensor(4, (E, F, D), 4)
    w_down = tensor(5, (E, D, F), 4)
    cfg = moe.make_config(T=T, d_model=D, n_experts=E, top_k=K, d_ff=F)
    ws = moe.alloc_workspace(cfg)
    out = torch.empty(T, D, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    moe.moe_layer_forward(cfg, x, w_router, None, w_gate, w_up, w_down, out, ws, topk_idx_out=idx,
                          counts_out=counts)
    assert moe.moe_get_device_error(ws) == moe.MOE_OK
    assert (idx.cpu().numpy() == c_idx).all()
    assert (counts.cpu().numpy() == c_counts).all() and int(c_counts.sum()) == T * K
    assert (out.view(torch.int16).cpu().numpy().view(np.uint16) == c_out).all()
    assert np.isfinite(out.float().cpu().numpy()).all() and np.abs(out.float().cpu().numpy()).max() > 0
