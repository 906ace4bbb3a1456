"""The seeded input generator: host C == numpy restatement, sane moments, RNE bf16."""
import math

import numpy as np
import pytest
import torch

import synth


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("start", [0, 12345, (1 << 33) + 7])
def test_host_c_matches_numpy(dtype, start):
    a = synth.normal(0, 4, (4097,), 0.02, dtype, start=start)
    b = synth.normal_numpy(0, 4, start, 4097, 0.02, dtype)
    assert a.dtype == b.dtype and (a == b).all()


def test_streams_differ_and_repeat():
    a = synth.normal(0, 1, (1000,), 1.0, "f32")
    assert (a == synth.normal(0, 1, (1000,), 1.0, "f32")).all()
    assert (a != synth.normal(0, 2, (1000,), 1.0, "f32")).mean() > 0.99
    assert (a != synth.normal(1, 1, (1000,), 1.0, "f32")).mean() > 0.99


def test_slab_start_reproduces_whole_tensor():
    w = synth.WORKLOADS["mini_deepseek"]
    whole = synth.host_tensor(w, "w_down")
    for g in (0, 5, w.G - 1):
        _, _, wd = synth.host_expert(w, g)
        assert (wd == whole[g]).all()


def test_moments_and_support():
    v = synth.normal(0, 3, (1 << 20,), 1.0, "f32").astype(np.float64)
    assert abs(v.mean()) < 5.0 / math.sqrt(v.size)
    assert v.std() == pytest.approx(1.0, rel=3e-3)
    assert np.abs(v).max() <= math.sqrt(12.0) + 1e-6   # Irwin-Hall(4) support


def test_bf16_rounding_matches_torch():
    f = synth.normal(0, 5, (1 << 16,), 0.02, "f32")
    mine = synth.bf16_bits_from_f32(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (mine == ref).all()
    # the bf16 stream is the RNE rounding of the f32 stream
    assert (synth.normal(0, 5, (1 << 16,), 0.02, "bf16") == mine).all()


def test_router_bias_is_zipf():
    b = synth.router_bias(8, 1.0)
    w = np.exp(b.astype(np.float64))
    assert w / w[0] == pytest.approx([1.0 / (e + 1) for e in range(8)], rel=1e-6)
    assert synth.router_bias(8, 0.0) is None
