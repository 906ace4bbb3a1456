"""Workload shapes and input recipes for the MoE FFN layer.

The five full-size workloads are synthetic stand-ins for the model shapes the
source pages cite ("Mixtral 8x7B contains eight feed-forward experts ... routes
every token to two of them": techbonafide.com, "How Does Routing Work in an MoE
Layer?"; DeepSeek-V3 and Qwen3-30B-A3B with 128-256 fine-grained experts, top-8,
and shared experts: shubhamtatvamasi.com "Mixture of Experts", sections "The
router" and the introduction). No dataset or trained weight is involved: every
tensor is drawn from the generator in this package with seed 0.

The ``mini_*`` workloads keep each family's structure (score function,
capacity policy, shared expert, skew) at sizes the fp64 oracle finishes in
seconds while still spanning several GEMM tiles with ragged tails.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict, replace

# stream ids of the generated tensors
TENSOR_ID = {"x": 1, "w_router": 2, "w_gate": 3, "w_up": 4, "w_down": 5}


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens in the batch
    d_model: int
    n_experts: int         # routed experts E
    top_k: int
    d_ff: int              # expert hidden width F (shared expert uses the same F)
    n_shared: int = 0      # always-on shared experts S (0 or 1)
    score: str = "softmax"  # "softmax" | "sigmoid"
    renormalize: bool = True
    capacity_factor: float = 0.0   # <= 0: dropless
    bias_s: float = 0.0    # Zipf exponent of the synthetic router bias; 0: no bias
    x_sigma: float = 1.0
    w_sigma: float = 0.02
    dtype: str = "bf16"    # "bf16" | "f32"
    seed: int = 0
    description: str = ""

    @property
    def G(self) -> int:
        return self.n_experts + self.n_shared

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def as_dict(self) -> dict:
        return asdict(self)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_f32", T=64, d_model=64, n_experts=8, top_k=2, d_ff=128, x_sigma=0.02, dtype="f32",
                 description="tiny fp32 layer, softmax top-2 renormalised, dropless"),
        Workload("mixtral_8x7b", T=4096, d_model=4096, n_experts=8, top_k=2, d_ff=14336, bias_s=1.0,
                 description="Mixtral-8x7B-shaped prefill, softmax top-2, dropless, Zipf(1.0) expert loads"),
        Workload("qwen3_30b_a3b", T=8192, d_model=2048, n_experts=128, top_k=8, d_ff=768,
                 description="Qwen3-30B-A3B-shaped fine-grained layer, softmax top-8, dropless"),
        Workload("deepseek_v3", T=4096, d_model=7168, n_experts=256, top_k=8, d_ff=2048, n_shared=1,
                 score="sigmoid", capacity_factor=1.25, bias_s=1.2,
                 description="DeepSeek-V3-shaped layer, 256 routed + 1 shared, sigmoid top-8, capacity 1.25, Zipf(1.2)"),
        Workload("decode_qwen3", T=32, d_model=2048, n_experts=128, top_k=8, d_ff=768,
                 description="decode-shaped batch of 32 tokens on the Qwen3-shaped layer"),
        # beyond the five: decode on the DeepSeek-V3-shaped layer (dropless, as decode runs)
        Workload("decode_deepseek", T=32, d_model=7168, n_experts=256, top_k=8, d_ff=2048, n_shared=1,
                 score="sigmoid", bias_s=1.2,
                 description="decode-shaped batch of 32 tokens on the DeepSeek-V3-shaped layer, dropless"),
        # reduced sizes for full element-by-element parity against the oracle
        Workload("mini_mixtral", T=300, d_model=256, n_experts=8, top_k=2, d_ff=384, bias_s=1.0),
        Workload("mini_qwen3", T=333, d_model=512, n_experts=32, top_k=8, d_ff=256),
        Workload("mini_deepseek", T=257, d_model=512, n_experts=48, top_k=6, d_ff=256, n_shared=1,
                 score="sigmoid", capacity_factor=1.25, bias_s=1.2),
        Workload("mini_decode", T=5, d_model=256, n_experts=64, top_k=8, d_ff=128),
        # Mixtral-shaped tiles on two experts (0.7 GB of weights): small enough for a
        # many-pass profiler capture, still far larger than L2
        Workload("prof_mixtral_e2", T=2048, d_model=4096, n_experts=2, top_k=2, d_ff=14336),
    ]
}

FULL = ["tiny_f32", "mixtral_8x7b", "qwen3_30b_a3b", "deepseek_v3", "decode_qwen3"]
FULL_EXTRA = ["decode_deepseek"]          # full-size parity cases beyond the five benchmarked layers
MINI = ["tiny_f32", "mini_mixtral", "mini_qwen3", "mini_deepseek", "mini_decode"]
