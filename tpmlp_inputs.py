"""Seeded synthetic inputs for the tensor-parallel MLP workloads.

This module only draws random tensors of the right shapes, distributions and
dtypes. It contains none of the MLP's arithmetic, so that both the CUDA path
(through the tests and the benchmark) and the float64 oracle can be fed the
very same values without sharing any code beyond this.

Workloads (T tokens, hidden D, MLP width F, N shards; the MLP is
Y = GeLU(X A) B with A of shape (D, F) and B of shape (F, D), as set out on
scratchllm.com "Tensor-Parallel MLP (Megatron)", section "The problem"):

  tiny_fp32   T=64,    D=64,   F=256,   N=4  fp32   X~N(0,1), A~N(0,1/sqrt(D)), B~N(0,1/sqrt(F))
  gpt2_small  T=4096,  D=768,  F=3072,  N=4  bf16   X~N(0,1), A,B~N(0,0.02)
  seq128      T=1024,  D=1024, F=4096,  N=4  bf16   (batch 8 x seq 128)
  seq256      T=2048,  D=1024, F=4096,  N=4  bf16   (batch 8 x seq 256)
  seq512      T=4096,  D=1024, F=4096,  N=4  bf16   (batch 8 x seq 512)
  large       T=16384, D=4096, F=16384, N=8  bf16   X~N(0,1), A,B~N(0,0.02)
  fwd_bwd     T=8192,  D=8192, F=32768, N=8  bf16   X~N(0,1), A,B~N(0,0.01), dY~N(0,1)

Attention workloads (ATTN_WORKLOADS: batch x seq tokens, D, heads, N ranks;
duoan.github.io "Tensor Parallelism in Megatron-LM" §4): attn_tiny_fp32
(2 x 16, D=64, 4 heads, N=2, W~N(0,1/8)) and attn_seq{128,256,512} (8 x seq,
D=1024, 16 heads of 64, N=4, bf16, X~N(0,1), W~N(0,0.02)), and
attn_long{1024,2048,4096} (4096 tokens as 4 x 1024, 2 x 2048, 1 x 4096,
otherwise the same); X uses seed+0,
Wq..Wo seeds +1..+4.

"N(0, s)" means a normal with standard deviation s. Each tensor gets its own
CPU torch.Generator: X uses seed+0, A seed+1, B seed+2, dY seed+3. Values are
drawn in float32, scaled, then rounded once to the workload's dtype; the
rounded tensors are what both sides receive (the oracle widens them exactly
to float64).
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    D: int
    F: int
    N: int
    dtype: str          # "f32" or "bf16": storage type of X, A, B, dY
    x_std: float
    a_std: float
    b_std: float
    dy_std: float = 1.0
    backward: bool = False

    @property
    def Fs(self) -> int:
        return self.F // self.N

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def fwd_flops(self) -> int:
        """4*T*D*F: two GEMMs of 2*T*D*F each."""
        return 4 * self.T * self.D * self.F

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_fp32", 64, 64, 256, 4, "f32", 1.0, 1.0 / math.sqrt(64), 1.0 / math.sqrt(256)),
        Workload("gpt2_small", 4096, 768, 3072, 4, "bf16", 1.0, 0.02, 0.02),
        Workload("seq128", 8 * 128, 1024, 4096, 4, "bf16", 1.0, 0.02, 0.02),
        Workload("seq256", 8 * 256, 1024, 4096, 4, "bf16", 1.0, 0.02, 0.02),
        Workload("seq512", 8 * 512, 1024, 4096, 4, "bf16", 1.0, 0.02, 0.02),
        Workload("large", 8 * 2048, 4096, 16384, 8, "bf16", 1.0, 0.02, 0.02),
        Workload("fwd_bwd", 8192, 8192, 32768, 8, "bf16", 1.0, 0.01, 0.01, 1.0, True),
    ]
}


def _draw(shape, std: float, seed: int, dtype: torch.dtype) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def make_inputs(w: Workload, seed: int = 0, with_dy: bool | None = None) -> dict[str, torch.Tensor]:
    """Return CPU tensors X [T,D], A [D,F], B [F,D] (and dY [T,D]) in w's dtype."""
    dt = w.torch_dtype
    out = {
        "X": _draw((w.T, w.D), w.x_std, seed + 0, dt),
        "A": _draw((w.D, w.F), w.a_std, seed + 1, dt),
        "B": _draw((w.F, w.D), w.b_std, seed + 2, dt),
    }
    if with_dy if with_dy is not None else w.backward:
        out["dY"] = _draw((w.T, w.D), w.dy_std, seed + 3, dt)
    return out


def make_block_inputs(w: Workload, seed: int = 0, with_dout: bool | None = None) -> dict[str, torch.Tensor]:
    """Inputs of the block's FFN half: the residual stream x [T, D] plus A, B (and dout [T, D]).

    Each row of x is offset and scaled on its own (offset uniform in [-1, 1],
    scale log-uniform in [0.5, 2]) so that the layer norm's centring and
    scaling both matter; A, B and dout are drawn as in make_inputs.
    """
    inp = make_inputs(w, seed, with_dy=with_dout)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 4)
    offset = torch.rand((w.T, 1), generator=g, dtype=torch.float32) * 2.0 - 1.0
    scale = torch.exp((torch.rand((w.T, 1), generator=g, dtype=torch.float32) * 2.0 - 1.0) * math.log(2.0))
    x = (inp.pop("X").to(torch.float32) * scale + offset).to(w.torch_dtype)
    out = {"x": x, "A": inp["A"], "B": inp["B"]}
    if "dY" in inp:
        out["dout"] = inp["dY"]
    return out


@dataclass(frozen=True)
class AttnWorkload:
    """Head-split attention: X [batch*seq, D], Wq, Wk, Wv, Wo [D, D], `heads`
    heads of D/heads, N ranks (heads divisible by N)."""

    name: str
    batch: int
    seq: int
    D: int
    heads: int
    N: int
    dtype: str  # "f32" or "bf16"
    x_std: float
    w_std: float

    @property
    def T(self) -> int:
        return self.batch * self.seq

    @property
    def dh(self) -> int:
        return self.D // self.heads

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def fwd_flops(self) -> float:
        """QKV projection 6 T D^2, scores and weighted values 4 batch seq^2 D, output projection 2 T D^2."""
        return 8.0 * self.T * self.D * self.D + 4.0 * self.batch * self.seq * self.seq * self.D


# The attention counterpart of the sequence sweep: batch 8, D=1024 with
# GPT-2's head size of 64 (16 heads), 4 ranks; and a tiny fp32 case.
ATTN_WORKLOADS: dict[str, AttnWorkload] = {
    "attn_tiny_fp32": AttnWorkload("attn_tiny_fp32", 2, 16, 64, 4, 2, "f32", 1.0, 0.125),
    "attn_seq128": AttnWorkload("attn_seq128", 8, 128, 1024, 16, 4, "bf16", 1.0, 0.02),
    "attn_seq256": AttnWorkload("attn_seq256", 8, 256, 1024, 16, 4, "bf16", 1.0, 0.02),
    "attn_seq512": AttnWorkload("attn_seq512", 8, 512, 1024, 16, 4, "bf16", 1.0, 0.02),
    # Longer sequences at the same 4096 tokens: the attention core grows with seq.
    "attn_long1024": AttnWorkload("attn_long1024", 4, 1024, 1024, 16, 4, "bf16", 1.0, 0.02),
    "attn_long2048": AttnWorkload("attn_long2048", 2, 2048, 1024, 16, 4, "bf16", 1.0, 0.02),
    "attn_long4096": AttnWorkload("attn_long4096", 1, 4096, 1024, 16, 4, "bf16", 1.0, 0.02),
}


def make_attn_inputs(w: AttnWorkload, seed: int = 0) -> dict[str, torch.Tensor]:
    """X [T, D] (seed+0) and Wq, Wk, Wv, Wo [D, D] (seeds +1..+4) in w's dtype."""
    dt = w.torch_dtype
    out = {"X": _draw((w.T, w.D), w.x_std, seed, dt)}
    for k, name in enumerate(("Wq", "Wk", "Wv", "Wo")):
        out[name] = _draw((w.D, w.D), w.w_std, seed + 1 + k, dt)
    return out


def sample_indices(n: int, k: int, seed: int) -> list[int]:
    """k distinct sorted indices in [0, n), always including the first and last."""
    if k >= n:
        return list(range(n))
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    idx = set(torch.randperm(n, generator=g)[: max(k - 2, 0)].tolist())
    idx.update({0, n - 1})
    return sorted(idx)
