"""Seeded synthetic inputs for the block-scaled FP8 linear layer.

This module is shared by the tests, the oracle checks and the benchmark.  It
holds none of the layer's arithmetic (no quantization, no scaling, no GEMM of
the method): it only draws Gaussian tensors and builds the shapes the layer is
exercised on.  Every tensor is drawn in FP32 from a seeded ``torch.Generator``
and rounded to BF16 with round-half-to-even (torch's cast).

Workloads (model shapes from the Puro-2B report, which trains Qwen3-1.7B-class
models, and from the 3.8B LLaMA-style model of the n1n.ai "$998 3.8B" article,
"model architecture" table: hidden 3072, 32 attention heads with 8 KV heads):

  tiny      A fp32 256x512 ~N(0,1), B fp32 512x384 ~N(0,0.02), seed 0;
            the weight is W = B^T [384, 512]
  qkv_1p7b  Qwen3-1.7B QKV Fprop: X 8192x2048, W 4096x2048 (16 q + 8 kv heads
            x 128), seed 1
  swiglu    gate+up X 16384x2048 -> 12288, then down 6144 -> 2048 on
            H = silu(g) * u, seed 2
  up_bwd    backward of the 2048 -> 6144 up-projection, 16384 tokens:
            dY 16384x6144 ~N(0,1e-3), X 16384x2048, W 6144x2048, seed 3
  layer_3p8b  one 3.8B-shaped transformer layer at 32768 tokens: QKV
            3072 -> 4608 (32 q + 8 kv heads x 96), O 3072 -> 3072, gate+up
            3072 -> 16384, down 8192 -> 3072; Fprop, Dgrad and Wgrad each, seed 4

Distributions: activations ~N(0,1) with 0.1% outlier input channels
(max(1, round(0.001 K)) columns picked by a seeded permutation, multiplied by
50 in FP32 before the BF16 cast, on every token); weights ~N(0,0.02);
gradients ~N(0,1e-3).  The second parameter of N(., .) is the standard
deviation.  The down-projection input is H = silu(g) * u where g and u are the
gate and up outputs of the generated X and W computed with a plain torch
matmul in FP32 (this is input generation, not the layer under test).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import torch

ACT_STD = 1.0
WEIGHT_STD = 0.02
GRAD_STD = 1e-3
OUTLIER_FRACTION = 0.001
OUTLIER_GAIN = 50.0


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def gaussian(shape, std: float, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """FP32 N(0, std) draw."""
    t = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t


def outlier_channels(K: int, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """Indices of the outlier input channels: max(1, round(0.001 K)) of them."""
    n = max(1, int(round(OUTLIER_FRACTION * K)))
    perm = torch.randperm(K, generator=gen, device=device)
    return perm[:n]


def activations(M: int, K: int, gen: torch.Generator, device="cpu", outliers: bool = True) -> torch.Tensor:
    """BF16 [M, K] activations ~N(0,1) with 0.1% outlier channels x50."""
    x = gaussian((M, K), ACT_STD, gen, device)
    if outliers:
        idx = outlier_channels(K, gen, device)
        x[:, idx] *= OUTLIER_GAIN
    return x.to(torch.bfloat16)


def weight(N: int, K: int, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """BF16 [N, K] weight (nn.Linear layout) ~N(0,0.02)."""
    return gaussian((N, K), WEIGHT_STD, gen, device).to(torch.bfloat16)


def grads(M: int, N: int, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """BF16 [M, N] output gradient ~N(0,1e-3)."""
    return gaussian((M, N), GRAD_STD, gen, device).to(torch.bfloat16)


def swiglu_input(x: torch.Tensor, w_gate: torch.Tensor, w_up: torch.Tensor) -> torch.Tensor:
    """H = silu(g) * u with g = x w_gate^T, u = x w_up^T in FP32, rounded to BF16.
    Plain torch arithmetic: it only shapes the input distribution of the
    down-projection."""
    xf = x.float()
    g = xf @ w_gate.float().t()
    u = xf @ w_up.float().t()
    return (torch.nn.functional.silu(g) * u).to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Named workloads
# ---------------------------------------------------------------------------

@dataclasses.dataclass
class Linear:
    """One linear layer's operands: X [M, K], W [N, K], dY [M, N] (any may be None)."""
    name: str
    M: int
    K: int
    N: int
    x: torch.Tensor = None
    w: torch.Tensor = None
    dy: torch.Tensor = None

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


def tiny(device="cpu") -> Linear:
    """256x512 @ 512x384, FP32 operands, seed 0.  W = B^T."""
    gen = generator(0, "cpu")
    a = gaussian((256, 512), ACT_STD, gen)
    b = gaussian((512, 384), WEIGHT_STD, gen)
    return Linear("tiny", 256, 512, 384, x=a.to(device), w=b.t().contiguous().to(device))


def qkv_1p7b(device="cpu", M: int = 8192) -> Linear:
    gen = generator(1, device)
    x = activations(M, 2048, gen, device)
    w = weight(4096, 2048, gen, device)
    return Linear("qkv_1p7b", M, 2048, 4096, x=x, w=w)


def swiglu(device="cpu", M: int = 16384) -> Tuple[Linear, Linear]:
    """Gate+up (2048 -> 12288, gate rows first) and down (6144 -> 2048)."""
    gen = generator(2, device)
    x = activations(M, 2048, gen, device)
    w_gu = weight(12288, 2048, gen, device)
    w_down = weight(2048, 6144, gen, device)
    h = swiglu_input(x, w_gu[:6144], w_gu[6144:])
    return (Linear("gate_up", M, 2048, 12288, x=x, w=w_gu),
            Linear("down", M, 6144, 2048, x=h, w=w_down))


def up_bwd(device="cpu", M: int = 16384) -> Linear:
    gen = generator(3, device)
    dy = grads(M, 6144, gen, device)
    x = activations(M, 2048, gen, device)
    w = weight(6144, 2048, gen, device)
    return Linear("up_bwd", M, 2048, 6144, x=x, w=w, dy=dy)


LAYER_3P8B: List[Tuple[str, int, int]] = [
    ("qkv", 3072, 4608),       # 32 q heads x 96 + 2 x 8 kv heads x 96
    ("o", 3072, 3072),
    ("gate_up", 3072, 16384),  # gate 8192 rows, then up 8192 rows
    ("down", 8192, 3072),
]


def layer_3p8b(device="cpu", M: int = 32768) -> List[Linear]:
    """All four linears of one 3.8B-shaped layer with X, W and dY each."""
    gen = generator(4, device)
    out: Dict[str, Linear] = {}
    for name, K, N in LAYER_3P8B:
        w = weight(N, K, gen, device)
        if name == "down":
            gu = out["gate_up"]
            x = swiglu_input(gu.x, gu.w[:8192], gu.w[8192:])
        else:
            x = activations(M, K, gen, device)
        dy = grads(M, N, gen, device)
        out[name] = Linear(name, M, K, N, x=x, w=w, dy=dy)
    return [out[n] for n, _, _ in LAYER_3P8B]


def bf16_bits(t: torch.Tensor):
    """Host numpy view of a BF16 tensor's 16-bit patterns (for the oracle)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
