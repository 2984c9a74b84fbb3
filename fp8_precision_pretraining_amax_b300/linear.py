"""One nn.Linear on the block-scaled FP8 path: Fprop, Dgrad and Wgrad.

The Puro-2B report (section 2, "FP8") runs the matrix multiplications of the
main linear layers in FP8 with DeepSeek-V3-style fine-grained quantization and
keeps everything else in BF16/FP32.  For a layer with input X [M, K], weight
W [N, K] and output gradient dY [M, N] one training step does:

  forward    W -> 128x128 block codes (+ transposed)
             X -> row-wise 1x128 codes and column-wise 128x1 codes (one pass)
             Y  = Fprop(Xq, Wq)                                         [M, N]
  backward   dY -> row-wise and column-wise codes (one pass)
             dX = Dgrad(dYq, Wq^T)                                      [M, K]
             dW = Wgrad(dYq^T, Xq^T)                                    [N, K]

`LinearFP8` owns the code/scale buffers for one shape so that a step performs
no allocation; every call is a C-ABI launch on the current stream.
"""
from __future__ import annotations

import torch

from . import fp8bq


class LinearFP8:
    """Pre-allocated workspace for one linear layer of shape (M, K) -> N."""

    def __init__(self, M: int, K: int, N: int, device="cuda"):
        self.M, self.K, self.N = M, K, N
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        e = lambda *shape, dt: torch.empty(shape, dtype=dt, device=device)
        # forward
        self.xq, self.sx = e(M, K, dt=u8), e(K // 128, M, dt=f32)
        self.wq, self.wqT, self.sw = e(N, K, dt=u8), e(K, N, dt=u8), e(N // 128, K // 128, dt=f32)
        # backward
        self.dyq, self.sdy = e(M, N, dt=u8), e(N // 128, M, dt=f32)
        self.dyqT, self.sdyT = e(N, M, dt=u8), e(M // 128, N, dt=f32)
        self.xqT, self.sxT = e(K, M, dt=u8), e(M // 128, K, dt=f32)
        self.y, self.dx, self.dw = e(M, N, dt=bf), e(M, K, dt=bf), e(N, K, dt=bf)
        self._wscratch = None

    @property
    def wscratch(self) -> torch.Tensor:
        """This layer's scratch for the balanced Wgrad (zeroed once, left zero by every call)."""
        if self._wscratch is None:
            self._wscratch = fp8bq.wgrad_scratch(self.dw.device)
        return self._wscratch

    @property
    def flops_per_gemm(self) -> int:
        return 2 * self.M * self.N * self.K

    def forward(self, x: torch.Tensor, w: torch.Tensor, for_backward: bool = True) -> torch.Tensor:
        """Quantize W (both layouts) and X, then Fprop.  With for_backward the
        column-wise codes of X that Wgrad needs come out of the same pass over X."""
        fp8bq.fp8bq_quantize_weight_block(w, self.wq, self.wqT, self.sw)
        if for_backward:
            fp8bq.fp8bq_quantize_rowcol(x, self.xq, self.sx, self.xqT, self.sxT)
        else:
            fp8bq.fp8bq_quantize_rowwise(x, self.xq, self.sx)
        fp8bq.fp8bq_gemm_fprop(self.xq, self.sx, self.wq, self.sw, self.y)
        return self.y

    def backward(self, dy: torch.Tensor):
        """Needs forward(for_backward=True) first (wqT, sw, xqT, sxT are reused)."""
        fp8bq.fp8bq_quantize_rowcol(dy, self.dyq, self.sdy, self.dyqT, self.sdyT)
        fp8bq.fp8bq_gemm_dgrad(self.dyq, self.sdy, self.wqT, self.sw, self.dx)
        fp8bq.fp8bq_gemm_wgrad_balanced(self.dyqT, self.sdyT, self.xqT, self.sxT, self.dw, self.wscratch)
        return self.dx, self.dw

    def step(self, x: torch.Tensor, w: torch.Tensor, dy: torch.Tensor):
        """Fprop + Dgrad + Wgrad: 3 GEMMs and 3 quantizer launches (weight block,
        row+column pass over X, row+column pass over dY)."""
        self.forward(x, w)
        self.backward(dy)
        return self.y, self.dx, self.dw

    LAUNCHES_PER_STEP = 6


class LinearMX:
    """The same linear layer on the MX variant: E4M3 codes with one
    power-of-two scale per 1x32 block along each GEMM's reduction dimension,
    applied by the tensor cores inside the MMA.  Every operand is quantized
    along the dimension its GEMM reduces over, so X, W and dY each need both
    layouts; one pass over each tensor produces them.

      forward    W -> row-wise (Fprop) and column-wise (Dgrad) codes, one pass
                 X -> row-wise (Fprop) and column-wise (Wgrad) codes, one pass
                 Y  = MX GEMM(Xq, Wq)                                   [M, N]
      backward   dY -> row-wise (Dgrad) and column-wise (Wgrad) codes, one pass
                 dX = MX GEMM(dYq, Wq^T)                                [M, K]
                 dW = MX GEMM(dYq^T, Xq^T)                              [N, K]
    """

    def __init__(self, M: int, K: int, N: int, device="cuda"):
        self.M, self.K, self.N = M, K, N
        u8, bf = torch.uint8, torch.bfloat16
        e = lambda *shape, dt=u8: torch.empty(shape, dtype=dt, device=device)
        self.xq, self.ex = e(M, K), e(K // 128, M, 4)
        self.xqT, self.exT = e(K, M), e(M // 128, K, 4)
        self.wq, self.ew = e(N, K), e(K // 128, N, 4)
        self.wqT, self.ewT = e(K, N), e(N // 128, K, 4)
        self.dyq, self.edy = e(M, N), e(N // 128, M, 4)
        self.dyqT, self.edyT = e(N, M), e(M // 128, N, 4)
        self.y, self.dx, self.dw = e(M, N, dt=bf), e(M, K, dt=bf), e(N, K, dt=bf)

    @property
    def flops_per_gemm(self) -> int:
        return 2 * self.M * self.N * self.K

    def forward(self, x: torch.Tensor, w: torch.Tensor) -> torch.Tensor:
        fp8bq.fp8bq_mx_quantize_rowcol(w, self.wq, self.ew, self.wqT, self.ewT)
        fp8bq.fp8bq_mx_quantize_rowcol(x, self.xq, self.ex, self.xqT, self.exT)
        fp8bq.fp8bq_mx_gemm(self.xq, self.ex, self.wq, self.ew, self.y)
        return self.y

    def backward(self, dy: torch.Tensor):
        fp8bq.fp8bq_mx_quantize_rowcol(dy, self.dyq, self.edy, self.dyqT, self.edyT)
        fp8bq.fp8bq_mx_gemm(self.dyq, self.edy, self.wqT, self.ewT, self.dx)
        fp8bq.fp8bq_mx_gemm(self.dyqT, self.edyT, self.xqT, self.exT, self.dw)
        return self.dx, self.dw

    def step(self, x: torch.Tensor, w: torch.Tensor, dy: torch.Tensor):
        self.forward(x, w)
        self.backward(dy)
        return self.y, self.dx, self.dw

    LAUNCHES_PER_STEP = 6


class SwiGLUMLPFP8:
    """Forward of a SwiGLU MLP (x -> gate/up -> silu(g) * u -> down) on the FP8
    path, with the SwiGLU gate fused into the down projection's quantizer.

    The gate/up projection writes g and u side by side ([M, 2F] BF16); one
    pass over them forms H = silu(g) * u and emits the down projection's
    row-wise codes (for its Fprop) and column-wise codes (kept for its Wgrad),
    so H itself is never written or re-read."""

    def __init__(self, M: int, D: int, F: int, device="cuda"):
        self.M, self.D, self.F = M, D, F
        u8, f32, bf = torch.uint8, torch.float32, torch.bfloat16
        e = lambda *shape, dt: torch.empty(shape, dtype=dt, device=device)
        self.gate_up = LinearFP8(M, D, 2 * F, device=device)
        self.hq, self.sh = e(M, F, dt=u8), e(F // 128, M, dt=f32)
        self.hqT, self.shT = e(F, M, dt=u8), e(M // 128, F, dt=f32)
        self.wdq, self.wdqT, self.swd = e(D, F, dt=u8), e(F, D, dt=u8), e(D // 128, F // 128, dt=f32)
        self.out = e(M, D, dt=bf)

    def forward(self, x: torch.Tensor, w_gate_up: torch.Tensor, w_down: torch.Tensor) -> torch.Tensor:
        """x [M, D], w_gate_up [2F, D] (gate rows first), w_down [D, F] -> [M, D]."""
        gu = self.gate_up.forward(x, w_gate_up)
        fp8bq.fp8bq_swiglu_quantize(gu, None, self.hq, self.sh, self.hqT, self.shT)
        fp8bq.fp8bq_quantize_weight_block(w_down, self.wdq, self.wdqT, self.swd)
        fp8bq.fp8bq_gemm_fprop(self.hq, self.sh, self.wdq, self.swd, self.out)
        return self.out
