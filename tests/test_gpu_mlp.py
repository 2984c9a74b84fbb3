"""The SwiGLU MLP forward with the gate fused into the quantizer equals the
unfused composition (gate/up Fprop, SwiGLU with H written out, row+column
quantization of that H, down Fprop) bit for bit."""
import pytest
import torch

from fp8_precision_pretraining_amax_b300 import synth

pytestmark = pytest.mark.gpu


def test_swiglu_mlp_matches_unfused_composition():
    from fp8_precision_pretraining_amax_b300 import fp8bq
    from fp8_precision_pretraining_amax_b300.linear import SwiGLUMLPFP8
    M, D, F = 512, 384, 640
    gen = synth.generator(81)
    x = synth.activations(M, D, gen).cuda()
    w_gu = synth.weight(2 * F, D, gen).cuda()
    w_d = synth.weight(D, F, gen).cuda()
    mlp = SwiGLUMLPFP8(M, D, F)
    out = mlp.forward(x, w_gu, w_d).clone()
    # unfused: same gate/up output, H materialised, then the separate quantizers
    gu = fp8bq.gemm_fprop(*fp8bq.quantize_rowwise(x), *fp8bq.quantize_weight_block(w_gu, transpose=False)[::2])
    h, _, _, _, _ = fp8bq.swiglu_quantize(gu, F, keep_h=True)
    hq, sh, hqT, shT = fp8bq.quantize_rowcol(h)
    wq, _, sw = fp8bq.quantize_weight_block(w_d)
    ref = fp8bq.gemm_fprop(hq, sh, wq, sw)
    fp8bq.check()
    assert torch.equal(out, ref)
    assert torch.equal(mlp.hqT, hqT) and torch.equal(mlp.shT, shT)
