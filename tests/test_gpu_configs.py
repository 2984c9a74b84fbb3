"""Parity of the whole layer step at the workloads' full sizes, in the launch
configuration the benchmark times.

Each test runs the product path on device-generated synthetic inputs
(LinearFP8: the weight-block quantizer, the row+column pass over X, Fprop,
the row+column pass over dY, Dgrad, Wgrad, every launch through the C ABI)
and has the oracle quantize the host copies of the same inputs.  On each GEMM
output it checks 64 tiles of 128 x 128 (a seeded 8 x 8 grid of random block
rows and block columns) plus the four corner tiles against the oracle's
binary64 product, with the acceptance bound |C - C_exact| <= 2e-3 *
sum_k |a_k b_k| + 1 BF16 ulp, and it checks the GPU's codes and scales bit
for bit on every operand block those tiles read.
"""
import numpy as np
import pytest
import torch

from fp8_precision_pretraining_amax_b300 import synth
from tests.helpers import OracleLinear, assert_codes_equal, assert_scales_equal, check_output_tile, grid_tiles

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _check_codes_rows(layer_q, layer_s, ref, b, what):
    """Row-wise codes q [R, C] and scales s [C/128, R] of row block b."""
    q, s = ref
    assert_codes_equal(layer_q[b * 128:(b + 1) * 128].cpu().numpy(), q, what)
    assert_scales_equal(layer_s[:, b * 128:(b + 1) * 128].cpu().numpy(), s, what + " scales")


def _check_codes_cols(layer_qT, layer_s, ref, b, what):
    """Column-wise codes qT [C, M] and scales s [M/128, C] of column block b."""
    qT, s = ref
    assert_codes_equal(layer_qT[b * 128:(b + 1) * 128].cpu().numpy(), qT, what)
    assert_scales_equal(layer_s[:, b * 128:(b + 1) * 128].cpu().numpy(), s, what + " scales")


def check_step(layer, lin, rng, gemms=("fprop", "dgrad", "wgrad")):
    """Check a LinearFP8 that has run step() (or forward()) on lin's inputs."""
    ref = OracleLinear(lin.x, lin.w, lin.dy)
    M, K, N = lin.M, lin.K, lin.N
    worst = {}
    if "fprop" in gemms:
        w = 0.0
        for bi, bj in grid_tiles(rng, M, N):
            _check_codes_rows(layer.xq, layer.sx, ref.x_rows(bi), bi, f"{lin.name} xq")
            wq, _, sw = ref.w_rows(bj)
            assert_codes_equal(layer.wq[bj * 128:(bj + 1) * 128].cpu().numpy(), wq, f"{lin.name} wq")
            assert_scales_equal(layer.sw[bj:bj + 1].cpu().numpy(), sw, f"{lin.name} sw")
            w = max(w, check_output_tile(layer.y, bi, bj, *ref.fprop(bi, bj), what=f"{lin.name} fprop"))
        worst["fprop"] = w
    if "dgrad" in gemms:
        w = 0.0
        for bi, bk in grid_tiles(rng, M, K):
            _check_codes_rows(layer.dyq, layer.sdy, ref.dy_rows(bi), bi, f"{lin.name} dyq")
            _, wqT, _ = ref.w_cols(bk)   # block column bk of W, transposed: rows bk of Wq^T
            assert_codes_equal(layer.wqT[bk * 128:(bk + 1) * 128].cpu().numpy(), wqT, f"{lin.name} wqT")
            w = max(w, check_output_tile(layer.dx, bi, bk, *ref.dgrad(bi, bk), what=f"{lin.name} dgrad"))
        worst["dgrad"] = w
    if "wgrad" in gemms:
        w = 0.0
        for bn, bk in grid_tiles(rng, N, K):
            _check_codes_cols(layer.dyqT, layer.sdyT, ref.dy_cols(bn), bn, f"{lin.name} dyqT")
            _check_codes_cols(layer.xqT, layer.sxT, ref.x_cols(bk), bk, f"{lin.name} xqT")
            w = max(w, check_output_tile(layer.dw, bn, bk, *ref.wgrad(bn, bk), what=f"{lin.name} wgrad"))
        worst["wgrad"] = w
    return worst


def test_layer_3p8b_full_step_parity():
    """3.8B-shaped layer at 32768 tokens (the benchmark's workload): all four
    linears (QKV 3072->4608, O 3072->3072, gate+up 3072->16384, down
    8192->3072), twelve GEMMs; Wgrad reduces over 256 chunks."""
    from fp8_precision_pretraining_amax_b300.linear import LinearFP8
    rng = np.random.default_rng(501)
    lins = synth.layer_3p8b("cuda")
    for lin in lins:
        layer = LinearFP8(lin.M, lin.K, lin.N)
        layer.step(lin.x, lin.w, lin.dy)
        torch.cuda.synchronize()
        from fp8_precision_pretraining_amax_b300 import fp8bq
        fp8bq.check()
        worst = check_step(layer, lin, rng)
        assert all(v <= 1.0 for v in worst.values()), worst
        del layer
        torch.cuda.empty_cache()


def test_up_proj_backward_full_step_parity():
    """Backward of the 2048 -> 6144 up-projection at 16384 tokens on the
    workload's own distributions (dY ~ N(0, 1e-3), activations with outlier
    channels): Dgrad reduces over 6144, Wgrad over 16384 tokens."""
    from fp8_precision_pretraining_amax_b300 import fp8bq
    from fp8_precision_pretraining_amax_b300.linear import LinearFP8
    rng = np.random.default_rng(502)
    lin = synth.up_bwd("cuda")
    layer = LinearFP8(lin.M, lin.K, lin.N)
    layer.step(lin.x, lin.w, lin.dy)
    fp8bq.check()
    worst = check_step(layer, lin, rng)
    assert all(v <= 1.0 for v in worst.values()), worst


def test_swiglu_mlp_fprop_full_size_parity():
    """SwiGLU MLP Fprop at 16384 tokens: gate+up 2048 -> 12288 and down
    6144 -> 2048, whose input is H = silu(g) * u of the generated gate/up
    (input generation in plain torch FP32)."""
    from fp8_precision_pretraining_amax_b300 import fp8bq
    from fp8_precision_pretraining_amax_b300.linear import LinearFP8
    rng = np.random.default_rng(503)
    for lin in synth.swiglu("cuda"):
        layer = LinearFP8(lin.M, lin.K, lin.N)
        layer.forward(lin.x, lin.w)
        fp8bq.check()
        worst = check_step(layer, lin, rng, gemms=("fprop",))
        assert worst["fprop"] <= 1.0, worst
        del layer
        torch.cuda.empty_cache()
