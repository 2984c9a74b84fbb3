"""One rank of the data-parallel layer on the GPU (no process group: the
all-reduce is the identity): its outputs equal the single-GPU layer's, and
its FP32 dW rounds to the single-GPU BF16 dW bit for bit."""
import pytest
import torch

from fp8_precision_pretraining_amax_b300 import synth

pytestmark = pytest.mark.gpu


def test_dp_rank_matches_single_gpu_layer():
    from fp8_precision_pretraining_amax_b300 import fp8bq
    from fp8_precision_pretraining_amax_b300.dp import LinearFP8DP
    from fp8_precision_pretraining_amax_b300.linear import LinearFP8
    M, K, N = 512, 384, 640
    gen = synth.generator(50)
    x, w, dy = synth.activations(M, K, gen).cuda(), synth.weight(N, K, gen).cuda(), synth.grads(M, N, gen).cuda()
    ref = LinearFP8(M, K, N)
    y, dx, dw16 = ref.step(x, w, dy)
    dp = LinearFP8DP(M, K, N)
    y2, dx2, dw32 = dp.step(x, w, dy)
    fp8bq.check()
    assert torch.equal(y, y2) and torch.equal(dx, dx2)
    assert torch.equal(dw32.to(torch.bfloat16), dw16)
