"""fp8bq_gemm_wgrad_balanced_static: the balanced Wgrad with the library's
own device-memory scratch instead of a caller buffer.  On a shape whose
tiles are split between clusters, two calls of it and two calls of
fp8bq_gemm_wgrad_balanced (with a zeroed caller buffer) give the same bits,
and the result is within the oracle's bound."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import check_gemm_tiles, random_codes, random_scales, to_dev

pytestmark = pytest.mark.gpu


def test_static_scratch_wgrad_matches_the_caller_scratch_entry_point():
    from fp8_precision_pretraining_amax_b300 import fp8bq
    rng = np.random.default_rng(37)
    M, N, K = 2048, 2304, 2304           # 81 output tiles of 256 x 256, 16 chunks each
    dyqT, xqT = random_codes(rng, (N, M)), random_codes(rng, (K, M))
    sdyT, sxT = random_scales(rng, (M // 128, N)), random_scales(rng, (M // 128, K))
    dev = [to_dev(a) for a in (dyqT, sdyT, xqT, sxT)]
    scratch = fp8bq.wgrad_scratch(dev[0].device)
    outs = []
    for _ in range(2):
        for static in (True, False):
            dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
            if static:
                fp8bq.fp8bq_gemm_wgrad_balanced_static(*dev, dw)
            else:
                fp8bq.fp8bq_gemm_wgrad_balanced(*dev, dw, scratch)
            outs.append(dw)
    fp8bq.check()
    torch.cuda.synchronize()
    for dw in outs[1:]:
        assert torch.equal(dw.view(torch.int16), outs[0].view(torch.int16))
    rows = sorted({(0, 0), (5, 11), (17, 17), (9, 3)})
    check_gemm_tiles(outs[0], oracle.gemm_wgrad_mm, (dyqT, sdyT, xqT, sxT), rows, what="wgrad static scratch")
