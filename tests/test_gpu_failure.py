"""Device-side failure detection without a GPU fault: a kernel waits on a
barrier that nothing completes, gives up after a short limit, and the host
reads FP8BQ_ERR_TIMEOUT from the status word; the context stays usable."""
import pytest
import torch

from fp8_precision_pretraining_amax_b300 import synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    from fp8_precision_pretraining_amax_b300 import fp8bq as fb
    fb.check()                                   # clean slate
    fb.selftest_wait_timeout(20_000_000)         # 20 ms
    with pytest.raises(fb.Fp8bqError) as e:
        fb.check()
    assert e.value.status == fb.ERR_TIMEOUT
    fb.check()                                   # the status word was cleared
    x = synth.activations(128, 256, synth.generator(1)).cuda()
    q, s = fb.quantize_rowwise(x)
    fb.check()
    torch.cuda.synchronize()
    assert q.shape == (128, 256)
