"""Pins of the oracle's SwiGLU gate h = silu(g) * u (binary64)."""
import numpy as np
import torch

import oracle
from fp8_precision_pretraining_amax_b300 import synth


def _bits(x):
    return synth.bf16_bits(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def test_swiglu_closed_forms():
    g = np.array([0.0, -0.0, 1.0, 2.0, -3.0, 40.0, -200.0], dtype=np.float32)
    u = np.array([5.0, -5.0, 1.0, 1.0, 2.0, 0.5, 7.0], dtype=np.float32)
    h = oracle.swiglu(_bits(g), _bits(u))
    assert h[0] == 0.0 and h[1] == 0.0
    assert abs(h[2] - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15        # silu(1) = sigmoid(1)
    assert abs(h[5] - 20.0) < 1e-12                               # silu(40) = 40 (to 1e-17)
    assert h[6] == 0.0                                            # silu(-200): FP32 exp overflow -> 0


def test_swiglu_fp32_exp_overflow_threshold():
    """exp(-g) is taken as +inf beyond the FP32 range: h = 0 for g = -89 but
    not for g = -88.5, where exp(88.5) = 2.7e38 is still finite."""
    g = np.array([-88.5, -89.0], dtype=np.float32)
    u = np.array([1.0, 1.0], dtype=np.float32)
    h = oracle.swiglu(_bits(g), _bits(u))
    assert h[1] == 0.0
    assert abs(h[0] - (-88.5) * np.exp(-88.5)) < 1e-50


def test_swiglu_odd_identity():
    """silu(g) - silu(-g) = g for every g (sigmoid(g) + sigmoid(-g) = 1)."""
    rng = np.random.default_rng(61)
    g = rng.normal(0, 4, 4096).astype(np.float32)
    ones = np.ones_like(g)
    gb = _bits(g)
    gn = gb ^ np.uint16(0x8000)
    a = oracle.swiglu(gb, _bits(ones))
    b = oracle.swiglu(gn, _bits(ones))
    gv = oracle.bf16_bits_to_f64(gb)
    assert np.max(np.abs((a - b) - gv) / np.maximum(np.abs(gv), 1e-30)) < 1e-14


def test_swiglu_matches_torch_silu_in_float64():
    rng = np.random.default_rng(62)
    g = rng.normal(0, 3, 10000).astype(np.float32)
    u = rng.normal(0, 1, 10000).astype(np.float32)
    gb, ub = _bits(g), _bits(u)
    gd = torch.from_numpy(oracle.bf16_bits_to_f64(gb))
    ud = torch.from_numpy(oracle.bf16_bits_to_f64(ub))
    want = (torch.nn.functional.silu(gd) * ud).numpy()
    got = oracle.swiglu(gb, ub)
    assert np.allclose(got, want, rtol=1e-14, atol=1e-300)


def test_swiglu_check_accepts_rounding_and_rejects_two_ulps():
    rng = np.random.default_rng(63)
    gb = _bits(rng.normal(0, 2, 2000).astype(np.float32))
    ub = _bits(rng.normal(0, 1, 2000).astype(np.float32))
    exact = oracle.swiglu(gb, ub)
    rounded = oracle.bf16_from_double(exact)
    ok, _ = oracle.swiglu_check(rounded, gb, ub)
    assert ok
    off = rounded.astype(np.int32)
    off[::7] += 2                                                 # two BF16 ulps away
    ok, _ = oracle.swiglu_check(off.astype(np.uint16), gb, ub)
    assert not ok
