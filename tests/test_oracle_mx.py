"""Pins of the oracle's MX variant: a power-of-two scale 2^E per 1x32 block
along the reduction dimension (the block shape and 8-bit exponent scale of the
OCP Microscaling formats specification), E the smallest integer >= -127 with
amax <= 448 * 2^E (the layer's amax/448 scale rounded up to a power of two),
codes E4M3(x * 2^-E) with round-half-to-even.

What pins it, independently of the oracle's own code: a closed form of E from
the binary32 fields, a block quantized by hand (tests/golden), the range the
largest element must land in, the 2^-4 relative error bound, exponent
equivariance, the transposed layout, brute-force exact rationals and a float64
library matmul for the GEMM, and integer products that must come out exact.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from fp8_precision_pretraining_amax_b300 import synth
from tests.conftest import GOLDEN


def _exponent_closed_form(amax: np.ndarray) -> np.ndarray:
    """amax = f * 2^k with f in [1, 2): 448 = 1.75 * 2^8, so amax <= 448 * 2^E
    holds first at E = k - 8 when f <= 1.75 and at E = k - 7 otherwise."""
    a = np.asarray(amax, dtype=np.float32)
    bits = a.view(np.uint32)
    bexp = ((bits >> 23) & 0xFF).astype(np.int64)
    mant = (bits & 0x7FFFFF).astype(np.int64)
    k = bexp - 127
    e = k - 8 + (mant > 0x600000)
    e = np.where(bexp == 0, -127, e)          # zero and binary32 subnormals
    return np.maximum(e, -127)


def test_exponent_closed_form_on_random_and_boundary_values():
    rng = np.random.default_rng(11)
    vals = np.concatenate([
        (rng.standard_normal(4000) * np.exp2(rng.integers(-140, 120, 4000))).astype(np.float32),
        np.float32([0.0, 448.0, 224.0, 896.0, 1.0, 1.75, 2.0 ** -130, 2.0 ** -149, 3.0e38]),
        np.nextafter(np.float32([448.0, 224.0, 896.0, 1.75]), np.float32(np.inf)),
        np.nextafter(np.float32([448.0, 224.0, 896.0, 1.75]), np.float32(0)),
    ])
    vals = np.abs(vals)
    want = _exponent_closed_form(vals)
    got = np.array([oracle.mx_exponent(v) for v in vals])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(vals[i]), int(got[i]), int(want[i])) for i in bad[:5]]
    # the defining inequality, checked in binary64
    for v, e in zip(vals, got):
        if e > -127:
            assert float(v) <= 448.0 * 2.0 ** e and float(v) > 448.0 * 2.0 ** (e - 1)


def _load_worked_row():
    x = np.zeros(128, dtype=np.float32)
    codes = np.zeros(128, dtype=np.uint8)
    exps = {}
    for line in open(os.path.join(GOLDEN, "mx_block_worked.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        p = line.split()
        if p[0] == "block":
            exps[int(p[1])] = int(p[2])
            continue
        i = int(p[0])
        x[i] = np.float32(float(p[1]))
        codes[i] = int(p[3], 16)
    return x, codes, exps


def test_worked_block_fp32_and_bf16():
    x, codes, exps = _load_worked_row()
    xb = synth.bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    assert np.array_equal((xb.astype(np.uint32) << 16).view(np.float32), x), "fixture is BF16-exact"
    for inp in (x.reshape(1, 128), xb.reshape(1, 128)):
        q, e8 = oracle.mx_quantize_rowwise(inp)
        assert e8.shape == (1, 1, 4)
        assert [int(v) - 127 for v in e8[0, 0]] == [exps[b] for b in range(4)]
        bad = [(i, hex(a), hex(b)) for i, (a, b) in enumerate(zip(q[0], codes)) if a != b]
        assert not bad, bad
        # the same row as a column of a [128, 1] matrix, column-wise
        qT, e8T = oracle.mx_quantize_colwise(inp.reshape(128, 1))
        assert np.array_equal(qT[0], codes) and np.array_equal(e8T[0, 0], e8[0, 0])


def _check_blocks(x, q, e8):
    """x [R, C] float32, q [R, C], e8 [C/128, R, 4]: every MX block property."""
    R, C = x.shape
    E = (e8.astype(np.int64) - 127).transpose(1, 0, 2).reshape(R, C // 32)   # [R, blocks]
    xb = x.reshape(R, C // 32, 32).astype(np.float64)
    qb = q.reshape(R, C // 32, 32)
    amax = np.max(np.abs(xb), axis=2)
    assert np.array_equal(E, _exponent_closed_form(amax.astype(np.float32)))
    scaled = xb * np.exp2(-E)[..., None]
    assert np.all(np.abs(scaled) <= 448.0), "no element needs saturation"
    deq = oracle.e4m3_decode(qb) * np.exp2(E)[..., None]
    top = np.take_along_axis(oracle.e4m3_decode(qb), np.argmax(np.abs(xb), axis=2)[..., None], 2)[..., 0]
    unclamped = (amax > 0) & (E > -127)
    assert np.all((np.abs(top[unclamped]) >= 224.0) & (np.abs(top[unclamped]) <= 448.0))
    err = np.abs(deq - xb)
    normal = np.abs(scaled) >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(xb[normal]))
    sub_bound = np.broadcast_to(np.exp2(E)[..., None] * 2.0 ** -10, err.shape)
    assert np.all(err[~normal] <= sub_bound[~normal])
    assert np.all(((qb & 0x80) != 0) == np.signbit(xb))


def test_rowwise_properties_bf16_with_outliers_and_zero_blocks():
    gen = synth.generator(21)
    x = synth.activations(64, 512, gen)
    x[3, 64:96] = 0.0
    x[5, :] = 0.0
    xb = synth.bf16_bits(x)
    q, e8 = oracle.mx_quantize_rowwise(xb)
    assert e8[0, 3, 2] == 0 and e8[:, 5, :].max() == 0
    _check_blocks(x.float().numpy(), q, e8)


def test_rowwise_properties_fp32_wide_range():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((16, 256)) * np.exp2(rng.integers(-60, 60, (16, 1)))).astype(np.float32)
    q, e8 = oracle.mx_quantize_rowwise(x)
    _check_blocks(x, q, e8)


@pytest.mark.parametrize("j", [-20, -1, 1, 13])
def test_exponent_equivariance(j):
    gen = synth.generator(22)
    x = synth.activations(8, 256, gen).float().numpy()
    q0, e0 = oracle.mx_quantize_rowwise(x)
    q1, e1 = oracle.mx_quantize_rowwise((x * np.float32(2.0 ** j)).astype(np.float32))
    assert np.array_equal(q0, q1)
    assert np.array_equal(e1.astype(np.int64), e0.astype(np.int64) + j)


def test_colwise_equals_rowwise_of_transpose():
    gen = synth.generator(23)
    x = synth.grads(256, 96, gen)
    xb = synth.bf16_bits(x)
    qT, e8T = oracle.mx_quantize_colwise(xb)
    q, e8 = oracle.mx_quantize_rowwise(np.ascontiguousarray(xb.T))
    assert np.array_equal(qT, q) and np.array_equal(e8T, e8)


def _rand_codes(rng, shape, hi=0x7E):
    mag = rng.integers(0, hi + 1, size=shape).astype(np.uint8)
    return mag | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)


def _deq(codes, e8):
    """Dequantize K-major codes [R, K] with exponent bytes [K/128, R, 4]."""
    R, K = codes.shape
    E = (e8.astype(np.int64) - 127).transpose(1, 0, 2).reshape(R, K // 32)
    return oracle.e4m3_decode(codes) * np.repeat(np.exp2(E), 32, axis=1)


def test_gemm_exact_rational_brute_force_tiny():
    rng = np.random.default_rng(31)
    I, J, K = 3, 2, 256
    a = _rand_codes(rng, (I, K))
    b = _rand_codes(rng, (J, K))
    ea = rng.integers(100, 140, size=(K // 128, I, 4)).astype(np.uint8)
    eb = rng.integers(100, 140, size=(K // 128, J, 4)).astype(np.uint8)
    table = [Fraction(v) if np.isfinite(v) else None for v in oracle.e4m3_table()]
    val, absd = oracle.mx_gemm(a, ea, b, eb)
    for i in range(I):
        for j in range(J):
            tot = Fraction(0)
            tot_abs = Fraction(0)
            for k in range(K):
                c, t = k // 128, (k // 32) % 4
                p = (table[a[i, k]] * Fraction(2) ** (int(ea[c, i, t]) - 127)
                     * table[b[j, k]] * Fraction(2) ** (int(eb[c, j, t]) - 127))
                tot += p
                tot_abs += abs(p)
            assert abs(Fraction(val[i, j]) - tot) <= abs(tot_abs) * Fraction(2) ** -50
            assert abs(Fraction(absd[i, j]) - tot_abs) <= tot_abs * Fraction(2) ** -50


def test_gemm_matches_float64_matmul_and_transposes():
    rng = np.random.default_rng(32)
    I, J, K = 40, 24, 384
    a = _rand_codes(rng, (I, K))
    b = _rand_codes(rng, (J, K))
    ea = rng.integers(110, 135, size=(K // 128, I, 4)).astype(np.uint8)
    eb = rng.integers(110, 135, size=(K // 128, J, 4)).astype(np.uint8)
    val, absd = oracle.mx_gemm(a, ea, b, eb)
    da, db = _deq(a, ea), _deq(b, eb)
    ref = da @ db.T
    assert np.all(np.abs(val - ref) <= 1e-12 * (np.abs(da) @ np.abs(db).T))
    assert np.allclose(absd, np.abs(da) @ np.abs(db).T, rtol=1e-12, atol=0)
    valT, _ = oracle.mx_gemm(b, eb, a, ea)
    assert np.array_equal(valT.T, val)


def test_gemm_exact_integer_case():
    """Blocks whose amax is exactly 448 get E = 0, so codes equal the values;
    integer operands then give an integer product exactly."""
    rng = np.random.default_rng(33)
    I, J, K = 16, 8, 256
    ints = np.array([0, 1, 2, 3, 4, 5, 6, 7, 8, 10, 12, 16], dtype=np.float32)
    xa = rng.choice(ints, size=(I, K)) * rng.choice([-1, 1], size=(I, K))
    xb = rng.choice(ints, size=(J, K)) * rng.choice([-1, 1], size=(J, K))
    xa[:, ::32] = 448.0
    xb[:, ::32] = -448.0
    xa, xb = xa.astype(np.float32), xb.astype(np.float32)
    qa, ea = oracle.mx_quantize_rowwise(xa)
    qb, eb = oracle.mx_quantize_rowwise(xb)
    assert np.all(ea == 127) and np.all(eb == 127)
    val, _ = oracle.mx_gemm(qa, ea, qb, eb)
    assert np.array_equal(val, xa.astype(np.float64) @ xb.astype(np.float64).T)


def test_gemm_block_exponent_selection():
    """Raising one block's exponent by 3 multiplies exactly that block's
    contribution by 8: pins which 32 elements each exponent byte covers."""
    rng = np.random.default_rng(34)
    I, J, K = 4, 4, 256
    a = _rand_codes(rng, (I, K), hi=0x70)
    b = _rand_codes(rng, (J, K), hi=0x70)
    ea = np.full((K // 128, I, 4), 127, dtype=np.uint8)
    eb = np.full((K // 128, J, 4), 127, dtype=np.uint8)
    base, _ = oracle.mx_gemm(a, ea, b, eb)
    c, i, t = 1, 2, 3
    ea2 = ea.copy()
    ea2[c, i, t] += 3
    val, _ = oracle.mx_gemm(a, ea2, b, eb)
    ks = slice(128 * c + 32 * t, 128 * c + 32 * t + 32)
    block = oracle.e4m3_decode(a[i, ks]) @ oracle.e4m3_decode(b[:, ks]).T
    want = base.copy()
    want[i] += 7.0 * block
    assert np.allclose(val, want, rtol=0, atol=1e-12 * np.max(np.abs(want)))
    assert np.array_equal(np.delete(val, i, 0), np.delete(base, i, 0))


def test_accuracy_against_the_fp32_scale_layer_on_outlier_activations():
    """The comparison the MX variant exists for, on the oracle alone: an
    Fprop on Qwen3-1.7B-style operands (N(0,1) activations with 0.1 % outlier
    channels x50, N(0,0.02) weights), both quantized products against the
    exact binary64 product of the unquantized BF16 operands.  Every element of
    either quantizer is within 2^-4 of its input, so each relative error is
    well inside 2 * 2^-4; the measured values (about 3.0 % for the FP32-scale
    layer and 3.8 % for MX with these seeds) are reported, not tuned."""
    gen = synth.generator(1)
    M, N, K = 512, 256, 2048
    x = synth.activations(M, K, gen)
    w = synth.weight(N, K, gen)
    xb, wb = synth.bf16_bits(x), synth.bf16_bits(w)
    exact = x.double().numpy() @ w.double().numpy().T
    xq, sx = oracle.quantize_rowwise(xb)
    wq, _, sw = oracle.quantize_weight_block(wb)
    y_fp32_scale, _ = oracle.gemm_fprop(xq, sx, wq, sw)
    xm, ex = oracle.mx_quantize_rowwise(xb)
    wm, ew = oracle.mx_quantize_rowwise(wb)
    y_mx, _ = oracle.mx_gemm(xm, ex, wm, ew)
    rel = lambda y: float(np.linalg.norm(y - exact) / np.linalg.norm(exact))
    e_bs, e_mx = rel(y_fp32_scale), rel(y_mx)
    print(f"relative error: FP32-scale 1x128/128x128 {e_bs:.4f}, MX 1x32 power-of-two {e_mx:.4f}")
    assert 0 < e_bs < 2 * 2.0 ** -4 and 0 < e_mx < 2 * 2.0 ** -4


def test_accuracy_against_the_fp32_scale_layer_on_gradients():
    """The same comparison for a Dgrad-shaped product of N(0,1e-3) output
    gradients (no outliers) with N(0,0.02) weights: dX = dY W, dY row-wise
    along N, W column-wise (MX) or in 128x128 blocks (FP32-scale layer).
    Measured about 3.7 % (FP32-scale) and 3.8 % (MX) with these seeds."""
    gen = synth.generator(3)
    M, N, K = 512, 2048, 256
    dy = synth.grads(M, N, gen)
    w = synth.weight(N, K, gen)
    dyb, wb = synth.bf16_bits(dy), synth.bf16_bits(w)
    exact = dy.double().numpy() @ w.double().numpy()
    dyq, sdy = oracle.quantize_rowwise(dyb)
    wq, _, sw = oracle.quantize_weight_block(wb)
    dx_fp32_scale, _ = oracle.gemm_dgrad(dyq, sdy, wq, sw)
    dym, edy = oracle.mx_quantize_rowwise(dyb)
    wmT, ewT = oracle.mx_quantize_colwise(wb)
    dx_mx, _ = oracle.mx_gemm(dym, edy, wmT, ewT)
    rel = lambda y: float(np.linalg.norm(y - exact) / np.linalg.norm(exact))
    e_bs, e_mx = rel(dx_fp32_scale), rel(dx_mx)
    print(f"relative error (Dgrad): FP32-scale {e_bs:.4f}, MX {e_mx:.4f}")
    assert 0 < e_bs < 2 * 2.0 ** -4 and 0 < e_mx < 2 * 2.0 ** -4


def test_mx_and_fp32_scale_gemms_agree_when_every_scale_is_one():
    """With every MX exponent byte 127 (scale 1) and every FP32 scale 1 the two
    oracle GEMMs compute the same plain product of the codes: a cross-check of
    the two independently written reductions and of their operand layouts."""
    rng = np.random.default_rng(35)
    M, K = 24, 384
    x = _rand_codes(rng, (M, K))
    w = _rand_codes(rng, (256, K))
    ex = np.full((K // 128, M, 4), 127, dtype=np.uint8)
    ew = np.full((K // 128, 256, 4), 127, dtype=np.uint8)
    mx_val, mx_abs = oracle.mx_gemm(x, ex, w, ew)
    sx = np.ones((K // 128, M), dtype=np.float32)
    sw = np.ones((2, K // 128), dtype=np.float32)
    bs_val, bs_abs = oracle.gemm_fprop(x, sx, w, sw)
    assert np.allclose(mx_val, bs_val, rtol=0, atol=1e-12 * np.max(bs_abs))
    assert np.allclose(mx_abs, bs_abs, rtol=1e-15, atol=0)
