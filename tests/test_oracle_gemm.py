"""Pins of the oracle's block-scaled GEMMs (Fprop, Dgrad, Wgrad).

Each GEMM sums, over 128-wide reduction chunks, the chunk's exact FP8 dot
product times the product of the two operands' scales for that chunk.  In
exact arithmetic that equals the plain matmul of the dequantized operands,
which is what these tests compare against (exact rationals on tiny shapes, a
float64 library matmul on larger ones, integer matmul on exact cases).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from fp8_precision_pretraining_amax_b300 import synth


def _rand_codes(rng, shape, lo=0, hi=0x7E):
    mag = rng.integers(lo, hi + 1, size=shape).astype(np.uint8)
    sign = (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)
    return mag | sign


def _pow2_scales(rng, shape, lo=-6, hi=4):
    return np.exp2(rng.integers(lo, hi + 1, size=shape)).astype(np.float32)


def _rand_scales(rng, shape):
    return (rng.uniform(0.5, 2.0, size=shape) * np.exp2(rng.integers(-8, 3, size=shape))).astype(np.float32)


def _deq_rows(codes, s_chunk_major):
    """Dequantize row-tile codes [R, C] with scales [C/128, R]."""
    R, C = codes.shape
    s = np.repeat(s_chunk_major.T.astype(np.float64), 128, axis=1)  # [R, C]
    return oracle.e4m3_decode(codes) * s


def _deq_blocks(codes, s_blocks):
    """Dequantize weight codes [N, K] with block scales [N/128, K/128]."""
    s = np.kron(s_blocks.astype(np.float64), np.ones((128, 128)))
    return oracle.e4m3_decode(codes) * s


def _deq_cols_T(codesT, s_chunk_major):
    """Dequantize column-tile codes stored transposed [C, M] with scales [M/128, C]
    into the natural [M, C] matrix."""
    C, M = codesT.shape
    s = np.repeat(s_chunk_major.astype(np.float64), 128, axis=0)  # [M, C]
    return oracle.e4m3_decode(codesT).T * s


def test_fprop_exact_rational_brute_force_tiny():
    rng = np.random.default_rng(1)
    M, N, K = 4, 3, 256
    xq = _rand_codes(rng, (M, K))
    wq = _rand_codes(rng, (128, K))
    sx = _rand_scales(rng, (K // 128, M))
    sw = _rand_scales(rng, (1, K // 128))
    got, got_abs = oracle.gemm_fprop(xq, sx, wq, sw, rows=np.arange(M), cols=np.arange(N))
    dec = {c: Fraction(float(v)) if np.isfinite(v) else None for c, v in enumerate(oracle.e4m3_table())}
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            tabs = Fraction(0)
            for k in range(K):
                a = Fraction(float(sx[k // 128, m])) * dec[int(xq[m, k])]
                b = Fraction(float(sw[n // 128, k // 128])) * dec[int(wq[n, k])]
                tot += a * b
                tabs += abs(a * b)
            assert abs(Fraction(got[m, n]) - tot) <= Fraction(2) ** -50 * tabs
            assert abs(Fraction(got_abs[m, n]) - tabs) <= Fraction(2) ** -50 * tabs


def test_fprop_matches_float64_matmul_of_dequantized_operands_tiny_config():
    lin = synth.tiny()
    xq, sx = oracle.quantize_rowwise(lin.x.numpy())
    wq, _, sw = oracle.quantize_weight_block(lin.w.numpy())
    y, yabs = oracle.gemm_fprop(xq, sx, wq, sw)
    a = _deq_rows(xq, sx)
    b = _deq_blocks(wq, sw)
    ref = a @ b.T
    refabs = np.abs(a) @ np.abs(b).T
    assert np.all(np.abs(y - ref) <= 1e-13 * refabs + 1e-300)
    assert np.allclose(yabs, refabs, rtol=1e-13, atol=0)
    # and the block-scaled FP8 result is close to the unquantized product
    exact = lin.x.numpy().astype(np.float64) @ lin.w.numpy().astype(np.float64).T
    assert np.max(np.abs(y - exact)) <= 2.0 ** -3 * np.max(np.abs(np.abs(lin.x.numpy()) @ np.abs(lin.w.numpy()).T))


def test_scale_selection_fprop_blocks_not_transposed():
    # distinct power-of-two scales per (n-block, k-chunk) and per (chunk, row)
    rng = np.random.default_rng(2)
    M, N, K = 256, 384, 512
    xq = _rand_codes(rng, (M, K), hi=0x60)
    wq = _rand_codes(rng, (N, K), hi=0x60)
    sx = _pow2_scales(rng, (K // 128, M))
    sw = _pow2_scales(rng, (N // 128, K // 128))
    y, _ = oracle.gemm_fprop(xq, sx, wq, sw)
    ref = _deq_rows(xq, sx) @ _deq_blocks(wq, sw).T
    assert np.array_equal(y, ref) or np.max(np.abs(y - ref) / (np.abs(ref) + 1e-300)) < 1e-15


def test_dgrad_matches_float64_matmul():
    rng = np.random.default_rng(3)
    M, N, K = 256, 384, 256
    dyq = _rand_codes(rng, (M, N))
    sdy = _rand_scales(rng, (N // 128, M))
    wq = _rand_codes(rng, (N, K))
    sw = _rand_scales(rng, (N // 128, K // 128))
    dx, dxabs = oracle.gemm_dgrad(dyq, sdy, wq, sw)
    a = _deq_rows(dyq, sdy)
    b = _deq_blocks(wq, sw)
    ref = a @ b
    refabs = np.abs(a) @ np.abs(b)
    assert np.all(np.abs(dx - ref) <= 1e-13 * refabs)
    assert np.allclose(dxabs, refabs, rtol=1e-13, atol=0)


def test_wgrad_matches_float64_matmul():
    rng = np.random.default_rng(4)
    M, N, K = 384, 256, 128
    dyqT = _rand_codes(rng, (N, M))
    sdyT = _rand_scales(rng, (M // 128, N))
    xqT = _rand_codes(rng, (K, M))
    sxT = _rand_scales(rng, (M // 128, K))
    dw, dwabs = oracle.gemm_wgrad(dyqT, sdyT, xqT, sxT)
    dy = _deq_cols_T(dyqT, sdyT)   # [M, N]
    x = _deq_cols_T(xqT, sxT)      # [M, K]
    ref = dy.T @ x
    refabs = np.abs(dy).T @ np.abs(x)
    assert np.all(np.abs(dw - ref) <= 1e-13 * refabs)
    assert np.allclose(dwabs, refabs, rtol=1e-13, atol=0)


def _integer_codes(rng, shape, with_448_at=None):
    """Codes of small integers in [-3, 3] (s = 1 tiles need a 448 in each tile)."""
    table = oracle.e4m3_table()
    ints = np.array([-3, -2, -1, 0, 1, 2, 3], dtype=np.float32)
    codes_of = {float(v): int(oracle.e4m3_encode(np.array([v], np.float32))[0]) for v in ints}
    vals = rng.choice(ints, size=shape, p=[0.05, 0.1, 0.15, 0.4, 0.15, 0.1, 0.05])
    codes = np.vectorize(lambda v: codes_of[float(v)])(vals).astype(np.uint8)
    assert np.all(table[codes] == vals)
    return codes, vals.astype(np.int64)


def test_exact_integer_case_all_three_gemms():
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 384
    xq, xv = _integer_codes(rng, (M, K))
    wq, wv = _integer_codes(rng, (N, K))
    one = lambda shape: np.ones(shape, dtype=np.float32)
    y, _ = oracle.gemm_fprop(xq, one((K // 128, M)), wq, one((N // 128, K // 128)))
    assert np.array_equal(y, (xv @ wv.T).astype(np.float64))
    dyq, dyv = _integer_codes(rng, (M, N))
    dx, _ = oracle.gemm_dgrad(dyq, one((N // 128, M)), wq, one((N // 128, K // 128)))
    assert np.array_equal(dx, (dyv @ wv).astype(np.float64))
    dyqT = np.ascontiguousarray(dyq.T)
    xqT = np.ascontiguousarray(xq.T)
    dw, _ = oracle.gemm_wgrad(dyqT, one((M // 128, N)), xqT, one((M // 128, K)))
    assert np.array_equal(dw, (dyv.T @ xv).astype(np.float64))


def test_single_nonzero_chunk_selects_its_scales():
    rng = np.random.default_rng(6)
    M, N, K = 128, 256, 512
    xq, xv = _integer_codes(rng, (M, K))
    wq, wv = _integer_codes(rng, (N, K))
    xq[:, :256] = 0
    xq[:, 384:] = 0       # only chunk 2 is nonzero
    xv[:, :256] = 0
    xv[:, 384:] = 0
    sx = np.ones((4, M), np.float32)
    sx[2] = 2.0 ** np.arange(M, dtype=np.float32).clip(max=20) / 2.0 ** 10
    sw = np.ones((2, 4), np.float32)
    sw[0, 2] = 4.0
    sw[1, 2] = 0.25
    sw[1, 1] = 1024.0     # a scale of a zero chunk must not leak in
    y, _ = oracle.gemm_fprop(xq, sx, wq, sw)
    ref = (xv @ wv.T).astype(np.float64) * sx[2][:, None].astype(np.float64) \
        * np.repeat(sw[:, 2], 128)[None, :].astype(np.float64)
    assert np.array_equal(y, ref)


def test_k_equals_128_single_chunk():
    rng = np.random.default_rng(7)
    xq = _rand_codes(rng, (128, 128))
    wq = _rand_codes(rng, (128, 128))
    sx = _rand_scales(rng, (1, 128))
    sw = _rand_scales(rng, (1, 1))
    y, _ = oracle.gemm_fprop(xq, sx, wq, sw)
    a, b = _deq_rows(xq, sx), _deq_blocks(wq, sw)
    ref = a @ b.T
    assert np.all(np.abs(y - ref) <= 1e-13 * (np.abs(a) @ np.abs(b).T))


def test_sampled_rows_and_columns_equal_full_result():
    rng = np.random.default_rng(8)
    xq = _rand_codes(rng, (256, 256))
    wq = _rand_codes(rng, (384, 256))
    sx = _rand_scales(rng, (2, 256))
    sw = _rand_scales(rng, (3, 2))
    full, fabs = oracle.gemm_fprop(xq, sx, wq, sw)
    rows = np.array([0, 5, 255, 128])
    cols = np.array([383, 0, 129])
    part, pabs = oracle.gemm_fprop(xq, sx, wq, sw, rows=rows, cols=cols)
    assert np.array_equal(part, full[np.ix_(rows, cols)])
    assert np.array_equal(pabs, fabs[np.ix_(rows, cols)])


# ---------------------------------------------------------------------------
# BF16 rounding and the tolerance
# ---------------------------------------------------------------------------

def test_bf16_rounding_matches_torch_on_fp32_exact_values():
    rng = np.random.default_rng(9)
    v = (rng.standard_normal(1 << 16) * np.exp2(rng.integers(-130, 120, 1 << 16))).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_from_double(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rounding_is_direct_not_double():
    # 1 + 2^-8 + 2^-30: above the BF16 midpoint 1 + 2^-8, so it rounds up to
    # 1 + 2^-7; rounding to FP32 first would land on the midpoint and go to 1.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    got = oracle.bf16_bits_to_f64(oracle.bf16_from_double(np.array([v])))[0]
    assert got == 1.0 + 2.0 ** -7
    assert oracle.bf16_bits_to_f64(oracle.bf16_from_double(np.array([1.0 + 2.0 ** -8])))[0] == 1.0
    assert oracle.bf16_bits_to_f64(oracle.bf16_from_double(np.array([1.0 + 3 * 2.0 ** -8])))[0] == 1.0 + 2.0 ** -6


def test_bf16_ulp_and_tolerance():
    assert oracle.bf16_ulp(np.array([1.0]))[0] == 2.0 ** -7
    assert oracle.bf16_ulp(np.array([1.99]))[0] == 2.0 ** -7
    assert oracle.bf16_ulp(np.array([-3.0]))[0] == 2.0 ** -6
    assert oracle.bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133
    assert oracle.bf16_ulp(np.array([2.0 ** -130]))[0] == 2.0 ** -133
    tol = oracle.gemm_tolerance(np.array([1.0]), np.array([10.0]))
    assert tol[0] == pytest.approx(2e-3 * 10 + 2.0 ** -7)
    ok, worst, _ = oracle.gemm_check(oracle.bf16_from_double(np.array([1.0 + 2 ** -7])), np.array([1.0]), np.array([0.0]))
    assert ok and worst == 1.0
    ok, _, _ = oracle.gemm_check(oracle.bf16_from_double(np.array([1.0 + 2 ** -6])), np.array([1.0]), np.array([0.0]))
    assert not ok


def test_f32_ulp_matches_numpy_spacing():
    """f32_ulp against numpy's nextafter-based spacing (upward gap) on normal,
    subnormal and power-of-two magnitudes."""
    rng = np.random.default_rng(31)
    vals = np.concatenate([rng.uniform(-1e6, 1e6, 1000), np.ldexp(1.0, np.arange(-149, 120)),
                           rng.uniform(0, 1, 100) * 2.0 ** -130]).astype(np.float32)
    want = np.spacing(np.abs(vals)).astype(np.float64)
    got = oracle.f32_ulp(vals.astype(np.float64))
    assert np.array_equal(got, want)
    assert oracle.f32_ulp(0.0) == 2.0 ** -149


def test_f32_tolerance_accepts_rounding_and_rejects_one_extra_ulp_of_s():
    """An FP32 output that is the correctly rounded exact value passes; the bound
    grows by one FP32 ulp when the product is added into a base array."""
    rng = np.random.default_rng(32)
    exact = rng.normal(0, 3, 1000)
    absd = np.abs(exact) * 1.5
    ok, _, _ = oracle.gemm_check_f32(exact.astype(np.float32), exact, absd)
    assert ok
    bad = exact + 2e-3 * absd + 2 * oracle.f32_ulp(exact)
    ok, _, _ = oracle.gemm_check_f32(bad, exact, absd)
    assert not ok
    base = rng.normal(0, 100, 1000).astype(np.float32)
    summed = (base.astype(np.float64) + exact).astype(np.float32)
    ok, _, _ = oracle.gemm_check_f32(summed, exact, absd, base=base)
    assert ok


# ---------------------------------------------------------------------------
# The matmul-step forms (gemm_*_mm) against the literal C loops
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 640), (384, 256, 1024)])
def test_matmul_step_forms_are_bit_identical_to_the_loops(M, N, K):
    """Same definition, same binary64 operations outside the exact chunk
    sums: values and |.|-sums must agree bit for bit on random codes of every
    magnitude (subnormals and signed zeros included) and random scales, on
    ragged row/column selections."""
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    rows = np.sort(rng.choice(M, size=min(M, 96), replace=False))
    cols = np.sort(rng.choice(N, size=min(N, 80), replace=False))
    # Fprop: xq [M, K], wq [N, K]
    xq, wq = _rand_codes(rng, (M, K)), _rand_codes(rng, (N, K))
    sx, sw = _rand_scales(rng, (K // 128, M)), _rand_scales(rng, (N // 128, K // 128))
    for got, want in zip(oracle.gemm_fprop_mm(xq, sx, wq, sw, rows, cols),
                         oracle.gemm_fprop(xq, sx, wq, sw, rows, cols)):
        assert np.array_equal(got.view(np.uint64), want.view(np.uint64))
    # Dgrad: dyq [M, N] reduced over N, wq2 [N, K] natural layout
    dyq, wq2 = _rand_codes(rng, (M, N)), _rand_codes(rng, (N, K))
    sdy, sw2 = _rand_scales(rng, (N // 128, M)), _rand_scales(rng, (N // 128, K // 128))
    kcols = np.sort(rng.choice(K, size=min(K, 72), replace=False))
    for got, want in zip(oracle.gemm_dgrad_mm(dyq, sdy, wq2, sw2, rows, kcols),
                         oracle.gemm_dgrad(dyq, sdy, wq2, sw2, rows, kcols)):
        assert np.array_equal(got.view(np.uint64), want.view(np.uint64))
    # Wgrad: dyqT [N, M], xqT [K, M] reduced over M
    dyqT, xqT = _rand_codes(rng, (N, M)), _rand_codes(rng, (K, M))
    sdyT, sxT = _rand_scales(rng, (M // 128, N)), _rand_scales(rng, (M // 128, K))
    nrows = np.sort(rng.choice(N, size=min(N, 64), replace=False))
    for got, want in zip(oracle.gemm_wgrad_mm(dyqT, sdyT, xqT, sxT, nrows, kcols),
                         oracle.gemm_wgrad(dyqT, sdyT, xqT, sxT, nrows, kcols)):
        assert np.array_equal(got.view(np.uint64), want.view(np.uint64))


def test_matmul_step_form_on_a_long_reduction():
    """A 4096-deep Wgrad reduction (32 chunks) with codes at the extremes of
    the E4M3 range, where a chunk sum needs the most bits."""
    rng = np.random.default_rng(77)
    N, K, M = 128, 128, 4096
    ext = np.array([0x01, 0x02, 0x7E, 0x7D, 0x81, 0xFE], dtype=np.uint8)
    dyqT = rng.choice(ext, size=(N, M)).astype(np.uint8)
    xqT = rng.choice(ext, size=(K, M)).astype(np.uint8)
    sdyT, sxT = _rand_scales(rng, (M // 128, N)), _rand_scales(rng, (M // 128, K))
    rows, cols = np.arange(0, N, 5), np.arange(0, K, 3)
    for got, want in zip(oracle.gemm_wgrad_mm(dyqT, sdyT, xqT, sxT, rows, cols),
                         oracle.gemm_wgrad(dyqT, sdyT, xqT, sxT, rows, cols)):
        assert np.array_equal(got.view(np.uint64), want.view(np.uint64))
