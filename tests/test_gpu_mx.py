"""GPU parity of the MX variant (power-of-two scale per 1x32 block) with the
oracle: quantizer codes and exponent bytes bit for bit, the block-scaled MMA
GEMM within |C - C_exact| <= 2e-3 * sum_k |a_k b_k| + 1 BF16 ulp, exact
integer products bit for bit.  Expected values come from `oracle` only."""
import numpy as np
import pytest
import torch

import oracle
from fp8_precision_pretraining_amax_b300 import synth
from tests.helpers import assert_codes_equal, check_gemm_tiles, host_input, random_codes, sample_tiles, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_precision_pretraining_amax_b300 import fp8bq
    return fp8bq


def _rowwise_case(fb, x):
    q, e8 = fb.mx_quantize_rowwise(x)
    fb.check()
    wq, we = oracle.mx_quantize_rowwise(host_input(x))
    assert_codes_equal(q.cpu().numpy(), wq, "mx rowwise codes")
    assert_codes_equal(e8.cpu().numpy(), we, "mx rowwise exponents")


@pytest.mark.parametrize("R,C", [(1, 128), (3, 384), (257, 256), (64, 2048), (1000, 640)])
def test_mx_rowwise_bf16(fb, R, C):
    gen = synth.generator(100 + R + C)
    x = synth.activations(R, C, gen).cuda()
    x[0, :32] = 0.0                     # an all-zero block
    x[-1, -32:] *= 2.0 ** -120          # tiny values: BF16 subnormals, clamped exponent
    _rowwise_case(fb, x)


@pytest.mark.parametrize("R,C", [(5, 128), (130, 384)])
def test_mx_rowwise_fp32_wide_range(fb, R, C):
    rng = np.random.default_rng(R * C)
    x = (rng.standard_normal((R, C)) * np.exp2(rng.integers(-80, 80, (R, 1)))).astype(np.float32)
    x[1, 5] = -0.0
    _rowwise_case(fb, torch.from_numpy(x).cuda())


def test_mx_rowwise_every_bf16_magnitude(fb):
    """Every positive finite BF16 value as the amax of a block (with a
    neighbour of each sign below it): all exponents from -127 to 121."""
    mags = np.arange(1, 0x7F80, dtype=np.uint32)
    n = mags.size
    R = (n + 3) // 4
    bits = np.zeros((R * 4, 32), dtype=np.uint16)
    bits[:n, 0] = mags
    bits[:n, 1] = np.maximum(mags, 2) - 1
    bits[:n, 2] = (np.maximum(mags, 3) - 2) | 0x8000
    x = torch.from_numpy(bits.reshape(R, 128).view(np.int16)).view(torch.bfloat16).cuda()
    _rowwise_case(fb, x)


def test_mx_rowwise_with_row_pitch(fb):
    gen = synth.generator(7)
    full = synth.activations(96, 640, gen).cuda()
    _rowwise_case(fb, full[:, 128:512])


def _colwise_case(fb, x):
    qT, e8 = fb.mx_quantize_colwise(x)
    fb.check()
    wq, we = oracle.mx_quantize_colwise(host_input(x))
    assert_codes_equal(qT.cpu().numpy(), wq, "mx colwise codes")
    assert_codes_equal(e8.cpu().numpy(), we, "mx colwise exponents")


@pytest.mark.parametrize("M,C", [(128, 128), (256, 384), (640, 256)])
def test_mx_colwise_bf16(fb, M, C):
    gen = synth.generator(200 + M + C)
    x = synth.grads(M, C, gen).cuda()
    x[32:64, 3] = 0.0
    _colwise_case(fb, x)


def test_mx_colwise_fp32_and_pitch(fb):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((256, 512)) * np.exp2(rng.integers(-40, 40, (1, 512)))).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    _colwise_case(fb, xt)
    _colwise_case(fb, xt[:, 128:384])


def _rowcol_case(fb, x):
    q, e8, qT, e8T = fb.mx_quantize_rowcol(x)
    fb.check()
    h = host_input(x)
    wq, we = oracle.mx_quantize_rowwise(h)
    wqT, weT = oracle.mx_quantize_colwise(h)
    assert_codes_equal(q.cpu().numpy(), wq, "mx rowcol row-wise codes")
    assert_codes_equal(e8.cpu().numpy(), we, "mx rowcol row-wise exponents")
    assert_codes_equal(qT.cpu().numpy(), wqT, "mx rowcol column-wise codes")
    assert_codes_equal(e8T.cpu().numpy(), weT, "mx rowcol column-wise exponents")


@pytest.mark.parametrize("M,C", [(128, 128), (384, 256), (256, 640)])
def test_mx_rowcol_bf16(fb, M, C):
    gen = synth.generator(300 + M + C)
    x = synth.activations(M, C, gen).cuda()
    x[5, 32:64] = 0.0
    x[64:96, 7] = 0.0
    x[-1, :] *= 2.0 ** -118
    _rowcol_case(fb, x)


def test_mx_rowcol_fp32_and_pitch(fb):
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((256, 640)) * np.exp2(rng.integers(-50, 50, (256, 1)))).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    _rowcol_case(fb, xt)
    _rowcol_case(fb, xt[:, 128:512])
    gen = synth.generator(10)
    _rowcol_case(fb, synth.activations(128, 768, gen).cuda()[:, 256:640])


def _rand_exps(rng, shape, lo=112, hi=136):
    return rng.integers(lo, hi + 1, size=shape).astype(np.uint8)


def _mx_gemm(fb, a, ea, b, eb):
    d = fb.mx_gemm(to_dev(a), to_dev(ea), to_dev(b), to_dev(eb))
    fb.check()
    return d


def _tiles(I, J):
    return [(i, j) for i in range(I // 128) for j in range(J // 128)]


@pytest.mark.parametrize("I,J,K", [(128, 128, 128), (128, 256, 256), (256, 384, 512), (384, 640, 640),
                                   (256, 1152, 1280), (1024, 896, 384)])
def test_mx_gemm_random_codes(fb, I, J, K):
    """Output tiles are 192 columns wide: J = 384 and 1152 end on a full
    tile, J = 128, 256, 640 and 896 on a partial one."""
    rng = np.random.default_rng(I + 3 * J + 7 * K)
    a, b = random_codes(rng, (I, K)), random_codes(rng, (J, K))
    ea, eb = _rand_exps(rng, (K // 128, I, 4)), _rand_exps(rng, (K // 128, J, 4))
    d = _mx_gemm(fb, a, ea, b, eb)
    assert d.shape == (I, J)
    picks = _tiles(I, J) if I * J <= 384 * 384 else sample_tiles(rng, I, J, 16)
    check_gemm_tiles(d, oracle.mx_gemm, (a, ea, b, eb), picks, what=f"mx gemm {I}x{J}x{K}")


def test_mx_gemm_exact_integers(fb):
    """Blocks with amax 448 get exponent 0 and integer operands give an
    integer product: the BF16 output must equal the rounded integer result."""
    rng = np.random.default_rng(41)
    I, J, K = 256, 384, 512
    ints = np.array([0, 1, 2, 3, 4, 6, 8], dtype=np.float32)
    xa = rng.choice(ints, size=(I, K)) * rng.choice([-1, 1], size=(I, K))
    xb = rng.choice(ints, size=(J, K)) * rng.choice([-1, 1], size=(J, K))
    xa[:, ::32] = 448.0
    xb[:, 1::32] = 448.0
    qa, ea = oracle.mx_quantize_rowwise(xa.astype(np.float32))
    qb, eb = oracle.mx_quantize_rowwise(xb.astype(np.float32))
    d = _mx_gemm(fb, qa, ea, qb, eb)
    want = oracle.bf16_from_double(xa.astype(np.float64) @ xb.astype(np.float64).T)
    got = synth.bf16_bits(d)
    assert np.array_equal(got, want), int(np.sum(got != want))


def test_mx_gemm_block_exponents_select_their_32_elements(fb):
    """One nonzero 32-element block per row pair (different block for each
    output row): pins which byte of which word the MMA applies to which K."""
    rng = np.random.default_rng(42)
    I, J, K = 128, 256, 512
    a = np.zeros((I, K), dtype=np.uint8)
    b = random_codes(rng, (J, K), max_mag=0x60)
    blk = rng.integers(0, K // 32, size=I)
    for i in range(I):
        a[i, 32 * blk[i]:32 * blk[i] + 32] = random_codes(rng, (32,), max_mag=0x60)
    ea, eb = _rand_exps(rng, (K // 128, I, 4), 100, 150), _rand_exps(rng, (K // 128, J, 4), 100, 150)
    d = _mx_gemm(fb, a, ea, b, eb)
    check_gemm_tiles(d, oracle.mx_gemm, (a, ea, b, eb), _tiles(I, J), what="mx single-block rows")


def test_mx_gemm_empty_reduction_writes_zeros(fb):
    d = torch.full((128, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    e = torch.empty((0, 128, 4), dtype=torch.uint8, device="cuda")
    fb.fp8bq_mx_gemm(torch.empty((128, 0), dtype=torch.uint8, device="cuda"), e,
                     torch.empty((256, 0), dtype=torch.uint8, device="cuda"),
                     torch.empty((0, 256, 4), dtype=torch.uint8, device="cuda"), d)
    fb.check()
    assert torch.count_nonzero(d).item() == 0


def test_mx_linear_layer_fprop_dgrad_wgrad(fb):
    """One step of LinearMX (three row+column quantizer passes, three MX
    GEMMs) on the GPU, against the oracle's quantizers and GEMM."""
    gen = synth.generator(43)
    M, K, N = 512, 384, 640
    x = synth.activations(M, K, gen).cuda()
    w = synth.weight(N, K, gen).cuda()
    dy = synth.grads(M, N, gen).cuda()
    from fp8_precision_pretraining_amax_b300.linear import LinearMX
    L = LinearMX(M, K, N, device="cuda")
    y, dx, dw = L.step(x, w, dy)
    fb.check()
    xq, ex, wq, ew, dyq, edy = L.xq, L.ex, L.wq, L.ew, L.dyq, L.edy
    wqT, ewT, dyqT, edyT, xqT, exT = L.wqT, L.ewT, L.dyqT, L.edyT, L.xqT, L.exT
    # every quantizer output equals the oracle's; the GEMM checks then take
    # the oracle's codes as their inputs
    want = {}
    for name, got, fn, src in (("xq", (xq, ex), oracle.mx_quantize_rowwise, x),
                               ("wq", (wq, ew), oracle.mx_quantize_rowwise, w),
                               ("dyq", (dyq, edy), oracle.mx_quantize_rowwise, dy),
                               ("wqT", (wqT, ewT), oracle.mx_quantize_colwise, w),
                               ("dyqT", (dyqT, edyT), oracle.mx_quantize_colwise, dy),
                               ("xqT", (xqT, exT), oracle.mx_quantize_colwise, x)):
        want[name] = fn(host_input(src))
        assert_codes_equal(got[0].cpu().numpy(), want[name][0], name)
        assert_codes_equal(got[1].cpu().numpy(), want[name][1], name + " exponents")
    check_gemm_tiles(y, oracle.mx_gemm, (*want["xq"], *want["wq"]), _tiles(M, N), what="mx fprop")
    check_gemm_tiles(dx, oracle.mx_gemm, (*want["dyq"], *want["wqT"]), _tiles(M, K), what="mx dgrad")
    check_gemm_tiles(dw, oracle.mx_gemm, (*want["dyqT"], *want["xqT"]), _tiles(N, K), what="mx wgrad")


@pytest.mark.slow
def test_mx_gate_up_3p8b_sampled(fb):
    """The 3.8B layer's gate+up projection (3072 -> 16384) at 8192 tokens in
    the launch configuration the benchmark uses, on sampled output tiles."""
    gen = synth.generator(44, "cuda")
    M, K, N = 8192, 3072, 16384
    x = synth.activations(M, K, gen, device="cuda")
    w = synth.weight(N, K, gen, device="cuda")
    xq, ex = fb.mx_quantize_rowwise(x)
    wq, ew = fb.mx_quantize_rowwise(w)
    y = fb.mx_gemm(xq, ex, wq, ew)
    fb.check()
    ox, ow = oracle.mx_quantize_rowwise(host_input(x)), oracle.mx_quantize_rowwise(host_input(w))
    assert_codes_equal(xq.cpu().numpy(), ox[0], "x codes")
    assert_codes_equal(ex.cpu().numpy(), ox[1], "x exponents")
    assert_codes_equal(wq.cpu().numpy(), ow[0], "w codes")
    assert_codes_equal(ew.cpu().numpy(), ow[1], "w exponents")
    rng = np.random.default_rng(44)
    check_gemm_tiles(y, oracle.mx_gemm, (*ox, *ow), sample_tiles(rng, M, N, 8), what="mx gate+up")
