"""GPU parity of the block-scaled GEMMs with the binary64 oracle.

Inputs to both sides are the same codes and scales, produced on the host by
the oracle's quantizers or drawn directly as random codes/scales (the GEMM
accepts any).  Acceptance per element: |C - C_exact| <= 2e-3 * sum_k |a_k b_k|
+ 1 BF16 ulp.  Exact-integer cases must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_precision_pretraining_amax_b300 import synth
from tests.helpers import check_gemm_tiles, host_input, random_codes, random_scales, sample_tiles, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_precision_pretraining_amax_b300 import fp8bq
    return fp8bq


def _all_tiles(rows, cols):
    return [(i, j) for i in range(rows // 128) for j in range(cols // 128)]


def _fprop(fb, xq, sx, wq, sw):
    y = fb.gemm_fprop(to_dev(xq), to_dev(sx), to_dev(wq), to_dev(sw))
    fb.check()
    return y


def _dgrad(fb, dyq, sdy, wq, sw):
    wqT = np.ascontiguousarray(wq.T)
    dx = fb.gemm_dgrad(to_dev(dyq), to_dev(sdy), to_dev(wqT), to_dev(sw))
    fb.check()
    return dx


def _wgrad(fb, dyqT, sdyT, xqT, sxT):
    dw = fb.gemm_wgrad(to_dev(dyqT), to_dev(sdyT), to_dev(xqT), to_dev(sxT))
    fb.check()
    return dw


def test_tiny_config_fprop_all_tiles(fb):
    lin = synth.tiny()
    xq, sx = oracle.quantize_rowwise(lin.x.numpy())
    wq, _, sw = oracle.quantize_weight_block(lin.w.numpy())
    y = _fprop(fb, xq, sx, wq, sw)
    assert y.shape == (256, 384)
    check_gemm_tiles(y, oracle.gemm_fprop, (xq, sx, wq, sw), _all_tiles(256, 384), what="tiny fprop")


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (128, 256, 256), (256, 384, 1152), (640, 640, 384),
                                   (2048, 2560, 512)])
def test_fprop_random_codes(fb, M, N, K):
    rng = np.random.default_rng(M + N + K)
    xq, wq = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sx, sw = random_scales(rng, (K // 128, M)), random_scales(rng, (N // 128, K // 128))
    y = _fprop(fb, xq, sx, wq, sw)
    picks = _all_tiles(M, N) if M * N <= 640 * 640 else sample_tiles(rng, M, N, 12)
    check_gemm_tiles(y, oracle.gemm_fprop, (xq, sx, wq, sw), picks, what=f"fprop {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 640), (384, 1024, 256)])
def test_dgrad_random_codes(fb, M, N, K):
    rng = np.random.default_rng(7 * M + N + K)
    dyq, wq = random_codes(rng, (M, N)), random_codes(rng, (N, K))
    sdy, sw = random_scales(rng, (N // 128, M)), random_scales(rng, (N // 128, K // 128))
    dx = _dgrad(fb, dyq, sdy, wq, sw)
    assert dx.shape == (M, K)
    check_gemm_tiles(dx, oracle.gemm_dgrad, (dyq, sdy, wq, sw), _all_tiles(M, K), what=f"dgrad {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (640, 384, 256), (256, 256, 640)])
def test_wgrad_random_codes(fb, M, N, K):
    rng = np.random.default_rng(11 * M + N + K)
    dyqT, xqT = random_codes(rng, (N, M)), random_codes(rng, (K, M))
    sdyT, sxT = random_scales(rng, (M // 128, N)), random_scales(rng, (M // 128, K))
    dw = _wgrad(fb, dyqT, sdyT, xqT, sxT)
    assert dw.shape == (N, K)
    check_gemm_tiles(dw, oracle.gemm_wgrad, (dyqT, sdyT, xqT, sxT), _all_tiles(N, K), what=f"wgrad {M}x{N}x{K}")


def _integer_operands(rng, shape):
    ints = np.array([-3, -2, -1, 0, 1, 2, 3], dtype=np.float32)
    vals = rng.choice(ints, size=shape, p=[0.05, 0.1, 0.15, 0.4, 0.15, 0.1, 0.05]).astype(np.float32)
    return oracle.e4m3_encode(vals), vals.astype(np.int64)


def test_exact_integer_cases_are_bit_exact(fb):
    """s = 1 (or a power of two) and small integers: every partial sum is exact
    in FP32, so the BF16 output must equal the oracle's RNE rounding bit for bit.
    Pins layout, indexing and scale wiring independently of the tolerance."""
    rng = np.random.default_rng(21)
    M, N, K = 384, 640, 512
    xq, xv = _integer_operands(rng, (M, K))
    wq, wv = _integer_operands(rng, (N, K))
    sx = np.exp2(rng.integers(-2, 3, size=(K // 128, M))).astype(np.float32)
    sw = np.exp2(rng.integers(-2, 3, size=(N // 128, K // 128))).astype(np.float32)
    y = _fprop(fb, xq, sx, wq, sw)
    exact, _ = oracle.gemm_fprop(xq, sx, wq, sw)
    assert np.array_equal(synth.bf16_bits(y), oracle.bf16_from_double(exact))

    dyq, _ = _integer_operands(rng, (M, N))
    sdy = np.exp2(rng.integers(-2, 3, size=(N // 128, M))).astype(np.float32)
    wq2, _ = _integer_operands(rng, (N, K))
    dx = _dgrad(fb, dyq, sdy, wq2, sw)
    exact, _ = oracle.gemm_dgrad(dyq, sdy, wq2, sw)
    assert np.array_equal(synth.bf16_bits(dx), oracle.bf16_from_double(exact))

    Mt = 512
    dyqT, _ = _integer_operands(rng, (N, Mt))
    xqT, _ = _integer_operands(rng, (K, Mt))
    sdyT = np.exp2(rng.integers(-2, 3, size=(Mt // 128, N))).astype(np.float32)
    sxT = np.exp2(rng.integers(-2, 3, size=(Mt // 128, K))).astype(np.float32)
    dw = _wgrad(fb, dyqT, sdyT, xqT, sxT)
    exact, _ = oracle.gemm_wgrad(dyqT, sdyT, xqT, sxT)
    assert np.array_equal(synth.bf16_bits(dw), oracle.bf16_from_double(exact))


def test_single_nonzero_chunk_and_scale_selection(fb):
    rng = np.random.default_rng(22)
    M, N, K = 256, 512, 640
    xq, _ = _integer_operands(rng, (M, K))
    wq, _ = _integer_operands(rng, (N, K))
    xq[:, :384] = 0
    xq[:, 512:] = 0                                      # only chunk 3 is nonzero
    sx = np.ones((K // 128, M), np.float32)
    sx[3] = np.exp2(np.arange(M) % 7 - 3).astype(np.float32)
    sx[1] = 1024.0                                        # scales of zero chunks must not leak
    sw = np.exp2(rng.integers(-3, 4, size=(N // 128, K // 128))).astype(np.float32)
    y = _fprop(fb, xq, sx, wq, sw)
    exact, _ = oracle.gemm_fprop(xq, sx, wq, sw)
    assert np.array_equal(synth.bf16_bits(y), oracle.bf16_from_double(exact))


def test_empty_reduction_writes_zeros(fb):
    dev = "cuda"
    y = torch.full((128, 256), 7.0, dtype=torch.bfloat16, device=dev)
    e8 = torch.empty((128, 0), dtype=torch.uint8, device=dev)
    fb.fp8bq_gemm_fprop(e8, torch.empty((0, 128), dtype=torch.float32, device=dev),
                        torch.empty((256, 0), dtype=torch.uint8, device=dev),
                        torch.empty((2, 0), dtype=torch.float32, device=dev), y)
    fb.check()
    assert torch.count_nonzero(y).item() == 0


def test_config_qkv_1p7b_fprop_from_real_distribution(fb):
    """Qwen3-1.7B QKV Fprop (M=8192, K=2048, N=4096): activations with outlier
    channels quantized by the oracle, 64 seeded random 128x128 output tiles
    plus the four corner tiles."""
    lin = synth.qkv_1p7b()
    xq, sx = oracle.quantize_rowwise(host_input(lin.x))
    wq, _, sw = oracle.quantize_weight_block(host_input(lin.w))
    y = _fprop(fb, xq, sx, wq, sw)
    rng = np.random.default_rng(23)
    worst = check_gemm_tiles(y, oracle.gemm_fprop, (xq, sx, wq, sw), sample_tiles(rng, 8192, 4096, 64),
                             what="qkv fprop")
    assert worst <= 1.0


@pytest.mark.slow
def test_full_size_up_proj_backward_sampled(fb):
    """Backward of the 2048 -> 6144 up-projection at 16384 tokens: Dgrad
    (reduce 6144) and Wgrad (reduce 16384) on random codes/scales of every
    magnitude at the full shapes, checked on sampled tiles (the workload's own
    distributions are covered in test_gpu_configs.py)."""
    rng = np.random.default_rng(24)
    M, N, K = 16384, 6144, 2048
    dyq, wq = random_codes(rng, (M, N)), random_codes(rng, (N, K))
    sdy, sw = random_scales(rng, (N // 128, M)), random_scales(rng, (N // 128, K // 128))
    dx = _dgrad(fb, dyq, sdy, wq, sw)
    check_gemm_tiles(dx, oracle.gemm_dgrad_mm, (dyq, sdy, wq, sw), sample_tiles(rng, M, K, 16), what="dgrad full")
    dyqT = np.ascontiguousarray(dyq.T)
    xqT = random_codes(rng, (K, M))
    sdyT, sxT = random_scales(rng, (M // 128, N)), random_scales(rng, (M // 128, K))
    dw = _wgrad(fb, dyqT, sdyT, xqT, sxT)
    check_gemm_tiles(dw, oracle.gemm_wgrad_mm, (dyqT, sdyT, xqT, sxT), sample_tiles(rng, N, K, 16),
                     what="wgrad full")


# ---------------------------------------------------------------------------
# Wgrad with an FP32 output (overwrite or accumulate into)
# ---------------------------------------------------------------------------

def _check_f32_tiles(got_dev, oracle_fn, args, picks, base=None, tile=128, what=""):
    got = got_dev.cpu().numpy()
    for (bi, bj) in picks:
        rows = np.arange(bi * tile, (bi + 1) * tile)
        cols = np.arange(bj * tile, (bj + 1) * tile)
        exact, absd = oracle_fn(*args, rows=rows, cols=cols)
        b = None if base is None else base[np.ix_(rows, cols)]
        ok, ratio, err = oracle.gemm_check_f32(got[np.ix_(rows, cols)], exact, absd, base=b)
        assert ok, f"{what} tile ({bi},{bj}): worst error/tolerance {ratio:.3g}"


@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (640, 384, 256), (256, 256, 640)])
def test_wgrad_f32_random_codes(fb, M, N, K):
    rng = np.random.default_rng(13 * M + N + K)
    dyqT, xqT = random_codes(rng, (N, M)), random_codes(rng, (K, M))
    sdyT, sxT = random_scales(rng, (M // 128, N)), random_scales(rng, (M // 128, K))
    dev = [to_dev(a) for a in (dyqT, sdyT, xqT, sxT)]
    dw = fb.gemm_wgrad_f32(*dev)
    fb.check()
    assert dw.dtype == torch.float32 and dw.shape == (N, K)
    _check_f32_tiles(dw, oracle.gemm_wgrad, (dyqT, sdyT, xqT, sxT), _all_tiles(N, K), what=f"wgrad f32 {M}x{N}x{K}")
    # the BF16 kernel rounds the same FP32 accumulators: identical after RNE
    dw16 = fb.gemm_wgrad(*dev)
    fb.check()
    assert torch.equal(dw.to(torch.bfloat16), dw16)


def test_wgrad_f32_accumulates_into_the_output(fb):
    rng = np.random.default_rng(41)
    M, N, K = 384, 256, 384
    dyqT, xqT = random_codes(rng, (N, M)), random_codes(rng, (K, M))
    sdyT, sxT = random_scales(rng, (M // 128, N)), random_scales(rng, (M // 128, K))
    base = (rng.normal(0, 50, (N, K))).astype(np.float32)
    dw = to_dev(base)
    fb.fp8bq_gemm_wgrad_f32(to_dev(dyqT), to_dev(sdyT), to_dev(xqT), to_dev(sxT), dw, accumulate=True)
    fb.check()
    _check_f32_tiles(dw, oracle.gemm_wgrad, (dyqT, sdyT, xqT, sxT), _all_tiles(N, K), base=base,
                     what="wgrad f32 accumulate")


def test_wgrad_f32_token_shards_sum_to_the_full_product(fb):
    """Accumulating the Wgrad of consecutive token shards into one FP32 array
    gives the Wgrad of all tokens (the data-parallel / micro-batch use)."""
    rng = np.random.default_rng(42)
    M, N, K = 768, 256, 384
    dyqT, xqT = random_codes(rng, (N, M)), random_codes(rng, (K, M))
    sdyT, sxT = random_scales(rng, (M // 128, N)), random_scales(rng, (M // 128, K))
    dw = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    for m0, m1 in ((0, 256), (256, 640), (640, 768)):
        fb.fp8bq_gemm_wgrad_f32(to_dev(np.ascontiguousarray(dyqT[:, m0:m1])), to_dev(sdyT[m0 // 128:m1 // 128]),
                                to_dev(np.ascontiguousarray(xqT[:, m0:m1])), to_dev(sxT[m0 // 128:m1 // 128]), dw,
                                accumulate=True)
    fb.check()
    exact, absd = oracle.gemm_wgrad(dyqT, sdyT, xqT, sxT)
    ok, ratio, _ = oracle.gemm_check_f32(dw.cpu().numpy(), exact, absd)
    assert ok, ratio


def test_wgrad_f32_exact_integer_case_is_bit_exact(fb):
    rng = np.random.default_rng(43)
    M, N, K = 512, 384, 256
    dyqT, _ = _integer_operands(rng, (N, M))
    xqT, _ = _integer_operands(rng, (K, M))
    sdyT = np.exp2(rng.integers(-2, 3, size=(M // 128, N))).astype(np.float32)
    sxT = np.exp2(rng.integers(-2, 3, size=(M // 128, K))).astype(np.float32)
    dw = fb.gemm_wgrad_f32(to_dev(dyqT), to_dev(sdyT), to_dev(xqT), to_dev(sxT))
    fb.check()
    exact, _ = oracle.gemm_wgrad(dyqT, sdyT, xqT, sxT)
    assert np.array_equal(dw.cpu().numpy(), exact.astype(np.float32))
    # empty reduction: overwrite writes zeros, accumulate leaves the array alone
    z = torch.full((N, K), 7.0, dtype=torch.float32, device="cuda")
    e8, e32 = torch.empty((N, 0), dtype=torch.uint8, device="cuda"), torch.empty((0, N), device="cuda")
    k8, k32 = torch.empty((K, 0), dtype=torch.uint8, device="cuda"), torch.empty((0, K), device="cuda")
    fb.fp8bq_gemm_wgrad_f32(e8, e32, k8, k32, z, accumulate=True)
    assert torch.all(z == 7.0)
    fb.fp8bq_gemm_wgrad_f32(e8, e32, k8, k32, z, accumulate=False)
    assert torch.all(z == 0.0)


# ---------------------------------------------------------------------------
# Fprop with a quantized output (the next linear's row-wise operand)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (384, 640, 256), (1024, 2048, 512)])
def test_fprop_q_matches_fprop_then_rowwise(fb, M, N, K):
    """The fused epilogue quantizes the BF16-rounded product exactly as the
    row-wise quantizer does; its BF16 output equals the plain Fprop's."""
    rng = np.random.default_rng(5 * M + N + K)
    xq, wq = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sx, sw = random_scales(rng, (K // 128, M)), random_scales(rng, (N // 128, K // 128))
    dev = [to_dev(a) for a in (xq, sx, wq, sw)]
    y_ref = fb.gemm_fprop(*dev)
    q_ref, s_ref = fb.quantize_rowwise(y_ref)
    y, yq, sy = fb.gemm_fprop_q(*dev)
    _, yq2, sy2 = fb.gemm_fprop_q(*dev, keep_bf16=False)
    fb.check()
    assert torch.equal(y, y_ref)
    assert torch.equal(yq, q_ref) and torch.equal(sy, s_ref)
    assert torch.equal(yq2, q_ref) and torch.equal(sy2, s_ref)
    # and against the oracle: codes of the GPU's BF16 output
    qo, so = oracle.quantize_rowwise(synth.bf16_bits(y))
    assert np.array_equal(yq.cpu().numpy(), qo)
    assert np.array_equal(sy.cpu().numpy().view(np.uint32), so.view(np.uint32))


def test_fprop_q_empty_reduction(fb):
    M, N = 256, 384
    e8 = torch.empty((M, 0), dtype=torch.uint8, device="cuda")
    w8 = torch.empty((N, 0), dtype=torch.uint8, device="cuda")
    yq = torch.full((M, N), 7, dtype=torch.uint8, device="cuda")
    sy = torch.zeros((N // 128, M), device="cuda")
    fb.fp8bq_gemm_fprop_q(e8, torch.empty((0, M), device="cuda"), w8, torch.empty((N // 128, 0), device="cuda"),
                          None, yq, sy)
    fb.check()
    assert torch.all(yq == 0) and torch.all(sy == 1.0)


def _split_counter_bytes(fb):
    """Bytes of the balanced Wgrad's arrival counters at the start of its
    scratch (one 4-byte counter per CTA rank and promotion warp, 16 per
    remaining tile, rounded up to 256 bytes); then each cluster's 512 KB of
    split slots."""
    total = fb.fp8bq_gemm_wgrad_scratch_bytes()
    return total - (total // (512 * 1024)) * (512 * 1024)


def test_wgrad_balanced_splits_tiles_and_repeats_bit_for_bit(fb):
    """81 output tiles of 256 x 256, 16 chunks each, over the persistent
    grid's clusters: one whole-tile round, then the chunks of the tiles left
    over shared out between all clusters, so that several clusters complete
    each of those tiles together.  Every output tile is within the bound, a
    second call gives the same bits, and the arrival counters are back at
    zero."""
    rng = np.random.default_rng(29)
    M, N, K = 2048, 2304, 2304
    dyqT, xqT = random_codes(rng, (N, M)), random_codes(rng, (K, M))
    sdyT, sxT = random_scales(rng, (M // 128, N)), random_scales(rng, (M // 128, K))
    dev = [to_dev(a) for a in (dyqT, sdyT, xqT, sxT)]
    scratch = fb.wgrad_scratch(dev[0].device)
    dw1 = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    dw2 = torch.empty_like(dw1)
    fb.fp8bq_gemm_wgrad_balanced(*dev, dw1, scratch)
    fb.fp8bq_gemm_wgrad_balanced(*dev, dw2, scratch)
    fb.check()
    torch.cuda.synchronize()
    assert torch.equal(dw1.view(torch.int16), dw2.view(torch.int16))
    nc = _split_counter_bytes(fb)
    assert nc > 0 and int(scratch[:nc].sum()) == 0
    check_gemm_tiles(dw1, oracle.gemm_wgrad_mm, (dyqT, sdyT, xqT, sxT), _all_tiles(N, K), what="wgrad balanced")


def test_wgrad_balanced_one_leftover_tile_many_parts(fb):
    """75 output tiles on at most 74 clusters, 32 chunks each: the whole-tile
    round matches fp8bq_gemm_wgrad bit for bit (same tiles, same chunk order),
    and the one tile left over is shared by up to 32 clusters, one chunk
    each, while the rest have empty shares; it is within the bound, the same
    on a second call, and the counters are back at zero."""
    rng = np.random.default_rng(41)
    M, N, K = 4096, 768, 6400
    dyqT, xqT = random_codes(rng, (N, M)), random_codes(rng, (K, M))
    sdyT, sxT = random_scales(rng, (M // 128, N)), random_scales(rng, (M // 128, K))
    dev = [to_dev(a) for a in (dyqT, sdyT, xqT, sxT)]
    scratch = fb.wgrad_scratch(dev[0].device)
    dw1 = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    dw2 = torch.empty_like(dw1)
    fb.fp8bq_gemm_wgrad_balanced(*dev, dw1, scratch)
    fb.fp8bq_gemm_wgrad_balanced(*dev, dw2, scratch)
    ref = fb.gemm_wgrad(*dev)
    fb.check()
    torch.cuda.synchronize()
    assert torch.equal(dw1.view(torch.int16), dw2.view(torch.int16))
    nc = _split_counter_bytes(fb)
    assert int(scratch[:nc].sum()) == 0
    # one cluster per two SMs (74 on a 148-SM B300): the tiles left over for
    # the last round are the last tiles in row-major order
    pairs = min(75, torch.cuda.get_device_properties(0).multi_processor_count // 2)
    last = (N // 256 - 1, K // 256 - 1)
    same = torch.ones(75, dtype=torch.bool)
    same[75 - 75 % pairs:] = False
    same = same.view(N // 256, K // 256)
    eq = (dw1.view(torch.int16) == ref.view(torch.int16)).view(N // 256, 256, K // 256, 256).all(3).all(1).cpu()
    assert bool(eq[same].all())
    picks = [(2 * last[0] + a, 2 * last[1] + b) for a in (0, 1) for b in (0, 1)] + [(0, 0), (3, 20)]
    check_gemm_tiles(dw1, oracle.gemm_wgrad_mm, (dyqT, sdyT, xqT, sxT), picks, what="wgrad balanced leftover")


def test_wgrad_balanced_exact_integer_case_is_bit_exact(fb):
    """Small integers and power-of-two scales: every partial sum is exact in
    FP32 however the chunks are grouped, so the balanced split must give the
    oracle's rounding bit for bit, split tiles included."""
    rng = np.random.default_rng(31)
    M, N, K = 1024, 2304, 2304
    dyqT, _ = _integer_operands(rng, (N, M))
    xqT, _ = _integer_operands(rng, (K, M))
    sdyT = np.exp2(rng.integers(-2, 3, size=(M // 128, N))).astype(np.float32)
    sxT = np.exp2(rng.integers(-2, 3, size=(M // 128, K))).astype(np.float32)
    scratch = fb.wgrad_scratch(torch.device("cuda"))
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    fb.fp8bq_gemm_wgrad_balanced(to_dev(dyqT), to_dev(sdyT), to_dev(xqT), to_dev(sxT), dw, scratch)
    fb.check()
    exact, _ = oracle.gemm_wgrad_mm(dyqT, sdyT, xqT, sxT)
    assert np.array_equal(synth.bf16_bits(dw), oracle.bf16_from_double(exact))
