"""GPU parity of the three quantizers with the oracle: codes and scales must
match bit for bit (the quantization rule has exactly one correct answer)."""
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_precision_pretraining_amax_b300 import synth
from tests.conftest import GOLDEN
from tests.helpers import assert_codes_equal, assert_scales_equal, host_input

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fb():
    from fp8_precision_pretraining_amax_b300 import fp8bq
    return fp8bq


def _rowwise_parity(fb, x: torch.Tensor, what: str):
    q, s = fb.quantize_rowwise(x)
    fb.check()
    qo, so = oracle.quantize_rowwise(host_input(x))
    assert_codes_equal(q.cpu().numpy(), qo, what + " codes")
    assert_scales_equal(s.cpu().numpy(), so, what + " scales")


def _special_bf16(rows: int, cols: int, seed: int) -> torch.Tensor:
    """Tiles that hit the edges of the rule: zero and -0 tiles, subnormal-only
    tiles (FP32 scale itself subnormal), huge values, exact E4M3 midpoints."""
    gen = synth.generator(seed)
    x = synth.gaussian((rows, cols), 1.0, gen)
    t = oracle.e4m3_table()[:0x7F]
    mids = torch.from_numpy(((t[:-1] + t[1:]) / 2).astype(np.float32))
    for r in range(rows):
        kind = r % 9
        seg = slice(0, 128)
        if kind == 0:
            x[r, seg] = 0.0
        elif kind == 1:
            x[r, seg] = -0.0
        elif kind == 2:
            x[r, seg] *= 2.0 ** -130           # BF16 subnormals: s is an FP32 subnormal
        elif kind == 3:
            x[r, seg] *= 1e37                  # near the top of the BF16 range
        elif kind == 4:
            x[r, :126] = mids * torch.where(torch.arange(126) % 2 == 0, 1.0, -1.0)
            x[r, 126] = 448.0                  # s = 1: every midpoint is a tie
            x[r, 127] = -0.0
        elif kind == 5:
            x[r, seg] = 2.0 ** -133            # a constant tile at the smallest BF16 subnormal
        elif kind == 6:
            x[r, seg] *= 2.0 ** -120
    return x.to(torch.bfloat16)


def test_rowwise_worked_tile(fb):
    x = np.zeros(128, dtype=np.float32)
    for line in open(os.path.join(GOLDEN, "rowwise_tile_worked.txt")):
        p = line.split()
        if p and p[0].isdigit():
            x[int(p[0])] = float(p[1])
    for dt in (torch.float32, torch.bfloat16):
        _rowwise_parity(fb, torch.from_numpy(x).reshape(1, 128).to(dt).cuda(), f"worked tile {dt}")


def test_rowwise_tiny_fp32(fb):
    _rowwise_parity(fb, synth.tiny().x.cuda(), "tiny A fp32")


@pytest.mark.parametrize("R,C", [(1, 128), (3, 256), (333, 1152), (1024, 2048)])
def test_rowwise_bf16_activations(fb, R, C):
    gen = synth.generator(100 + R)
    _rowwise_parity(fb, synth.activations(R, C, gen).cuda(), f"rowwise {R}x{C}")


def test_rowwise_special_values(fb):
    _rowwise_parity(fb, _special_bf16(72, 384, 5).cuda(), "rowwise specials")
    xf = _special_bf16(36, 256, 6).float()
    xf[0, :128] *= 2.0 ** -20                  # FP32-only magnitudes
    _rowwise_parity(fb, xf.cuda(), "rowwise specials fp32")


def test_rowwise_pitched_input(fb):
    gen = synth.generator(7)
    big = synth.activations(96, 768, gen).cuda()
    x = big[:, 128:640]                        # ldx = 768 > C = 512
    q, s = fb.quantize_rowwise(x)
    qo, so = oracle.quantize_rowwise(host_input(x.contiguous()))
    assert_codes_equal(q.cpu().numpy(), qo, "pitched codes")
    assert_scales_equal(s.cpu().numpy(), so, "pitched scales")


def test_rowwise_empty_and_ragged(fb):
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = fb.quantize_rowwise(x)
    assert q.shape == (0, 256) and s.shape == (2, 0)
    bad = torch.zeros((4, 200), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fb.Fp8bqError) as e:
        fb.fp8bq_quantize_rowwise(bad, torch.empty((4, 200), dtype=torch.uint8, device="cuda"),
                                  torch.empty((1, 4), dtype=torch.float32, device="cuda"))
    assert e.value.status == fb.ERR_SHAPE


def _colwise_parity(fb, x: torch.Tensor, what: str):
    qT, s = fb.quantize_colwise(x)
    fb.check()
    qo, so = oracle.quantize_colwise(host_input(x))
    assert_codes_equal(qT.cpu().numpy(), qo, what + " codes")
    assert_scales_equal(s.cpu().numpy(), so, what + " scales")


@pytest.mark.parametrize("M,C", [(128, 8), (384, 136), (256, 1024), (1024, 2056)])
def test_colwise_bf16(fb, M, C):
    gen = synth.generator(200 + C)
    _colwise_parity(fb, synth.activations(M, C, gen).cuda(), f"colwise {M}x{C}")


def test_colwise_grads_and_fp32(fb):
    gen = synth.generator(8)
    _colwise_parity(fb, synth.grads(512, 384, gen).cuda(), "colwise dY")
    _colwise_parity(fb, synth.gaussian((256, 72), 0.3, gen).cuda(), "colwise fp32")


def test_colwise_special_values(fb):
    x = _special_bf16(384, 256, 9)
    _colwise_parity(fb, x.t().contiguous().cuda(), "colwise specials")


def test_colwise_equals_rowwise_of_transpose_on_gpu(fb):
    gen = synth.generator(10)
    x = synth.activations(512, 768, gen).cuda()
    qT, s_col = fb.quantize_colwise(x)
    q_row, s_row = fb.quantize_rowwise(x.t().contiguous())
    assert torch.equal(qT, q_row) and torch.equal(s_col, s_row)


def _weight_parity(fb, w: torch.Tensor, what: str, transpose=True):
    q, qT, s = fb.quantize_weight_block(w, transpose=transpose)
    fb.check()
    qo, qTo, so = oracle.quantize_weight_block(host_input(w))
    assert_codes_equal(q.cpu().numpy(), qo, what + " codes")
    if transpose:
        assert_codes_equal(qT.cpu().numpy(), qTo, what + " transposed codes")
    assert_scales_equal(s.cpu().numpy(), so, what + " scales")


def test_weight_block_tiny_fp32(fb):
    _weight_parity(fb, synth.tiny().w.cuda(), "tiny W fp32")


@pytest.mark.parametrize("N,K", [(128, 128), (384, 640), (4096, 2048)])
def test_weight_block_bf16(fb, N, K):
    gen = synth.generator(300 + N)
    w = synth.weight(N, K, gen)
    w[:128, :128] = 0.0
    _weight_parity(fb, w.cuda(), f"weight {N}x{K}")


def test_weight_block_without_transpose_and_specials(fb):
    _weight_parity(fb, _special_bf16(256, 384, 11).cuda(), "weight specials", transpose=False)
    _weight_parity(fb, _special_bf16(256, 384, 12).cuda(), "weight specials T")


@pytest.mark.slow
def test_full_size_quantizers_sampled(fb):
    """Full-size tensors of the 3.8B layer / up-projection backward, checked on
    sampled rows (row-wise), sampled columns (column-wise) and in full for the
    weight; the launch configuration is the one the benchmark uses."""
    rng = np.random.default_rng(13)
    gen = synth.generator(14, "cuda")
    dy = synth.grads(16384, 6144, gen, "cuda")
    x = synth.activations(32768, 3072, gen, "cuda")
    w = synth.weight(16384, 3072, gen, "cuda")
    # row-wise on dY: 64 sampled rows with all their tiles
    q, s = fb.quantize_rowwise(dy)
    rows = np.sort(rng.choice(16384, 64, replace=False))
    rows[0], rows[-1] = 0, 16383
    qo, so = oracle.quantize_rowwise(host_input(dy[torch.from_numpy(rows).cuda()]))
    assert_codes_equal(q[torch.from_numpy(rows).cuda()].cpu().numpy(), qo, "full rowwise codes")
    assert_scales_equal(s[:, torch.from_numpy(rows).cuda()].cpu().numpy(), so, "full rowwise scales")
    # column-wise on X: 32 sampled columns over all 32768 tokens
    qT, sc = fb.quantize_colwise(x)
    cols = np.sort(rng.choice(3072, 32, replace=False))
    cols[0], cols[-1] = 0, 3071
    xc = x[:, torch.from_numpy(cols).cuda()].contiguous()
    qTo, sco = oracle.quantize_colwise(host_input(xc))
    assert_codes_equal(qT[torch.from_numpy(cols).cuda()].cpu().numpy(), qTo, "full colwise codes")
    assert_scales_equal(sc[:, torch.from_numpy(cols).cuda()].cpu().numpy(), sco, "full colwise scales")
    # weight block in full (50M elements)
    _weight_parity(fb, w, "full weight 16384x3072")


# ---------------------------------------------------------------------------
# fused row-wise + column-wise pass
# ---------------------------------------------------------------------------

def _rowcol_parity(fb, x: torch.Tensor, what: str):
    q, s_row, qT, s_col = fb.quantize_rowcol(x)
    fb.check()
    xh = host_input(x)
    qo, so = oracle.quantize_rowwise(xh)
    qTo, sco = oracle.quantize_colwise(xh)
    assert_codes_equal(q.cpu().numpy(), qo, what + " row-wise codes")
    assert_scales_equal(s_row.cpu().numpy(), so, what + " row-wise scales")
    assert_codes_equal(qT.cpu().numpy(), qTo, what + " column-wise codes")
    assert_scales_equal(s_col.cpu().numpy(), sco, what + " column-wise scales")


@pytest.mark.parametrize("M,C", [(128, 128), (384, 640), (1024, 2048)])
def test_rowcol_bf16(fb, M, C):
    gen = synth.generator(400 + M + C)
    _rowcol_parity(fb, synth.activations(M, C, gen).cuda(), f"rowcol {M}x{C}")


def test_rowcol_grads_fp32_and_specials(fb):
    gen = synth.generator(15)
    _rowcol_parity(fb, synth.grads(512, 768, gen).cuda(), "rowcol dY")
    _rowcol_parity(fb, synth.gaussian((256, 384), 0.3, gen).cuda(), "rowcol fp32")
    _rowcol_parity(fb, _special_bf16(384, 256, 16).cuda(), "rowcol specials")
    _rowcol_parity(fb, _special_bf16(128, 384, 17).float().cuda(), "rowcol specials fp32")


def test_rowcol_matches_separate_kernels_and_pitch(fb):
    gen = synth.generator(18)
    big = synth.activations(640, 1152, gen).cuda()
    x = big[:, 128:1024]                               # ldx = 1152 > C = 896
    q, s_row, qT, s_col = fb.quantize_rowcol(x)
    q2, s2 = fb.quantize_rowwise(x)
    qT2, sc2 = fb.quantize_colwise(x)
    assert torch.equal(q, q2) and torch.equal(s_row, s2)
    assert torch.equal(qT, qT2) and torch.equal(s_col, sc2)


def test_rowcol_rejects_partial_tiles(fb):
    x = torch.zeros((128, 200), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fb.Fp8bqError) as e:
        fb.fp8bq_quantize_rowcol(x, torch.empty((128, 200), dtype=torch.uint8, device="cuda"),
                                 torch.empty((1, 128), dtype=torch.float32, device="cuda"),
                                 torch.empty((200, 128), dtype=torch.uint8, device="cuda"),
                                 torch.empty((1, 200), dtype=torch.float32, device="cuda"))
    assert e.value.status == fb.ERR_SHAPE


# ---------------------------------------------------------------------------
# the quotient x / s near its hardest cases
# ---------------------------------------------------------------------------

def _every_bf16_amax(seed: int) -> torch.Tensor:
    """One 1x128 tile per positive finite BF16 value a (32640 rows, padded):
    element 0 is a, the rest are random BF16 values of magnitude <= a with
    random signs, so every scale a BF16 tile can have is exercised."""
    rng = np.random.default_rng(seed)
    a = np.arange(1, 0x7F80, dtype=np.uint32)                # positive finite BF16 bit patterns
    a = np.concatenate([a, a[-1:]])                           # 32640 rows = 255 x 128
    frac = rng.random((a.size, 127))
    mags = np.floor(frac * (a[:, None] + 1)).astype(np.uint32)  # bit patterns in [0, a]
    signs = rng.integers(0, 2, size=mags.shape, dtype=np.uint32) << 15
    bits = np.concatenate([a[:, None], mags | signs], axis=1).astype(np.uint16)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)


def test_every_bf16_tile_scale(fb):
    """Codes and scales for tiles of every possible BF16 amax, through the
    row-wise, fused and column-wise kernels."""
    x = _every_bf16_amax(19).cuda()
    _rowwise_parity(fb, x, "every amax rowwise")
    _rowcol_parity(fb, x[:, :128].contiguous(), "every amax rowcol")
    _colwise_parity(fb, x.t().contiguous(), "every amax colwise")


def test_fp32_quotients_next_to_rounding_midpoints(fb):
    """FP32 inputs x = RN(m s) and its FP32 neighbours for every midpoint m
    between adjacent E4M3 values and many scales s: x / s then lies within an
    ulp or two of a rounding boundary, where only the correctly rounded
    quotient gives the right code."""
    rng = np.random.default_rng(20)
    t = oracle.e4m3_table()[:0x7F].astype(np.float64)
    mids = ((t[:-1] + t[1:]) / 2)                              # 126 midpoints, all < 448
    rows = []
    for _ in range(64):
        amax = np.float32(rng.uniform(1, 2) * 2.0 ** rng.integers(-60, 60))
        s = np.float32(amax / np.float32(448.0))
        body = (mids * np.float64(s)).astype(np.float32)
        for nudge in (-1, 0, 1):
            v = body.view(np.uint32).astype(np.int64) + nudge
            row = np.concatenate([[amax], v.astype(np.uint32).view(np.float32)[:126], [-0.0]]).astype(np.float32)
            row[1:127] *= np.where(rng.random(126) < 0.5, -1, 1).astype(np.float32)
            rows.append(row)
    x = torch.from_numpy(np.stack(rows))                       # 192 x 128 FP32
    _rowwise_parity(fb, x.cuda(), "midpoints rowwise")
    _rowcol_parity(fb, x[:128].contiguous().cuda(), "midpoints rowcol")
    _colwise_parity(fb, x.t().contiguous().cuda(), "midpoints colwise")
    _weight_parity(fb, x[:128].contiguous().cuda(), "midpoints weight")


# ---------------------------------------------------------------------------
# SwiGLU gate fused into the down projection's quantizer
# ---------------------------------------------------------------------------

def _swiglu_case(fb, gu: torch.Tensor, F: int, what: str):
    h, q, s_row, qT, s_col = fb.swiglu_quantize(gu, F, keep_h=True)
    _, q2, s_row2, qT2, s_col2 = fb.swiglu_quantize(gu, F, keep_h=False)
    fb.check()
    g_bits = synth.bf16_bits(gu[:, :F].contiguous())
    u_bits = synth.bf16_bits(gu[:, F:2 * F].contiguous())
    h_bits = synth.bf16_bits(h)
    ok, worst = oracle.swiglu_check(h_bits, g_bits, u_bits)
    assert ok, f"{what}: H off by {worst:.3g} BF16 ulps"
    # codes and scales are exactly those of the H the kernel formed
    qo, so = oracle.quantize_rowwise(h_bits)
    qTo, sco = oracle.quantize_colwise(h_bits)
    assert_codes_equal(q.cpu().numpy(), qo, what + " row-wise codes")
    assert_scales_equal(s_row.cpu().numpy(), so, what + " row-wise scales")
    assert_codes_equal(qT.cpu().numpy(), qTo, what + " column-wise codes")
    assert_scales_equal(s_col.cpu().numpy(), sco, what + " column-wise scales")
    assert torch.equal(q, q2) and torch.equal(qT, qT2) and torch.equal(s_row, s_row2) and torch.equal(s_col, s_col2)
    # and the same as quantizing that H with the fused row+column pass
    q3, s3, qT3, sc3 = fb.quantize_rowcol(h)
    assert torch.equal(q, q3) and torch.equal(qT, qT3) and torch.equal(s_row, s3) and torch.equal(s_col, sc3)


@pytest.mark.parametrize("M,F", [(128, 128), (384, 640), (1024, 2048)])
def test_swiglu_quantize(fb, M, F):
    gen = synth.generator(500 + M + F)
    gu = (synth.gaussian((M, 2 * F), 1.5, gen)).to(torch.bfloat16).cuda()
    _swiglu_case(fb, gu, F, f"swiglu {M}x{F}")


def test_swiglu_quantize_extremes_and_pitch(fb):
    """Large |g| (FP32 exp overflow, silu -> 0 or g), zeros, and an input
    whose row pitch (3F) is larger than the 2F columns g and u occupy."""
    gen = synth.generator(71)
    M, F = 256, 384
    big = synth.gaussian((M, 3 * F), 1.0, gen)
    big[:, :F][::3] *= 60.0
    big[0, :] = 0.0
    big[1, :F] = -1e4
    gu = big.to(torch.bfloat16).cuda()
    _swiglu_case(fb, gu, F, "swiglu extremes")             # ldgu = 3F > 2F


def _weight_items(ws, transpose_mask):
    items = []
    for w, t in zip(ws, transpose_mask):
        N, K = w.shape
        items.append((w, torch.empty((N, K), dtype=torch.uint8, device=w.device),
                      torch.empty((K, N), dtype=torch.uint8, device=w.device) if t else None,
                      torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)))
    return items


def test_grouped_weight_quantizer_equals_one_call_per_weight(fb):
    """The grouped launch writes, for every weight, exactly what the per-weight
    quantizer writes (the 3.8B layer's four weights, one with the transposed
    codes skipped, plus a special-value weight), and the oracle agrees."""
    gen = synth.generator(310, "cuda")
    ws = [synth.weight(N, K, gen, "cuda") for _, K, N in synth.LAYER_3P8B]
    ws.append(_special_bf16(256, 384, 13).cuda())
    mask = [True, False, True, True, True]
    items = _weight_items(ws, mask)
    fb.fp8bq_quantize_weight_blocks(items)
    fb.check()
    for (w, q, qT, s), t in zip(items, mask):
        q1, qT1, s1 = fb.quantize_weight_block(w, transpose=t)
        fb.check()
        assert torch.equal(q, q1) and torch.equal(s, s1)
        if t:
            assert torch.equal(qT, qT1)
    w, q, qT, s = items[-1]
    qo, qTo, so = oracle.quantize_weight_block(host_input(w))
    assert_codes_equal(q.cpu().numpy(), qo, "grouped specials codes")
    assert_codes_equal(qT.cpu().numpy(), qTo, "grouped specials transposed codes")
    assert_scales_equal(s.cpu().numpy(), so, "grouped specials scales")


def test_grouped_weight_quantizer_long_list_fp32_and_empty(fb):
    """More entries than one launch takes (processed in several launches),
    FP32 weights, and an empty list."""
    gen = synth.generator(311, "cuda")
    ws = [synth.gaussian((128 * (1 + i % 3), 128 * (1 + i % 2)), 0.02, gen, "cuda") for i in range(19)]
    items = _weight_items(ws, [i % 2 == 0 for i in range(19)])
    fb.fp8bq_quantize_weight_blocks(items)
    fb.fp8bq_quantize_weight_blocks([])
    fb.check()
    for i, (w, q, qT, s) in enumerate(items):
        qo, qTo, so = oracle.quantize_weight_block(host_input(w))
        assert_codes_equal(q.cpu().numpy(), qo, f"fp32 weight {i}")
        assert_scales_equal(s.cpu().numpy(), so, f"fp32 weight {i} scales")
        if qT is not None:
            assert_codes_equal(qT.cpu().numpy(), qTo, f"fp32 weight {i} transposed")
