"""Pins of the oracle's quantizers (1x128 row tiles, 128x1 column tiles,
128x128 weight blocks) against properties the quantization rule fixes.

Rule: s = amax/448 in FP32 (s = 1 for an all-zero tile), code = E4M3
round-half-to-even of the correctly rounded FP32 quotient x/s, saturating at
+-448 (fine-grained block quantization of the Puro-2B report, section 2 "FP8",
after DeepSeek-V3).
"""
import os

import numpy as np
import pytest
import torch

import oracle
from fp8_precision_pretraining_amax_b300 import synth
from tests.conftest import GOLDEN


def _bf16_bits(t):
    return synth.bf16_bits(t)


def _f32_of_bits(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def _load_worked_tile():
    path = os.path.join(GOLDEN, "rowwise_tile_worked.txt")
    x = np.zeros(128, dtype=np.float32)
    codes = np.zeros(128, dtype=np.uint8)
    scale = None
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] == "scale":
            scale = float(parts[1])
            continue
        i = int(parts[0])
        x[i] = np.float32(float(parts[1]))
        codes[i] = int(parts[3], 16)
    return x, codes, scale


def test_worked_tile_fp32_and_bf16():
    x, codes, scale = _load_worked_tile()
    q, s = oracle.quantize_rowwise(x.reshape(1, 128))
    assert s[0, 0] == np.float32(scale)
    assert np.array_equal(q[0], codes), [(i, hex(a), hex(b)) for i, (a, b) in enumerate(zip(q[0], codes)) if a != b]
    xb = _bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    assert np.array_equal(_f32_of_bits(xb), x), "worked tile is BF16-exact"
    qb, sb = oracle.quantize_rowwise(xb.reshape(1, 128))
    assert sb[0, 0] == np.float32(scale) and np.array_equal(qb[0], codes)


def _check_tile_properties(x_tiles, q_tiles, s_tiles):
    """x_tiles [T,128] float32, q_tiles [T,128], s_tiles [T]."""
    amax = np.max(np.abs(x_tiles), axis=1)
    expect_s = np.where(amax == 0, np.float32(1), (amax / np.float32(448)).astype(np.float32))
    assert np.array_equal(s_tiles, expect_s)
    # the element that attains amax encodes to +-448
    idx = np.argmax(np.abs(x_tiles), axis=1)
    top = q_tiles[np.arange(len(idx)), idx]
    nz = amax > 0
    assert np.all((top[nz] & 0x7F) == 0x7E)
    # all-zero tiles: codes are signed zeros
    assert np.all((q_tiles[~nz] & 0x7F) == 0)
    # error bounds: 2^-4 relative in the normal range, s*2^-10 absolute below it
    deq = oracle.e4m3_decode(q_tiles) * s_tiles[:, None].astype(np.float64)
    x64 = x_tiles.astype(np.float64)
    err = np.abs(deq - x64)
    y = np.abs(x64) / s_tiles[:, None]
    normal = y >= 2.0 ** -6
    rel_bound = 2.0 ** -4 * np.abs(x64) * (1 + 2.0 ** -19)
    abs_bound = s_tiles[:, None].astype(np.float64) * 2.0 ** -10 * (1 + 2.0 ** -19)
    assert np.all(err[normal] <= rel_bound[normal])
    assert np.all(err[~normal] <= np.broadcast_to(abs_bound, err.shape)[~normal])
    # sign is copied
    assert np.all(((q_tiles & 0x80) != 0) == np.signbit(x_tiles))


def test_rowwise_tiny_fp32_properties():
    lin = synth.tiny()
    x = lin.x.numpy()
    q, s = oracle.quantize_rowwise(x)
    R, C = x.shape
    xt = x.reshape(R, C // 128, 128).transpose(1, 0, 2).reshape(-1, 128)
    qt = q.reshape(R, C // 128, 128).transpose(1, 0, 2).reshape(-1, 128)
    _check_tile_properties(xt, qt, s.reshape(-1))


def test_rowwise_bf16_with_outliers_and_zero_tiles():
    gen = synth.generator(5)
    xb = synth.activations(64, 1024, gen)
    xb[3, 128:256] = 0
    xb[5, :128] = -0.0
    xbits = _bf16_bits(xb)
    q, s = oracle.quantize_rowwise(xbits)
    x = _f32_of_bits(xbits)
    R, C = x.shape
    xt = x.reshape(R, C // 128, 128).transpose(1, 0, 2).reshape(-1, 128)
    qt = q.reshape(R, C // 128, 128).transpose(1, 0, 2).reshape(-1, 128)
    _check_tile_properties(xt, qt, s.reshape(-1))
    assert s[1, 3] == 1.0 and np.all(q[3, 128:256] == 0)
    assert s[0, 5] == 1.0 and np.all(q[5, :128] == 0x80)


@pytest.mark.parametrize("j", [-7, -1, 3, 9])
def test_power_of_two_equivariance(j):
    gen = synth.generator(6)
    x = synth.gaussian((32, 512), 1.0, gen).numpy()
    q0, s0 = oracle.quantize_rowwise(x)
    q1, s1 = oracle.quantize_rowwise((x * np.float32(2.0 ** j)).astype(np.float32))
    assert np.array_equal(q0, q1)
    assert np.array_equal(s1, (s0 * np.float32(2.0 ** j)).astype(np.float32))


def test_scale_is_correctly_rounded_quotient():
    # amax values whose quotient by 448 is inexact: s must be the RNE binary32 quotient.
    amax = np.array([3.0, 1.0, 0.1, 1e-3, 12345.678, 2.0 ** -120], dtype=np.float32)
    for a in amax:
        want = np.float32(np.float64(a) / 448.0)  # binary64 quotient then one rounding = RNE quotient
        assert oracle.tile_scale(a) == want


def test_colwise_equals_rowwise_of_transpose():
    gen = synth.generator(7)
    xb = synth.activations(384, 256, gen)
    xbits = _bf16_bits(xb)
    qT, s_col = oracle.quantize_colwise(xbits)
    q_row, s_row = oracle.quantize_rowwise(np.ascontiguousarray(xbits.T))
    assert np.array_equal(qT, q_row)
    assert np.array_equal(s_col, s_row)


def test_weight_block_properties():
    gen = synth.generator(8)
    wb = synth.weight(256, 384, gen)
    wb[128:256, 0:128] = 0
    wbits = _bf16_bits(wb)
    q, qT, s = oracle.quantize_weight_block(wbits)
    assert np.array_equal(qT, q.T)
    w = _f32_of_bits(wbits)
    for nb in range(2):
        for kb in range(3):
            blk = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            amax = np.max(np.abs(blk))
            want = np.float32(1) if amax == 0 else np.float32(amax / np.float32(448))
            assert s[nb, kb] == want
            # a block whose rows are quantized with the block's scale gives the same
            # codes as quantizing it as 128 row tiles that each contain the block amax
            qb = q[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            if amax > 0:
                i, jx = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
                assert qb[i, jx] & 0x7F == 0x7E
    assert s[1, 0] == 1.0 and np.all(q[128:256, 0:128] == 0)
    # flat property check with the block scale broadcast
    tiles = w.reshape(2, 128, 3, 128).transpose(0, 2, 1, 3).reshape(6, -1)
    qt = q.reshape(2, 128, 3, 128).transpose(0, 2, 1, 3).reshape(6, -1)
    deq = oracle.e4m3_decode(qt) * s.reshape(6, 1)
    err = np.abs(deq - tiles)
    y = np.abs(tiles) / s.reshape(6, 1)
    normal = y >= 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(tiles[normal]) * (1 + 2.0 ** -19))


def test_weight_block_equals_rowwise_when_block_amax_is_in_every_row():
    # Put the block amax into every row of the block: then each 1x128 row tile
    # has the block's amax, and row-wise codes/scales must equal the block ones.
    gen = synth.generator(9)
    w = synth.gaussian((128, 256), 0.02, gen).numpy()
    w[:, 5] = 1.0
    w[:, 130] = -1.0
    q_blk, _, s_blk = oracle.quantize_weight_block(w)
    q_row, s_row = oracle.quantize_rowwise(w)
    assert np.array_equal(q_blk, q_row)
    assert np.all(s_row[0] == s_blk[0, 0]) and np.all(s_row[1] == s_blk[0, 1])


def test_rowwise_respects_pitch_free_layout_and_scale_layout():
    # s is chunk-major: s[t, r] is the scale of row r's t-th tile
    x = np.zeros((3, 384), dtype=np.float32)
    for r in range(3):
        for t in range(3):
            x[r, t * 128 + 7] = 448.0 * 2.0 ** (r - t)
    q, s = oracle.quantize_rowwise(x)
    for r in range(3):
        for t in range(3):
            assert s[t, r] == np.float32(2.0 ** (r - t))
            assert q[r, t * 128 + 7] == 0x7E
