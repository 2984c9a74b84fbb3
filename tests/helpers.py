"""Shared helpers of the GPU parity tests (no method arithmetic here: the
expected values always come from `oracle`)."""
import numpy as np
import torch

import oracle
from fp8_precision_pretraining_amax_b300 import synth


def host_input(t: torch.Tensor) -> np.ndarray:
    """Host copy of a quantizer input in the oracle's format (bf16 bits or f32)."""
    if t.dtype == torch.bfloat16:
        return synth.bf16_bits(t)
    return t.detach().cpu().contiguous().numpy()


def u32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_codes_equal(got: np.ndarray, want: np.ndarray, what: str):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} codes differ; first at {i}: got {got[i]:#04x} want {want[i]:#04x}")


def assert_scales_equal(got: np.ndarray, want: np.ndarray, what: str):
    if not np.array_equal(u32(got), u32(want)):
        bad = np.argwhere(u32(got) != u32(want))
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} scales differ; first at {i}: got {got[i]!r} want {want[i]!r}")


def random_codes(rng, shape, max_mag=0x7E) -> np.ndarray:
    """Uniformly random finite E4M3 codes (both signs)."""
    mag = rng.integers(0, max_mag + 1, size=shape, dtype=np.uint8)
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8) << 7
    return (mag | sign).astype(np.uint8)


def random_scales(rng, shape) -> np.ndarray:
    """Positive FP32 scales spread over several binades (as amax/448 would be)."""
    return (rng.uniform(1.0, 2.0, size=shape) * np.exp2(rng.integers(-12, 2, size=shape))).astype(np.float32)


def sample_tiles(rng, rows: int, cols: int, n: int, tile: int = 128):
    """Row and column index lists covering n random tile x tile blocks plus
    the four corner blocks (as index sets of the union)."""
    rt = rows // tile
    ct = cols // tile
    picks = {(0, 0), (0, ct - 1), (rt - 1, 0), (rt - 1, ct - 1)}
    while len(picks) < min(n + 4, rt * ct):
        picks.add((int(rng.integers(rt)), int(rng.integers(ct))))
    return sorted(picks)


def to_dev(a: np.ndarray, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def check_gemm_tiles(got_dev: torch.Tensor, oracle_fn, args, picks, tile=128, what=""):
    """Compare BF16 GPU output tiles with the binary64 oracle on the picked tiles.
    Returns the worst error / tolerance ratio."""
    got = synth.bf16_bits(got_dev)
    worst = 0.0
    for (bi, bj) in picks:
        rows = np.arange(bi * tile, (bi + 1) * tile)
        cols = np.arange(bj * tile, (bj + 1) * tile)
        exact, absd = oracle_fn(*args, rows=rows, cols=cols)
        ok, ratio, err = oracle.gemm_check(got[np.ix_(rows, cols)], exact, absd)
        worst = max(worst, ratio)
        if not ok:
            k = np.unravel_index(np.argmax(err / oracle.gemm_tolerance(exact, absd)), err.shape)
            raise AssertionError(
                f"{what} tile ({bi},{bj}): error {err[k]:.3e} > tolerance at {k}; got "
                f"{oracle.bf16_bits_to_f64(got[np.ix_(rows, cols)])[k]!r} exact {exact[k]!r} (ratio {ratio:.3g})")
    return worst
