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


def grid_tiles(rng, rows: int, cols: int, n_side: int = 8, tile: int = 128):
    """n_side^2 tiles (a seeded grid of n_side random block rows x n_side
    random block columns, every pairing of them) plus the four corner tiles."""
    rt, ct = rows // tile, cols // tile
    br = rng.choice(rt, size=min(n_side, rt), replace=False)
    bc = rng.choice(ct, size=min(n_side, ct), replace=False)
    picks = {(int(i), int(j)) for i in br for j in bc}
    picks |= {(0, 0), (0, ct - 1), (rt - 1, 0), (rt - 1, ct - 1)}
    return sorted(picks)


class OracleLinear:
    """The oracle's view of one linear layer's inputs X [M, K], W [N, K] and
    dY [M, N] (device tensors, copied to the host slice by slice).

    Row tiles, column tiles and weight blocks are quantized independently of
    each other, so quantizing the 128-row (or 128-column) slice that a block
    of the output needs gives exactly the codes and scales of the whole
    tensor's quantization there; slices are cached.  fprop/dgrad/wgrad return
    the oracle's (exact value, sum |a b|) of one 128 x 128 output tile."""

    def __init__(self, x, w, dy):
        self.x, self.w, self.dy = x, w, dy
        self._cache = {}

    def _get(self, key, fn):
        if key not in self._cache:
            self._cache[key] = fn()
        return self._cache[key]

    @staticmethod
    def _rows(t, b):
        return host_input(t[b * 128:(b + 1) * 128])

    @staticmethod
    def _cols(t, b):
        return host_input(t[:, b * 128:(b + 1) * 128])

    def x_rows(self, b):
        return self._get(("xr", b), lambda: oracle.quantize_rowwise(self._rows(self.x, b)))

    def dy_rows(self, b):
        return self._get(("dyr", b), lambda: oracle.quantize_rowwise(self._rows(self.dy, b)))

    def x_cols(self, b):
        return self._get(("xc", b), lambda: oracle.quantize_colwise(self._cols(self.x, b)))

    def dy_cols(self, b):
        return self._get(("dyc", b), lambda: oracle.quantize_colwise(self._cols(self.dy, b)))

    def w_rows(self, b):
        return self._get(("wr", b), lambda: oracle.quantize_weight_block(self._rows(self.w, b)))

    def w_cols(self, b):
        return self._get(("wc", b), lambda: oracle.quantize_weight_block(self._cols(self.w, b)))

    def fprop(self, bi, bj):
        xq, sx = self.x_rows(bi)
        wq, _, sw = self.w_rows(bj)
        return oracle.gemm_fprop_mm(xq, sx, wq, sw)

    def dgrad(self, bi, bk):
        dyq, sdy = self.dy_rows(bi)
        wq, _, sw = self.w_cols(bk)
        return oracle.gemm_dgrad_mm(dyq, sdy, wq, sw)

    def wgrad(self, bn, bk):
        dyqT, sdyT = self.dy_cols(bn)
        xqT, sxT = self.x_cols(bk)
        return oracle.gemm_wgrad_mm(dyqT, sdyT, xqT, sxT)


def check_output_tile(got_dev: torch.Tensor, bi: int, bj: int, exact, absd, what: str, tile: int = 128):
    """One BF16 output tile of the GPU against the oracle's exact values;
    returns the worst error / tolerance ratio."""
    got = synth.bf16_bits(got_dev[bi * tile:(bi + 1) * tile, bj * tile:(bj + 1) * tile])
    ok, ratio, err = oracle.gemm_check(got, exact, absd)
    if not ok:
        k = np.unravel_index(np.argmax(err / oracle.gemm_tolerance(exact, absd)), err.shape)
        raise AssertionError(f"{what} tile ({bi},{bj}): error {err[k]:.3e} > tolerance at {k} "
                             f"(exact {exact[k]!r}, ratio {ratio:.3g})")
    return ratio
