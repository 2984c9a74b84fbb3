"""Plain CPU oracle for the block-scaled FP8 linear layer.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only users.  The product path (the
CUDA library and its Python binding) never imports this package, and this
package never imports the product path.

The arithmetic lives in ``fp8bq_oracle.c`` (plain C, binary32/binary64, no
fast-math, no FMA contraction, no flush-to-zero); this module compiles it with
gcc on first use and wraps it with numpy.  What it follows: the Puro-2B
technical report, section 2 "FP8" (main linear-layer matmuls in FP8 with
DeepSeek-V3-style fine-grained block quantization, sensitive work kept in
BF16/FP32), with the numerical contract of the layer: 1x128 activation and
gradient tiles, 128x128 weight blocks, E4M3 codes, FP32 scale amax/448 (1 for
an all-zero tile), round-half-to-even with saturation at +-448, per-128-chunk
scale promotion in FP32 or better, BF16 output.

Functions and what pins them (tests/test_oracle_*.py):
  e4m3_decode / e4m3_encode     exhaustive 256-code round trip, OCP table
                                values (tests/golden), every midpoint, the
                                independent arithmetic encoder, torch's and
                                ml_dtypes' float8_e4m3fn casts
  quantize_rowwise / _colwise / weight_block
                                amax element -> +-448, zero tile -> s = 1,
                                2^-4 relative error bound, power-of-two
                                equivariance, colwise(X) == rowwise(X^T),
                                qT == q^T, hand-worked tile (tests/golden)
  gemm_fprop / _dgrad / _wgrad  brute-force Python on tiny shapes, float64
                                matmul of the dequantized operands, exact
                                integer cases, single-chunk scale selection
  gemm_tolerance                the acceptance bound: |C - C_exact| <=
                                2e-3 * sum_k |a_k b_k| + 1 BF16 ulp
  f32_ulp / gemm_tolerance_f32  the same bound for FP32 outputs (one FP32 ulp;
                                one more for an add into an FP32 array),
                                pinned against numpy's spacing()
  swiglu / swiglu_check         silu(g) * u in binary64; pinned by g = 0,
                                the identity silu(g) - silu(-g) = g, the
                                limits g -> +-inf, and torch's silu in float64
  mx_exponent / mx_quantize_rowwise / _colwise / mx_gemm
                                the MX variant (power-of-two scale per 1x32
                                block): closed form of the exponent from the
                                binary32 fields, largest element in (224, 448],
                                2^-4 relative bound, exponent equivariance,
                                colwise(X) == rowwise(X^T), a hand-worked block
                                (tests/golden), brute-force Python and float64
                                matmul of the dequantized operands, exact
                                integer products
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8bq_oracle.c")
_SO = os.path.join(_HERE, "libfp8bq_oracle.so")
_lock = threading.Lock()
_lib_handle = None

BF16 = 0
F32 = 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (IEEE arithmetic: no fast-math, no FMA
    contraction).  Rebuilds when the source is newer than the library."""
    with _lock:
        if (not force and os.path.exists(_SO)
                and os.path.getmtime(_SO) >= os.path.getmtime(_SRC)):
            return _SO
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", "-fno-unsafe-math-optimizations",
               "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
        return _SO


def _lib():
    global _lib_handle
    if _lib_handle is None:
        build()
        lib = ctypes.CDLL(_SO)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.fp8bq_oracle_e4m3_decode.restype = ctypes.c_double
        lib.fp8bq_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fp8bq_oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.fp8bq_oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.fp8bq_oracle_e4m3_encode_arith.restype = ctypes.c_uint8
        lib.fp8bq_oracle_e4m3_encode_arith.argtypes = [ctypes.c_float]
        lib.fp8bq_oracle_tile_scale.restype = ctypes.c_float
        lib.fp8bq_oracle_tile_scale.argtypes = [ctypes.c_float]
        for name in ("fp8bq_oracle_quantize_rowwise", "fp8bq_oracle_quantize_colwise"):
            fn = getattr(lib, name)
            fn.restype = None
            fn.argtypes = [ctypes.c_void_p, ctypes.c_int, i64, i64, i64, u8p, f32p]
        lib.fp8bq_oracle_quantize_weight_block.restype = None
        lib.fp8bq_oracle_quantize_weight_block.argtypes = [
            ctypes.c_void_p, ctypes.c_int, i64, i64, i64, u8p, u8p, f32p]
        for name in ("fp8bq_oracle_gemm_fprop", "fp8bq_oracle_gemm_dgrad", "fp8bq_oracle_gemm_wgrad"):
            fn = getattr(lib, name)
            fn.restype = None
            fn.argtypes = [u8p, f32p, u8p, f32p, i64, i64, i64, i64p, i64, i64p, i64, f64p, f64p]
        lib.fp8bq_oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.fp8bq_oracle_bf16_from_double.argtypes = [ctypes.c_double]
        lib.fp8bq_oracle_e4m3_decode_array.argtypes = [u8p, i64, f64p]
        lib.fp8bq_oracle_e4m3_encode_array.argtypes = [f32p, i64, u8p]
        lib.fp8bq_oracle_e4m3_encode_arith_array.argtypes = [f32p, i64, u8p]
        lib.fp8bq_oracle_bf16_from_double_array.argtypes = [f64p, i64, ctypes.POINTER(ctypes.c_uint16)]
        lib.fp8bq_oracle_mx_exponent.restype = ctypes.c_int
        lib.fp8bq_oracle_mx_exponent.argtypes = [ctypes.c_float]
        for name in ("fp8bq_oracle_mx_quantize_rowwise", "fp8bq_oracle_mx_quantize_colwise"):
            fn = getattr(lib, name)
            fn.restype = None
            fn.argtypes = [ctypes.c_void_p, ctypes.c_int, i64, i64, i64, u8p, u8p]
        lib.fp8bq_oracle_mx_gemm.restype = None
        lib.fp8bq_oracle_mx_gemm.argtypes = [u8p, u8p, u8p, u8p, i64, i64, i64, i64p, i64, i64p, i64, f64p, f64p]
        lib.fp8bq_oracle_num_threads.restype = ctypes.c_int
        lib.fp8bq_oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib_handle = lib
    return _lib_handle


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def num_threads() -> int:
    return int(_lib().fp8bq_oracle_num_threads())


def set_num_threads(n: int) -> None:
    _lib().fp8bq_oracle_set_num_threads(int(n))


# --------------------------------------------------------------------------
# Codec
# --------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Exact value of each E4M3 code (OCP FP8 E4M3 definition), float64."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    _lib().fp8bq_oracle_e4m3_decode_array(_ptr(codes, ctypes.c_uint8), codes.size, _ptr(out, ctypes.c_double))
    return out


def e4m3_table() -> np.ndarray:
    """Values of all 256 codes (index = code), float64 (NaN for the two NaN codes)."""
    return e4m3_decode(np.arange(256, dtype=np.uint8))


def e4m3_encode(values) -> np.ndarray:
    """Brute-force nearest-value E4M3 encoding of binary32 values
    (ties to even code, saturating at +-448, sign copied)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _lib().fp8bq_oracle_e4m3_encode_array(_ptr(v, ctypes.c_float), v.size, _ptr(out, ctypes.c_uint8))
    return out


def e4m3_encode_arith(values) -> np.ndarray:
    """Independent arithmetic E4M3 encoder (cross-check of e4m3_encode)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _lib().fp8bq_oracle_e4m3_encode_arith_array(_ptr(v, ctypes.c_float), v.size, _ptr(out, ctypes.c_uint8))
    return out


def tile_scale(amax: float) -> np.float32:
    """s = amax / 448 in binary32, 1 for amax == 0."""
    return np.float32(_lib().fp8bq_oracle_tile_scale(float(np.float32(amax))))


# --------------------------------------------------------------------------
# Quantizers
# --------------------------------------------------------------------------

def _as_input(x: np.ndarray):
    """Accept float32 arrays or BF16 bit patterns (uint16 arrays)."""
    if x.dtype == np.uint16:
        return np.ascontiguousarray(x), BF16
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    raise TypeError(f"oracle input must be float32 or uint16 (bf16 bits), got {x.dtype}")


def quantize_rowwise(x: np.ndarray):
    """1x128 tiles along the last dim.  x [R, C] -> (q [R, C] uint8, s [C/128, R] float32)."""
    x, dt = _as_input(x)
    R, C = x.shape
    assert C % 128 == 0
    q = np.empty((R, C), dtype=np.uint8)
    s = np.empty((C // 128, R), dtype=np.float32)
    _lib().fp8bq_oracle_quantize_rowwise(x.ctypes.data, dt, R, C, C, _ptr(q, ctypes.c_uint8), _ptr(s, ctypes.c_float))
    return q, s


def quantize_colwise(x: np.ndarray):
    """128x1 tiles along the first dim, emitted transposed.
    x [M, C] -> (qT [C, M] uint8, s [M/128, C] float32)."""
    x, dt = _as_input(x)
    M, C = x.shape
    assert M % 128 == 0
    qT = np.empty((C, M), dtype=np.uint8)
    s = np.empty((M // 128, C), dtype=np.float32)
    _lib().fp8bq_oracle_quantize_colwise(x.ctypes.data, dt, M, C, C, _ptr(qT, ctypes.c_uint8), _ptr(s, ctypes.c_float))
    return qT, s


def quantize_weight_block(w: np.ndarray):
    """128x128 blocks.  w [N, K] -> (q [N, K], qT [K, N], s [N/128, K/128])."""
    w, dt = _as_input(w)
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    q = np.empty((N, K), dtype=np.uint8)
    qT = np.empty((K, N), dtype=np.uint8)
    s = np.empty((N // 128, K // 128), dtype=np.float32)
    _lib().fp8bq_oracle_quantize_weight_block(w.ctypes.data, dt, N, K, K, _ptr(q, ctypes.c_uint8),
                                              _ptr(qT, ctypes.c_uint8), _ptr(s, ctypes.c_float))
    return q, qT, s


# --------------------------------------------------------------------------
# GEMMs (binary64)
# --------------------------------------------------------------------------

def _gemm(fn, a, sa, b, sb, M, N, K, rows, cols):
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    val = np.empty((rows.size, cols.size), dtype=np.float64)
    absd = np.empty((rows.size, cols.size), dtype=np.float64)
    fn(_ptr(a, ctypes.c_uint8), _ptr(sa, ctypes.c_float), _ptr(b, ctypes.c_uint8), _ptr(sb, ctypes.c_float),
       M, N, K, _ptr(rows, ctypes.c_int64), rows.size, _ptr(cols, ctypes.c_int64), cols.size,
       _ptr(val, ctypes.c_double), _ptr(absd, ctypes.c_double))
    return val, absd


def gemm_fprop(xq, sx, wq, sw, rows=None, cols=None):
    """Y = Xq Wq^T with per-chunk promotion.  xq [M,K], sx [K/128,M], wq [N,K],
    sw [N/128,K/128].  Returns (Y_exact [len(rows), len(cols)], abs_sum), float64."""
    M, K = xq.shape
    N = wq.shape[0]
    rows = np.arange(M) if rows is None else rows
    cols = np.arange(N) if cols is None else cols
    return _gemm(_lib().fp8bq_oracle_gemm_fprop, xq, sx, wq, sw, M, N, K, rows, cols)


def gemm_dgrad(dyq, sdy, wq, sw, rows=None, cols=None):
    """dX = dYq Wq with per-chunk promotion over the N chunks.  dyq [M,N],
    sdy [N/128,M], wq [N,K] (natural layout), sw [N/128,K/128].
    Returns (dX_exact [len(rows), len(cols)], abs_sum)."""
    M, N = dyq.shape
    K = wq.shape[1]
    rows = np.arange(M) if rows is None else rows
    cols = np.arange(K) if cols is None else cols
    return _gemm(_lib().fp8bq_oracle_gemm_dgrad, dyq, sdy, wq, sw, M, N, K, rows, cols)


def gemm_wgrad(dyqT, sdyT, xqT, sxT, rows=None, cols=None):
    """dW = dYq^T Xq reduced over tokens, from column-wise codes.  dyqT [N,M],
    sdyT [M/128,N], xqT [K,M], sxT [M/128,K].  Returns (dW_exact, abs_sum)."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    rows = np.arange(N) if rows is None else rows
    cols = np.arange(K) if cols is None else cols
    return _gemm(_lib().fp8bq_oracle_gemm_wgrad, dyqT, sdyT, xqT, sxT, M, N, K, rows, cols)


# --------------------------------------------------------------------------
# The same GEMMs with a float64 matmul as the chunk-sum step
# --------------------------------------------------------------------------
#
# gemm_*_mm evaluate the definition above for the requested rows and columns
# with one library step: the 128-term chunk sums P_c come from a float64
# matmul of the decoded codes.  Every product of two E4M3 values and every
# partial sum of one chunk is exact in binary64 (products carry at most 8
# significant bits and span at most 2^36, so 128 of them need at most 51
# bits), so P_c does not depend on the order the library adds in.  The scale
# product (double(sA) * double(sB)), its product with P_c and the sum over
# chunks in chunk order are the same binary64 operations, in the same order,
# as the C routines perform, so the results are bit-identical to gemm_fprop /
# gemm_dgrad / gemm_wgrad (tests/test_oracle_gemm.py checks that) at a
# fraction of the cost on long reductions; the large-shape parity tests use
# them.

def _chunked_product(a, sa, b, sb):
    """a [R, Kr] and b [C, Kr] codes (reduction contiguous), sa [Kr/128, R]
    and sb [Kr/128, C] per-chunk scales (float32).  Returns (value, abs_sum),
    each [R, C] float64: sum_c sa[c] sb[c] P_c and sum_c sa[c] sb[c] |.|_c."""
    table = e4m3_table()
    R, Kr = a.shape
    C = b.shape[0]
    KC = Kr // 128
    av = table[a].reshape(R, KC, 128).transpose(1, 0, 2)
    bv = table[b].reshape(C, KC, 128).transpose(1, 2, 0)
    p = np.matmul(av, bv)                       # [KC, R, C], exact chunk sums
    pa = np.matmul(np.abs(av), np.abs(bv))
    sa64 = np.asarray(sa, dtype=np.float32).astype(np.float64)
    sb64 = np.asarray(sb, dtype=np.float32).astype(np.float64)
    val = np.zeros((R, C), dtype=np.float64)
    absd = np.zeros((R, C), dtype=np.float64)
    for c in range(KC):
        scale = sa64[c][:, None] * sb64[c][None, :]
        val += scale * p[c]
        absd += scale * pa[c]
    return val, absd


def gemm_fprop_mm(xq, sx, wq, sw, rows=None, cols=None):
    """gemm_fprop (same arguments and result) with a float64 matmul step."""
    M, K = xq.shape
    N = wq.shape[0]
    rows = np.arange(M) if rows is None else np.asarray(rows)
    cols = np.arange(N) if cols is None else np.asarray(cols)
    sb = np.asarray(sw, dtype=np.float32)[cols // 128, :].T     # [K/128, len(cols)]
    return _chunked_product(np.asarray(xq)[rows], np.asarray(sx)[:, rows], np.asarray(wq)[cols], sb)


def gemm_dgrad_mm(dyq, sdy, wq, sw, rows=None, cols=None):
    """gemm_dgrad (same arguments: wq in its natural [N, K] layout) with a
    float64 matmul step."""
    M, N = dyq.shape
    K = wq.shape[1]
    rows = np.arange(M) if rows is None else np.asarray(rows)
    cols = np.arange(K) if cols is None else np.asarray(cols)
    b = np.ascontiguousarray(np.asarray(wq)[:, cols].T)          # [len(cols), N]
    sb = np.asarray(sw, dtype=np.float32)[:, cols // 128]        # [N/128, len(cols)]
    return _chunked_product(np.asarray(dyq)[rows], np.asarray(sdy)[:, rows], b, sb)


def gemm_wgrad_mm(dyqT, sdyT, xqT, sxT, rows=None, cols=None):
    """gemm_wgrad (same arguments and result) with a float64 matmul step."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows)
    cols = np.arange(K) if cols is None else np.asarray(cols)
    return _chunked_product(np.asarray(dyqT)[rows], np.asarray(sdyT)[:, rows], np.asarray(xqT)[cols],
                            np.asarray(sxT)[:, cols])


# --------------------------------------------------------------------------
# MX variant (power-of-two scales per 1x32 block)
# --------------------------------------------------------------------------

def mx_exponent(amax: float) -> int:
    """Shared exponent of an MX block: the smallest E >= -127 with
    amax <= 448 * 2^E (the tile scale amax/448 rounded up to a power of two)."""
    return int(_lib().fp8bq_oracle_mx_exponent(float(np.float32(amax))))


def mx_quantize_rowwise(x: np.ndarray):
    """1x32 blocks along the last dim.  x [R, C] -> (q [R, C] uint8,
    e8 [C/128, R, 4] uint8 holding E + 127 of block 4c + t of each row)."""
    x, dt = _as_input(x)
    R, C = x.shape
    assert C % 128 == 0
    q = np.empty((R, C), dtype=np.uint8)
    e8 = np.empty((C // 128, R, 4), dtype=np.uint8)
    _lib().fp8bq_oracle_mx_quantize_rowwise(x.ctypes.data, dt, R, C, C, _ptr(q, ctypes.c_uint8),
                                            _ptr(e8, ctypes.c_uint8))
    return q, e8


def mx_quantize_colwise(x: np.ndarray):
    """32x1 blocks along the first dim, emitted transposed.
    x [M, C] -> (qT [C, M] uint8, e8 [M/128, C, 4] uint8)."""
    x, dt = _as_input(x)
    M, C = x.shape
    assert M % 128 == 0
    qT = np.empty((C, M), dtype=np.uint8)
    e8 = np.empty((M // 128, C, 4), dtype=np.uint8)
    _lib().fp8bq_oracle_mx_quantize_colwise(x.ctypes.data, dt, M, C, C, _ptr(qT, ctypes.c_uint8),
                                            _ptr(e8, ctypes.c_uint8))
    return qT, e8


def mx_gemm(a, ea, b, eb, rows=None, cols=None):
    """D = (2^ea A)(2^eb B)^T for K-major a [I, K], b [J, K] with exponent
    bytes ea [K/128, I, 4], eb [K/128, J, 4].  Returns (D_exact, abs_sum),
    float64, on the requested rows and columns."""
    a = np.ascontiguousarray(a, dtype=np.uint8)
    b = np.ascontiguousarray(b, dtype=np.uint8)
    ea = np.ascontiguousarray(ea, dtype=np.uint8)
    eb = np.ascontiguousarray(eb, dtype=np.uint8)
    I, K = a.shape
    J = b.shape[0]
    rows = np.ascontiguousarray(np.arange(I) if rows is None else rows, dtype=np.int64)
    cols = np.ascontiguousarray(np.arange(J) if cols is None else cols, dtype=np.int64)
    val = np.empty((rows.size, cols.size), dtype=np.float64)
    absd = np.empty((rows.size, cols.size), dtype=np.float64)
    _lib().fp8bq_oracle_mx_gemm(_ptr(a, ctypes.c_uint8), _ptr(ea, ctypes.c_uint8), _ptr(b, ctypes.c_uint8),
                                _ptr(eb, ctypes.c_uint8), I, J, K, _ptr(rows, ctypes.c_int64), rows.size,
                                _ptr(cols, ctypes.c_int64), cols.size, _ptr(val, ctypes.c_double),
                                _ptr(absd, ctypes.c_double))
    return val, absd


# --------------------------------------------------------------------------
# BF16 helpers and the acceptance bound
# --------------------------------------------------------------------------

def bf16_from_double(v) -> np.ndarray:
    """Round binary64 values to BF16 (half to even) directly; returns uint16 bit patterns."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _lib().fp8bq_oracle_bf16_from_double_array(_ptr(v, ctypes.c_double), v.size, _ptr(out, ctypes.c_uint16))
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of BF16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_ulp(ref) -> np.ndarray:
    """One BF16 unit in the last place at |ref|: 2^(max(floor(log2|ref|), -126) - 7); 2^-133 at 0."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    _, ex = np.frexp(ref)                      # ref = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -126)
    ulp = np.ldexp(1.0, e - 7)
    return np.where(ref == 0.0, np.ldexp(1.0, -133), ulp)


def gemm_tolerance(exact, abs_sum) -> np.ndarray:
    """Per-element acceptance bound: 2e-3 * sum_k |a_k b_k| + ulp_bf16(bf16(exact))."""
    ref = bf16_bits_to_f64(bf16_from_double(exact))
    return 2e-3 * np.asarray(abs_sum, dtype=np.float64) + bf16_ulp(ref)


def f32_ulp(ref) -> np.ndarray:
    """One binary32 unit in the last place at |ref|: 2^(max(floor(log2|ref|), -126) - 23); 2^-149 at 0."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    _, ex = np.frexp(ref)
    e = np.maximum(ex - 1, -126)
    return np.where(ref == 0.0, np.ldexp(1.0, -149), np.ldexp(1.0, e - 23))


def gemm_tolerance_f32(exact, abs_sum, base=None) -> np.ndarray:
    """Acceptance bound for an FP32 GEMM output (the Wgrad variant that keeps
    weight gradients in FP32): the same 2e-3 * sum_k |a_k b_k| term, with one
    FP32 ulp of the exact value in place of the BF16 ulp, plus one FP32 ulp of
    the final sum when the product is added into an FP32 array `base`."""
    exact = np.asarray(exact, dtype=np.float64)
    tol = 2e-3 * np.asarray(abs_sum, dtype=np.float64) + f32_ulp(exact)
    if base is not None:
        tol = tol + f32_ulp(np.asarray(base, dtype=np.float64) + exact)
    return tol


def gemm_check_f32(got_f32, exact, abs_sum, base=None):
    """Compare FP32 outputs with the binary64 oracle (optionally base + product).
    Returns (ok: bool, worst_ratio: float, err array)."""
    got = np.asarray(got_f32, dtype=np.float32).astype(np.float64)
    want = np.asarray(exact, dtype=np.float64)
    if base is not None:
        want = np.asarray(base, dtype=np.float32).astype(np.float64) + want
    err = np.abs(got - want)
    tol = gemm_tolerance_f32(exact, abs_sum, None if base is None else np.asarray(base, dtype=np.float32))
    ratio = err / tol
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return bool(np.all(err <= tol) and np.all(np.isfinite(got))), worst, err


def swiglu(g_bits, u_bits) -> np.ndarray:
    """SwiGLU gate of the down projection's input, h = silu(g) * u =
    g * u / (1 + exp(-g)), in binary64 from BF16 inputs (bit patterns).  The
    3.8B architecture list on the n1n.ai page names SwiGLU; the SwiGLU MLP
    workload feeds the down projection with silu(g) * u of the gate/up output."""
    g = bf16_bits_to_f64(g_bits)
    u = bf16_bits_to_f64(u_bits)
    with np.errstate(over="ignore"):
        e = np.exp(-g)
    # The gate is evaluated in FP32 (as a BF16 model evaluates silu): exp(-g)
    # beyond the FP32 range is +inf there, which makes h zero.  For BF16 g
    # this happens exactly for g <= -89 (exp(88.5) is still finite).
    e = np.where(e > np.finfo(np.float32).max, np.inf, e)
    return g * u / (1.0 + e)


def swiglu_check(h_bf16_bits, g_bits, u_bits):
    """A BF16 value of silu(g) * u computed in FP32 and rounded once must lie
    within one BF16 ulp of the binary64 value.  Returns (ok, worst_ratio)."""
    exact = swiglu(g_bits, u_bits)
    got = bf16_bits_to_f64(h_bf16_bits)
    tol = bf16_ulp(exact)
    ratio = np.abs(got - exact) / tol
    return bool(np.all(np.abs(got - exact) <= tol)), float(np.max(ratio)) if ratio.size else 0.0


def gemm_check(got_bf16_bits, exact, abs_sum):
    """Compare BF16 outputs (uint16 bit patterns) with the binary64 oracle.
    Returns (ok: bool, worst_ratio: float, err array)."""
    got = bf16_bits_to_f64(got_bf16_bits)
    err = np.abs(got - exact)
    tol = gemm_tolerance(exact, abs_sum)
    ratio = err / tol
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return bool(np.all(err <= tol) and np.all(np.isfinite(got))), worst, err
