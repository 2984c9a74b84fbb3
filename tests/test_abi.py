"""The C-ABI library builds, loads without a GPU, exports every entry point
declared in include/fp8bq.h, and rejects bad arguments on the host before it
touches CUDA (these paths need no device)."""
import ctypes
import os
import re

import pytest

from fp8_precision_pretraining_amax_b300 import build as fbuild

HEADER = os.path.join(fbuild.ROOT, "include", "fp8bq.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8bq_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    path = fbuild.build()
    return ctypes.CDLL(path)


def test_header_declares_the_layer_api():
    names = _declared_functions()
    for n in ("fp8bq_quantize_rowwise", "fp8bq_quantize_colwise", "fp8bq_quantize_weight_block",
              "fp8bq_gemm_fprop", "fp8bq_gemm_dgrad", "fp8bq_gemm_wgrad", "fp8bq_check"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol(lib):
    from fp8_precision_pretraining_amax_b300 import fp8bq
    assert sorted(fp8bq.C_FUNCTIONS) == _declared_functions()
    for name in fp8bq.C_FUNCTIONS:
        assert callable(getattr(fp8bq, name))


def test_status_strings(lib):
    lib.fp8bq_status_string.restype = ctypes.c_char_p
    for code in range(8):
        s = lib.fp8bq_status_string(code)
        assert s and s != b"unknown status"
    assert lib.fp8bq_status_string(99) == b"unknown status"


OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE = 0, 1, 2, 3, 4
P = 0x10000  # a 16-byte-aligned fake device address (never dereferenced)


def test_quantizer_argument_errors_are_host_side(lib):
    f = lib.fp8bq_quantize_rowwise
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert f(P, 7, 128, 128, 128, P, P, None) == ERR_DTYPE
    assert f(P, 0, 128, 100, 128, P, P, None) == ERR_SHAPE        # ragged tile
    assert f(P, 0, -1, 128, 128, P, P, None) == ERR_SHAPE
    assert f(P, 0, 4, 256, 128, P, P, None) == ERR_SHAPE          # pitch < width
    assert f(P, 0, 0, 128, 128, None, None, None) == OK           # empty: no-op
    assert f(P, 0, 4, 0, 0, None, None, None) == OK
    assert f(None, 0, 4, 128, 128, P, P, None) == ERR_NULL
    assert f(P + 2, 0, 4, 128, 128, P, P, None) == ERR_ALIGN
    assert f(P, 0, 4, 128, 132, P, P, None) == ERR_ALIGN          # 264-byte pitch
    g = lib.fp8bq_quantize_colwise
    g.restype = ctypes.c_int
    g.argtypes = f.argtypes
    assert g(P, 0, 100, 128, 128, P, P, None) == ERR_SHAPE         # M not a multiple of 128
    assert g(P, 0, 128, 12, 16, P, P, None) == ERR_SHAPE           # C not a multiple of 8
    assert g(P, 0, 128, 128, 128, P, None, P) == ERR_NULL
    h = lib.fp8bq_quantize_weight_block
    h.restype = ctypes.c_int
    h.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert h(P, 0, 128, 192, 192, P, P, P, None) == ERR_SHAPE
    assert h(P, 0, 128, 128, 128, P, P + 8, P, None) == ERR_ALIGN
    assert h(P, 2, 128, 128, 128, P, P, P, None) == ERR_DTYPE


def test_gemm_argument_errors_are_host_side(lib):
    # (M, N, K) with an empty OUTPUT dimension: a host-side no-op.  (An empty
    # reduction dimension is not: it writes zeros on the device.)
    empty_out = {"fp8bq_gemm_fprop": (0, 128, 128), "fp8bq_gemm_dgrad": (0, 128, 128),
                 "fp8bq_gemm_wgrad": (128, 0, 128)}
    for name in ("fp8bq_gemm_fprop", "fp8bq_gemm_dgrad", "fp8bq_gemm_wgrad"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
        assert f(P, P, P, P, P, 128, 128, 100, None) == ERR_SHAPE
        assert f(P, P, P, P, P, 128, 192, 128, None) == ERR_SHAPE
        assert f(P, P, P, P, P, -128, 128, 128, None) == ERR_SHAPE
        assert f(P, P, P, P, P, *empty_out[name], None) == OK
        assert f(P, P, P, P, None, 128, 128, 128, None) == ERR_NULL
        assert f(None, P, P, P, P, 128, 128, 128, None) == ERR_NULL
        assert f(P, P, P + 4, P, P, 128, 128, 128, None) == ERR_ALIGN
        assert f(P, P, P, P, P + 2, 128, 128, 128, None) == ERR_ALIGN


def test_fused_and_fp32_entry_points_reject_bad_arguments_on_the_host(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    rc = lib.fp8bq_quantize_rowcol
    rc.restype, rc.argtypes = i32, [vp, i32, i64, i64, i64, vp, vp, vp, vp, vp]
    assert rc(P, 0, 128, 200, 200, P, P, P, P, None) == ERR_SHAPE      # C not a multiple of 128
    assert rc(P, 0, 100, 128, 128, P, P, P, P, None) == ERR_SHAPE      # M not a multiple of 128
    assert rc(P, 0, 128, 128, 128, P, P, None, P, None) == ERR_NULL
    assert rc(P, 0, 128, 128, 128, P, P, P + 4, P, None) == ERR_ALIGN
    assert rc(P, 3, 128, 128, 128, P, P, P, P, None) == ERR_DTYPE
    assert rc(P, 0, 0, 128, 128, None, None, None, None, None) == OK
    sq = lib.fp8bq_swiglu_quantize
    sq.restype, sq.argtypes = i32, [vp, i64, i64, i64, vp, vp, vp, vp, vp, vp]
    assert sq(P, 128, 128, 200, None, P, P, P, P, None) == ERR_SHAPE   # ldgu < 2F
    assert sq(P, 128, 192, 384, None, P, P, P, P, None) == ERR_SHAPE   # F not a multiple of 128
    assert sq(P, 128, 128, 256, None, P, None, P, P, None) == ERR_NULL
    assert sq(P, 128, 128, 256, P + 2, P, P, P, P, None) == ERR_ALIGN  # optional H misaligned
    assert sq(P, 128, 128, 260, None, P, P, P, P, None) == ERR_ALIGN   # 520-byte pitch
    assert sq(P, 0, 128, 256, None, None, None, None, None, None) == OK
    wf = lib.fp8bq_gemm_wgrad_f32
    wf.restype, wf.argtypes = i32, [vp] * 5 + [i64] * 3 + [i32, vp]
    assert wf(P, P, P, P, P, 128, 128, 128, 2, None) == ERR_SHAPE      # accumulate must be 0 or 1
    assert wf(P, P, P, P, P, 100, 128, 128, 0, None) == ERR_SHAPE
    assert wf(P, P, P, P, None, 128, 128, 128, 1, None) == ERR_NULL
    assert wf(P, P, P, P, P + 8, 128, 128, 128, 0, None) == ERR_ALIGN
    wb = lib.fp8bq_gemm_wgrad_balanced
    wb.restype, wb.argtypes = i32, [vp] * 5 + [i64] * 3 + [vp, i64, vp]
    assert wb(P, P, P, P, P, 128, 128, 128, None, 1 << 30, None) == ERR_NULL   # scratch required
    assert wb(P, P, P, P, P, 128, 128, 128, P + 4, 1 << 30, None) == ERR_ALIGN
    assert wb(P, P, P, P, P, 128, 128, 128, P, -1, None) == ERR_SHAPE
    assert wb(P, P, P, P, P, 100, 128, 128, P, 1 << 30, None) == ERR_SHAPE      # M not a multiple of 128
    assert wb(P, P, P, P, None, 128, 128, 128, P, 1 << 30, None) == ERR_NULL
    ws = lib.fp8bq_gemm_wgrad_balanced_static
    ws.restype, ws.argtypes = i32, [vp] * 5 + [i64] * 3 + [vp]
    assert ws(P, P, P, P, None, 128, 128, 128, None) == ERR_NULL
    sb = lib.fp8bq_gemm_wgrad_scratch_bytes
    sb.restype, sb.argtypes = i32, [vp]
    assert sb(None) == ERR_NULL
    fq = lib.fp8bq_gemm_fprop_q
    fq.restype, fq.argtypes = i32, [vp] * 7 + [i64] * 3 + [vp]
    assert fq(P, P, P, P, None, None, P, 128, 128, 128, None) == ERR_NULL   # codes required
    assert fq(P, P, P, P, None, P, None, 128, 128, 128, None) == ERR_NULL   # scales required
    assert fq(P, P, P, P, None, P, P, 128, 100, 128, None) == ERR_SHAPE
    assert fq(P, P, P, P, None, P + 4, P, 128, 128, 128, None) == ERR_ALIGN
    assert fq(P, P, P, P, None, P, P, 0, 128, 128, None) == OK               # empty output


def test_mx_entry_points_reject_bad_arguments_on_the_host(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    for name in ("fp8bq_mx_quantize_rowwise", "fp8bq_mx_quantize_colwise"):
        f = getattr(lib, name)
        f.restype, f.argtypes = i32, [vp, i32, i64, i64, i64, vp, vp, vp]
        assert f(P, 5, 128, 128, 128, P, P, None) == ERR_DTYPE
        assert f(P, 0, 128, 96, 96, P, P, None) == ERR_SHAPE         # C not a multiple of 128
        assert f(P, 0, 128, 256, 128, P, P, None) == ERR_SHAPE       # pitch < width
        assert f(P, 0, 0, 128, 128, None, None, None) == OK          # empty: no-op
        assert f(P, 0, 128, 128, 128, P, None, None) == ERR_NULL
        assert f(P, 0, 128, 128, 128, P, P + 4, None) == ERR_ALIGN
        assert f(P, 1, 128, 128, 130, P, P, None) == ERR_ALIGN       # 520-byte pitch
    g = lib.fp8bq_mx_quantize_colwise
    assert g(P, 0, 96, 128, 128, P, P, None) == ERR_SHAPE            # M not a multiple of 128
    rc = lib.fp8bq_mx_quantize_rowcol
    rc.restype, rc.argtypes = i32, [vp, i32, i64, i64, i64, vp, vp, vp, vp, vp]
    assert rc(P, 0, 128, 200, 200, P, P, P, P, None) == ERR_SHAPE
    assert rc(P, 0, 96, 128, 128, P, P, P, P, None) == ERR_SHAPE
    assert rc(P, 0, 128, 128, 128, P, P, None, P, None) == ERR_NULL
    assert rc(P, 0, 128, 128, 128, P, P, P, P + 2, None) == ERR_ALIGN
    assert rc(P, 9, 128, 128, 128, P, P, P, P, None) == ERR_DTYPE
    assert rc(P, 0, 0, 128, 128, None, None, None, None, None) == OK
    m = lib.fp8bq_mx_gemm
    m.restype, m.argtypes = i32, [vp] * 5 + [i64] * 3 + [vp]
    assert m(P, P, P, P, P, 128, 128, 100, None) == ERR_SHAPE
    assert m(P, P, P, P, P, 128, 192, 128, None) == ERR_SHAPE
    assert m(P, P, P, P, P, 0, 128, 128, None) == OK                # empty output
    assert m(P, P, P, P, None, 128, 128, 128, None) == ERR_NULL
    assert m(P, None, P, P, P, 128, 128, 128, None) == ERR_NULL
    assert m(P, P, P, P + 4, P, 128, 128, 128, None) == ERR_ALIGN


def test_grouped_weight_quantizer_rejects_bad_arguments_on_the_host(lib):
    from fp8_precision_pretraining_amax_b300.fp8bq import FP8BQWeight
    f = lib.fp8bq_quantize_weight_blocks
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(FP8BQWeight), ctypes.c_int, ctypes.c_int, ctypes.c_void_p]

    def entries(*ws):
        arr = (FP8BQWeight * len(ws))()
        for e, (w, N, K, ldw, q, qT, s) in zip(arr, ws):
            e.w, e.N, e.K, e.ldw, e.q, e.qT, e.s = w, N, K, ldw, q, qT, s
        return arr
    good = (P, 128, 256, 256, P, P, P)
    assert f(None, 0, 0, None) == OK                       # nothing to do
    assert f(None, 1, 0, None) == ERR_NULL
    assert f(entries(good), -1, 0, None) == ERR_SHAPE
    assert f(entries(good), 1, 7, None) == ERR_DTYPE
    assert f(entries(good, (P, 100, 256, 256, P, P, P)), 2, 0, None) == ERR_SHAPE   # N % 128
    assert f(entries(good, (P, 128, 256, 255, P, P, P)), 2, 0, None) == ERR_SHAPE   # pitch < width
    assert f(entries(good, (0, 128, 256, 256, P, P, P)), 2, 0, None) == ERR_NULL    # no input
    assert f(entries(good, (P, 128, 256, 256, P, None, None)), 2, 0, None) == ERR_NULL   # no scales
    assert f(entries(good, (P + 8, 128, 256, 256, P, P, P)), 2, 0, None) == ERR_ALIGN
    assert f(entries(good, (P, 128, 256, 260, P, P, P)), 2, 0, None) == ERR_ALIGN    # BF16 pitch 520 bytes
    assert f(entries((P, 0, 256, 256, 0, 0, 0), (0, 128, 0, 0, 0, 0, 0)), 2, 0, None) == OK   # only empty weights
