"""Python binding of libfp8bq (block-scaled FP8 linear layer for B300).

Argument marshalling only: every function passes torch tensors' device
pointers, sizes and the current CUDA stream to the C ABI of include/fp8bq.h
and raises on a non-OK status.  All arithmetic runs in the library's CUDA
kernels; there is no CPU or library fallback.  Importing this module fails
loudly when libfp8bq.so has not been built.

Functions carry the C names (fp8bq_quantize_rowwise, ...) and take every
buffer explicitly; the unprefixed forms (quantize_rowwise, gemm_fprop, ...)
allocate the outputs with torch and return them.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfp8bq.so")

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_DEVICE, ERR_CUDA, ERR_TIMEOUT = range(8)
BF16, F32 = 0, 1

#: Names of the C-ABI entry points declared in include/fp8bq.h.
C_FUNCTIONS = (
    "fp8bq_quantize_rowwise", "fp8bq_quantize_colwise", "fp8bq_quantize_rowcol", "fp8bq_swiglu_quantize",
    "fp8bq_quantize_weight_block", "fp8bq_quantize_weight_blocks", "fp8bq_gemm_fprop", "fp8bq_gemm_fprop_q", "fp8bq_gemm_dgrad",
    "fp8bq_gemm_wgrad", "fp8bq_gemm_wgrad_balanced", "fp8bq_gemm_wgrad_scratch_bytes",
    "fp8bq_gemm_wgrad_balanced_static", "fp8bq_gemm_wgrad_f32",
    "fp8bq_mx_quantize_rowwise", "fp8bq_mx_quantize_colwise",
    "fp8bq_mx_quantize_rowcol", "fp8bq_mx_gemm", "fp8bq_check", "fp8bq_status_string", "fp8bq_selftest_wait_timeout",
)


class FP8BQWeight(ctypes.Structure):
    """One entry of fp8bq_quantize_weight_blocks (struct fp8bq_weight)."""
    _fields_ = [("w", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("ldw", ctypes.c_int64),
                ("q", ctypes.c_void_p), ("qT", ctypes.c_void_p), ("s", ctypes.c_void_p)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"libfp8bq.so is not built ({_LIB_PATH}); run "
            "`python -m fp8_precision_pretraining_amax_b300.build` (needs nvcc with sm_103a)")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    sig = {
        "fp8bq_quantize_rowwise": [vp, i32, i64, i64, i64, vp, vp, vp],
        "fp8bq_quantize_colwise": [vp, i32, i64, i64, i64, vp, vp, vp],
        "fp8bq_quantize_rowcol": [vp, i32, i64, i64, i64, vp, vp, vp, vp, vp],
        "fp8bq_swiglu_quantize": [vp, i64, i64, i64, vp, vp, vp, vp, vp, vp],
        "fp8bq_quantize_weight_block": [vp, i32, i64, i64, i64, vp, vp, vp, vp],
        "fp8bq_quantize_weight_blocks": [ctypes.POINTER(FP8BQWeight), i32, i32, vp],
        "fp8bq_gemm_fprop": [vp, vp, vp, vp, vp, i64, i64, i64, vp],
        "fp8bq_gemm_fprop_q": [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, vp],
        "fp8bq_gemm_dgrad": [vp, vp, vp, vp, vp, i64, i64, i64, vp],
        "fp8bq_gemm_wgrad": [vp, vp, vp, vp, vp, i64, i64, i64, vp],
        "fp8bq_gemm_wgrad_balanced": [vp, vp, vp, vp, vp, i64, i64, i64, vp, i64, vp],
        "fp8bq_gemm_wgrad_scratch_bytes": [ctypes.POINTER(i64)],
        "fp8bq_gemm_wgrad_balanced_static": [vp, vp, vp, vp, vp, i64, i64, i64, vp],
        "fp8bq_gemm_wgrad_f32": [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp],
        "fp8bq_mx_quantize_rowwise": [vp, i32, i64, i64, i64, vp, vp, vp],
        "fp8bq_mx_quantize_colwise": [vp, i32, i64, i64, i64, vp, vp, vp],
        "fp8bq_mx_quantize_rowcol": [vp, i32, i64, i64, i64, vp, vp, vp, vp, vp],
        "fp8bq_mx_gemm": [vp, vp, vp, vp, vp, i64, i64, i64, vp],
        "fp8bq_check": [vp],
        "fp8bq_selftest_wait_timeout": [i64, vp],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = i32
    lib.fp8bq_status_string.argtypes = [i32]
    lib.fp8bq_status_string.restype = ctypes.c_char_p
    return lib


lib = _load()


class Fp8bqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def status_string(status: int) -> str:
    return lib.fp8bq_status_string(int(status)).decode()


def _raise(status: int, where: str) -> None:
    if status != OK:
        raise Fp8bqError(status, where)


def _stream(t: Optional[torch.Tensor] = None) -> int:
    dev = t.device if t is not None and t.is_cuda else None
    return torch.cuda.current_stream(dev).cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"input must be bfloat16 or float32, got {t.dtype}")


def _need(t: torch.Tensor, dtype, shape, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _rows_input(x: torch.Tensor, name: str) -> int:
    if x.dim() != 2 or not x.is_cuda:
        raise ValueError(f"{name} must be a 2-D CUDA tensor")
    if x.stride(1) != 1:
        raise ValueError(f"{name} must have unit inner stride")
    return x.stride(0) if x.shape[0] > 1 else x.shape[1]


# ---------------------------------------------------------------------------
# C-named entry points (caller supplies every buffer)
# ---------------------------------------------------------------------------

def fp8bq_quantize_rowwise(x: torch.Tensor, q: torch.Tensor, s: torch.Tensor) -> None:
    """x [R, C] bf16/f32 -> q [R, C] uint8 codes, s [C/128, R] f32 scales."""
    ldx = _rows_input(x, "x")
    R, C = x.shape
    _need(q, torch.uint8, (R, C), "q")
    _need(s, torch.float32, (C // 128, R), "s")
    with torch.cuda.device(x.device):
        _raise(lib.fp8bq_quantize_rowwise(_ptr(x), _dtype_code(x), R, C, ldx, _ptr(q), _ptr(s), _stream(x)),
               "fp8bq_quantize_rowwise")


def fp8bq_quantize_colwise(x: torch.Tensor, qT: torch.Tensor, s: torch.Tensor) -> None:
    """x [M, C] bf16/f32 -> qT [C, M] uint8 codes (128x1 tiles), s [M/128, C] f32."""
    ldx = _rows_input(x, "x")
    M, C = x.shape
    _need(qT, torch.uint8, (C, M), "qT")
    _need(s, torch.float32, (M // 128, C), "s")
    with torch.cuda.device(x.device):
        _raise(lib.fp8bq_quantize_colwise(_ptr(x), _dtype_code(x), M, C, ldx, _ptr(qT), _ptr(s), _stream(x)),
               "fp8bq_quantize_colwise")


def fp8bq_quantize_rowcol(x: torch.Tensor, q: torch.Tensor, s_row: torch.Tensor, qT: torch.Tensor,
                          s_col: torch.Tensor) -> None:
    """x [M, C] -> row-wise q [M, C], s_row [C/128, M] and column-wise qT [C, M], s_col [M/128, C]
    in one pass over x (same bits as fp8bq_quantize_rowwise + fp8bq_quantize_colwise)."""
    ldx = _rows_input(x, "x")
    M, C = x.shape
    _need(q, torch.uint8, (M, C), "q")
    _need(s_row, torch.float32, (C // 128, M), "s_row")
    _need(qT, torch.uint8, (C, M), "qT")
    _need(s_col, torch.float32, (M // 128, C), "s_col")
    with torch.cuda.device(x.device):
        _raise(lib.fp8bq_quantize_rowcol(_ptr(x), _dtype_code(x), M, C, ldx, _ptr(q), _ptr(s_row), _ptr(qT),
                                         _ptr(s_col), _stream(x)), "fp8bq_quantize_rowcol")


def fp8bq_swiglu_quantize(gu: torch.Tensor, h: Optional[torch.Tensor], q: torch.Tensor, s_row: torch.Tensor,
                          qT: torch.Tensor, s_col: torch.Tensor) -> None:
    """gu [M, >= 2F] bf16 (g = columns [0, F), u = [F, 2F)) -> H = bf16(silu(g) u) (h, optional) and its
    row-wise q [M, F], s_row [F/128, M] and column-wise qT [F, M], s_col [M/128, F] codes and scales."""
    if gu.dtype != torch.bfloat16:
        raise TypeError("gu must be bfloat16")
    ld = _rows_input(gu, "gu")
    M = gu.shape[0]
    F = q.shape[1]
    if gu.shape[1] < 2 * F:
        raise ValueError(f"gu needs at least {2 * F} columns, got {gu.shape[1]}")
    if h is not None:
        _need(h, torch.bfloat16, (M, F), "h")
    _need(q, torch.uint8, (M, F), "q")
    _need(s_row, torch.float32, (F // 128, M), "s_row")
    _need(qT, torch.uint8, (F, M), "qT")
    _need(s_col, torch.float32, (M // 128, F), "s_col")
    with torch.cuda.device(gu.device):
        _raise(lib.fp8bq_swiglu_quantize(_ptr(gu), M, F, ld, _ptr(h), _ptr(q), _ptr(s_row), _ptr(qT), _ptr(s_col),
                                         _stream(gu)), "fp8bq_swiglu_quantize")


def fp8bq_quantize_weight_block(w: torch.Tensor, q: torch.Tensor, qT: Optional[torch.Tensor],
                                s: torch.Tensor) -> None:
    """w [N, K] -> q [N, K], qT [K, N] (or None), s [N/128, K/128]."""
    ldw = _rows_input(w, "w")
    N, K = w.shape
    _need(q, torch.uint8, (N, K), "q")
    if qT is not None:
        _need(qT, torch.uint8, (K, N), "qT")
    _need(s, torch.float32, (N // 128, K // 128), "s")
    with torch.cuda.device(w.device):
        _raise(lib.fp8bq_quantize_weight_block(_ptr(w), _dtype_code(w), N, K, ldw, _ptr(q), _ptr(qT), _ptr(s),
                                               _stream(w)), "fp8bq_quantize_weight_block")


def fp8bq_quantize_weight_blocks(items) -> None:
    """Several weights in one launch: items = [(w, q, qT or None, s), ...],
    each as fp8bq_quantize_weight_block takes them, all of one dtype and on
    one device."""
    items = list(items)
    if not items:
        return
    entries = (FP8BQWeight * len(items))()
    dev, dt = items[0][0].device, items[0][0].dtype
    for e, (w, q, qT, s) in zip(entries, items):
        if w.device != dev or w.dtype != dt:
            raise ValueError("fp8bq_quantize_weight_blocks: every weight must share device and dtype")
        ldw = _rows_input(w, "w")
        N, K = w.shape
        _need(q, torch.uint8, (N, K), "q")
        if qT is not None:
            _need(qT, torch.uint8, (K, N), "qT")
        _need(s, torch.float32, (N // 128, K // 128), "s")
        e.w, e.N, e.K, e.ldw, e.q, e.qT, e.s = _ptr(w), N, K, ldw, _ptr(q), _ptr(qT), _ptr(s)
    with torch.cuda.device(dev):
        _raise(lib.fp8bq_quantize_weight_blocks(entries, len(items), _dtype_code(items[0][0]), _stream(items[0][0])),
               "fp8bq_quantize_weight_blocks")


def fp8bq_gemm_fprop(xq, sx, wq, sw, y) -> None:
    """Y [M, N] bf16 = Xq Wq^T with per-chunk scales sx [K/128, M], sw [N/128, K/128]."""
    M, K = xq.shape
    N = wq.shape[0]
    _need(xq, torch.uint8, (M, K), "xq")
    _need(sx, torch.float32, (K // 128, M), "sx")
    _need(wq, torch.uint8, (N, K), "wq")
    _need(sw, torch.float32, (N // 128, K // 128), "sw")
    _need(y, torch.bfloat16, (M, N), "y")
    with torch.cuda.device(y.device):
        _raise(lib.fp8bq_gemm_fprop(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), _ptr(y), M, N, K, _stream(y)),
               "fp8bq_gemm_fprop")


def fp8bq_gemm_fprop_q(xq, sx, wq, sw, y, yq, sy) -> None:
    """Fprop (as fp8bq_gemm_fprop; y may be None) whose epilogue also writes the row-wise
    codes yq [M, N] uint8 and scales sy [N/128, M] of the BF16 output."""
    M, K = xq.shape
    N = wq.shape[0]
    _need(xq, torch.uint8, (M, K), "xq")
    _need(sx, torch.float32, (K // 128, M), "sx")
    _need(wq, torch.uint8, (N, K), "wq")
    _need(sw, torch.float32, (N // 128, K // 128), "sw")
    if y is not None:
        _need(y, torch.bfloat16, (M, N), "y")
    _need(yq, torch.uint8, (M, N), "yq")
    _need(sy, torch.float32, (N // 128, M), "sy")
    with torch.cuda.device(yq.device):
        _raise(lib.fp8bq_gemm_fprop_q(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), _ptr(y), _ptr(yq), _ptr(sy), M, N, K,
                                      _stream(yq)), "fp8bq_gemm_fprop_q")


def fp8bq_gemm_dgrad(dyq, sdy, wqT, sw, dx) -> None:
    """dX [M, K] bf16 = dYq Wq with dyq [M, N], sdy [N/128, M], wqT [K, N], sw [N/128, K/128]."""
    M, N = dyq.shape
    K = wqT.shape[0]
    _need(dyq, torch.uint8, (M, N), "dyq")
    _need(sdy, torch.float32, (N // 128, M), "sdy")
    _need(wqT, torch.uint8, (K, N), "wqT")
    _need(sw, torch.float32, (N // 128, K // 128), "sw")
    _need(dx, torch.bfloat16, (M, K), "dx")
    with torch.cuda.device(dx.device):
        _raise(lib.fp8bq_gemm_dgrad(_ptr(dyq), _ptr(sdy), _ptr(wqT), _ptr(sw), _ptr(dx), M, N, K, _stream(dx)),
               "fp8bq_gemm_dgrad")


def fp8bq_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw) -> None:
    """dW [N, K] bf16 = dY^T X over tokens: dyqT [N, M], sdyT [M/128, N], xqT [K, M], sxT [M/128, K]."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    _need(dyqT, torch.uint8, (N, M), "dyqT")
    _need(sdyT, torch.float32, (M // 128, N), "sdyT")
    _need(xqT, torch.uint8, (K, M), "xqT")
    _need(sxT, torch.float32, (M // 128, K), "sxT")
    _need(dw, torch.bfloat16, (N, K), "dw")
    with torch.cuda.device(dw.device):
        _raise(lib.fp8bq_gemm_wgrad(_ptr(dyqT), _ptr(sdyT), _ptr(xqT), _ptr(sxT), _ptr(dw), M, N, K, _stream(dw)),
               "fp8bq_gemm_wgrad")


def fp8bq_gemm_wgrad_scratch_bytes(device=None) -> int:
    """Bytes of scratch fp8bq_gemm_wgrad_balanced needs on `device` (default: current)."""
    n = ctypes.c_int64(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _raise(lib.fp8bq_gemm_wgrad_scratch_bytes(ctypes.byref(n)), "fp8bq_gemm_wgrad_scratch_bytes")
    return int(n.value)


def wgrad_scratch(device) -> torch.Tensor:
    """A zeroed scratch buffer for fp8bq_gemm_wgrad_balanced on `device`."""
    return torch.zeros(max(16, fp8bq_gemm_wgrad_scratch_bytes(device)), dtype=torch.uint8, device=device)


def fp8bq_gemm_wgrad_balanced(dyqT, sdyT, xqT, sxT, dw, scratch) -> None:
    """fp8bq_gemm_wgrad with the balanced work split; scratch from wgrad_scratch (calls that share it
    must be ordered on one stream)."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    _need(dyqT, torch.uint8, (N, M), "dyqT")
    _need(sdyT, torch.float32, (M // 128, N), "sdyT")
    _need(xqT, torch.uint8, (K, M), "xqT")
    _need(sxT, torch.float32, (M // 128, K), "sxT")
    _need(dw, torch.bfloat16, (N, K), "dw")
    _need(scratch, torch.uint8, (scratch.numel(),), "scratch")
    with torch.cuda.device(dw.device):
        _raise(lib.fp8bq_gemm_wgrad_balanced(_ptr(dyqT), _ptr(sdyT), _ptr(xqT), _ptr(sxT), _ptr(dw), M, N, K,
                                             _ptr(scratch), scratch.numel(), _stream(dw)),
               "fp8bq_gemm_wgrad_balanced")


def fp8bq_gemm_wgrad_balanced_static(dyqT, sdyT, xqT, sxT, dw) -> None:
    """fp8bq_gemm_wgrad_balanced with the library's own scratch (no buffer argument); calls on one device
    must be ordered on one stream."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    _need(dyqT, torch.uint8, (N, M), "dyqT")
    _need(sdyT, torch.float32, (M // 128, N), "sdyT")
    _need(xqT, torch.uint8, (K, M), "xqT")
    _need(sxT, torch.float32, (M // 128, K), "sxT")
    _need(dw, torch.bfloat16, (N, K), "dw")
    with torch.cuda.device(dw.device):
        _raise(lib.fp8bq_gemm_wgrad_balanced_static(_ptr(dyqT), _ptr(sdyT), _ptr(xqT), _ptr(sxT), _ptr(dw), M, N, K,
                                                    _stream(dw)), "fp8bq_gemm_wgrad_balanced_static")


def fp8bq_gemm_wgrad_f32(dyqT, sdyT, xqT, sxT, dw, accumulate: bool = False) -> None:
    """dW [N, K] float32 = dY^T X over tokens (accumulate: dW += dY^T X), operands as fp8bq_gemm_wgrad."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    _need(dyqT, torch.uint8, (N, M), "dyqT")
    _need(sdyT, torch.float32, (M // 128, N), "sdyT")
    _need(xqT, torch.uint8, (K, M), "xqT")
    _need(sxT, torch.float32, (M // 128, K), "sxT")
    _need(dw, torch.float32, (N, K), "dw")
    with torch.cuda.device(dw.device):
        _raise(lib.fp8bq_gemm_wgrad_f32(_ptr(dyqT), _ptr(sdyT), _ptr(xqT), _ptr(sxT), _ptr(dw), M, N, K,
                                        1 if accumulate else 0, _stream(dw)), "fp8bq_gemm_wgrad_f32")


def fp8bq_mx_quantize_rowwise(x: torch.Tensor, q: torch.Tensor, e8: torch.Tensor) -> None:
    """MX variant.  x [R, C] bf16/f32 -> q [R, C] uint8 codes, e8 [C/128, R, 4] uint8 exponents (E + 127)."""
    ldx = _rows_input(x, "x")
    R, C = x.shape
    _need(q, torch.uint8, (R, C), "q")
    _need(e8, torch.uint8, (C // 128, R, 4), "e8")
    with torch.cuda.device(x.device):
        _raise(lib.fp8bq_mx_quantize_rowwise(_ptr(x), _dtype_code(x), R, C, ldx, _ptr(q), _ptr(e8), _stream(x)),
               "fp8bq_mx_quantize_rowwise")


def fp8bq_mx_quantize_colwise(x: torch.Tensor, qT: torch.Tensor, e8: torch.Tensor) -> None:
    """MX variant.  x [M, C] bf16/f32 -> qT [C, M] uint8 codes (32x1 blocks), e8 [M/128, C, 4] uint8."""
    ldx = _rows_input(x, "x")
    M, C = x.shape
    _need(qT, torch.uint8, (C, M), "qT")
    _need(e8, torch.uint8, (M // 128, C, 4), "e8")
    with torch.cuda.device(x.device):
        _raise(lib.fp8bq_mx_quantize_colwise(_ptr(x), _dtype_code(x), M, C, ldx, _ptr(qT), _ptr(e8), _stream(x)),
               "fp8bq_mx_quantize_colwise")


def fp8bq_mx_quantize_rowcol(x: torch.Tensor, q: torch.Tensor, e8: torch.Tensor, qT: torch.Tensor,
                             e8T: torch.Tensor) -> None:
    """MX variant, both layouts from one read: x [M, C] -> q [M, C], e8 [C/128, M, 4], qT [C, M], e8T [M/128, C, 4]."""
    ldx = _rows_input(x, "x")
    M, C = x.shape
    _need(q, torch.uint8, (M, C), "q")
    _need(e8, torch.uint8, (C // 128, M, 4), "e8")
    _need(qT, torch.uint8, (C, M), "qT")
    _need(e8T, torch.uint8, (M // 128, C, 4), "e8T")
    with torch.cuda.device(x.device):
        _raise(lib.fp8bq_mx_quantize_rowcol(_ptr(x), _dtype_code(x), M, C, ldx, _ptr(q), _ptr(e8), _ptr(qT),
                                            _ptr(e8T), _stream(x)), "fp8bq_mx_quantize_rowcol")


def fp8bq_mx_gemm(a, ea, b, eb, d) -> None:
    """MX variant.  d [I, J] bf16 = (2^ea a)(2^eb b)^T: a [I, K], ea [K/128, I, 4], b [J, K], eb [K/128, J, 4]."""
    I, K = a.shape
    J = b.shape[0]
    _need(a, torch.uint8, (I, K), "a")
    _need(ea, torch.uint8, (K // 128, I, 4), "ea")
    _need(b, torch.uint8, (J, K), "b")
    _need(eb, torch.uint8, (K // 128, J, 4), "eb")
    _need(d, torch.bfloat16, (I, J), "d")
    with torch.cuda.device(d.device):
        _raise(lib.fp8bq_mx_gemm(_ptr(a), _ptr(ea), _ptr(b), _ptr(eb), _ptr(d), I, J, K, _stream(d)),
               "fp8bq_mx_gemm")


def fp8bq_check(device=None) -> None:
    """Synchronize the current stream and raise if a kernel reported a device-side timeout."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _raise(lib.fp8bq_check(torch.cuda.current_stream(dev).cuda_stream), "fp8bq_check")


def fp8bq_selftest_wait_timeout(limit_ns: int, device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _raise(lib.fp8bq_selftest_wait_timeout(int(limit_ns), torch.cuda.current_stream(dev).cuda_stream),
               "fp8bq_selftest_wait_timeout")


def fp8bq_status_string(status: int) -> str:
    return status_string(status)


# ---------------------------------------------------------------------------
# Allocating forms
# ---------------------------------------------------------------------------

def quantize_rowwise(x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    s = torch.empty((C // 128, R), dtype=torch.float32, device=x.device)
    fp8bq_quantize_rowwise(x, q, s)
    return q, s


def quantize_colwise(x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    M, C = x.shape
    qT = torch.empty((C, M), dtype=torch.uint8, device=x.device)
    s = torch.empty((M // 128, C), dtype=torch.float32, device=x.device)
    fp8bq_quantize_colwise(x, qT, s)
    return qT, s


def quantize_rowcol(x: torch.Tensor):
    """Returns (q, s_row, qT, s_col)."""
    M, C = x.shape
    q = torch.empty((M, C), dtype=torch.uint8, device=x.device)
    s_row = torch.empty((C // 128, M), dtype=torch.float32, device=x.device)
    qT = torch.empty((C, M), dtype=torch.uint8, device=x.device)
    s_col = torch.empty((M // 128, C), dtype=torch.float32, device=x.device)
    fp8bq_quantize_rowcol(x, q, s_row, qT, s_col)
    return q, s_row, qT, s_col


def swiglu_quantize(gu: torch.Tensor, F: int, keep_h: bool = False):
    """Returns (h or None, q, s_row, qT, s_col) for H = silu(g) * u, g = gu[:, :F], u = gu[:, F:2F]."""
    M = gu.shape[0]
    d = gu.device
    h = torch.empty((M, F), dtype=torch.bfloat16, device=d) if keep_h else None
    q = torch.empty((M, F), dtype=torch.uint8, device=d)
    s_row = torch.empty((F // 128, M), dtype=torch.float32, device=d)
    qT = torch.empty((F, M), dtype=torch.uint8, device=d)
    s_col = torch.empty((M // 128, F), dtype=torch.float32, device=d)
    fp8bq_swiglu_quantize(gu, h, q, s_row, qT, s_col)
    return h, q, s_row, qT, s_col


def quantize_weight_block(w: torch.Tensor, transpose: bool = True):
    N, K = w.shape
    q = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    qT = torch.empty((K, N), dtype=torch.uint8, device=w.device) if transpose else None
    s = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    fp8bq_quantize_weight_block(w, q, qT, s)
    return q, qT, s


def gemm_fprop(xq, sx, wq, sw) -> torch.Tensor:
    y = torch.empty((xq.shape[0], wq.shape[0]), dtype=torch.bfloat16, device=xq.device)
    fp8bq_gemm_fprop(xq, sx, wq, sw, y)
    return y


def gemm_fprop_q(xq, sx, wq, sw, keep_bf16: bool = True):
    """Returns (y or None, yq, sy)."""
    M, N = xq.shape[0], wq.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device) if keep_bf16 else None
    yq = torch.empty((M, N), dtype=torch.uint8, device=xq.device)
    sy = torch.empty((N // 128, M), dtype=torch.float32, device=xq.device)
    fp8bq_gemm_fprop_q(xq, sx, wq, sw, y, yq, sy)
    return y, yq, sy


def gemm_dgrad(dyq, sdy, wqT, sw) -> torch.Tensor:
    dx = torch.empty((dyq.shape[0], wqT.shape[0]), dtype=torch.bfloat16, device=dyq.device)
    fp8bq_gemm_dgrad(dyq, sdy, wqT, sw, dx)
    return dx


def gemm_wgrad(dyqT, sdyT, xqT, sxT) -> torch.Tensor:
    dw = torch.empty((dyqT.shape[0], xqT.shape[0]), dtype=torch.bfloat16, device=dyqT.device)
    fp8bq_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw)
    return dw


def gemm_wgrad_f32(dyqT, sdyT, xqT, sxT) -> torch.Tensor:
    dw = torch.empty((dyqT.shape[0], xqT.shape[0]), dtype=torch.float32, device=dyqT.device)
    fp8bq_gemm_wgrad_f32(dyqT, sdyT, xqT, sxT, dw)
    return dw


def mx_quantize_rowwise(x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """MX variant: returns (q [R, C], e8 [C/128, R, 4])."""
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    e8 = torch.empty((C // 128, R, 4), dtype=torch.uint8, device=x.device)
    fp8bq_mx_quantize_rowwise(x, q, e8)
    return q, e8


def mx_quantize_colwise(x: torch.Tensor) -> Tuple[torch.Tensor, torch.Tensor]:
    """MX variant: returns (qT [C, M], e8 [M/128, C, 4])."""
    M, C = x.shape
    qT = torch.empty((C, M), dtype=torch.uint8, device=x.device)
    e8 = torch.empty((M // 128, C, 4), dtype=torch.uint8, device=x.device)
    fp8bq_mx_quantize_colwise(x, qT, e8)
    return qT, e8


def mx_quantize_rowcol(x: torch.Tensor):
    """MX variant: returns (q, e8, qT, e8T)."""
    M, C = x.shape
    q = torch.empty((M, C), dtype=torch.uint8, device=x.device)
    e8 = torch.empty((C // 128, M, 4), dtype=torch.uint8, device=x.device)
    qT = torch.empty((C, M), dtype=torch.uint8, device=x.device)
    e8T = torch.empty((M // 128, C, 4), dtype=torch.uint8, device=x.device)
    fp8bq_mx_quantize_rowcol(x, q, e8, qT, e8T)
    return q, e8, qT, e8T


def mx_gemm(a, ea, b, eb) -> torch.Tensor:
    d = torch.empty((a.shape[0], b.shape[0]), dtype=torch.bfloat16, device=a.device)
    fp8bq_mx_gemm(a, ea, b, eb, d)
    return d


check = fp8bq_check
selftest_wait_timeout = fp8bq_selftest_wait_timeout
