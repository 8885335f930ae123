"""CPU oracle for MX block-scaled quantize / dequantize / block_matmul.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The product library neither imports nor
calls this package, and this package imports nothing from the product.

The arithmetic lives in ``mx_oracle.c`` (plain C, binary64); this module only
marshals numpy arrays into it.  Element formats use the same numbering as the
public C header purely as an interface convention: 1 = E2M1 (MXFP4),
2 = E4M3FN (MXFP8).
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import build as _build

E2M1 = 1
E4M3 = 2
BLOCK = 32

_lib = None


def _configure(L: ctypes.CDLL) -> ctypes.CDLL:
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    vp = ctypes.c_void_p
    L.mxo_quantize.argtypes = [vp, i64, i64, i32, vp, vp]
    L.mxo_quantize.restype = i32
    L.mxo_dequantize.argtypes = [vp, vp, i64, i64, i32, vp]
    L.mxo_dequantize.restype = i32
    L.mxo_block_matmul.argtypes = [vp, vp, i32, vp, vp, i32, i64, i64, i64, vp, vp, vp]
    L.mxo_block_matmul.restype = i32
    L.mxo_block_matmul_entries.argtypes = [vp, vp, i32, vp, vp, i32, i64, vp, vp, vp, i64, vp, vp]
    L.mxo_block_matmul_entries.restype = i32
    L.mxo_decode_element.argtypes = [i32, i32]
    L.mxo_decode_element.restype = dbl
    L.mxo_decode_scale.argtypes = [i32]
    L.mxo_decode_scale.restype = dbl
    L.mxo_floor_log2.argtypes = [dbl]
    L.mxo_floor_log2.restype = i32
    L.mxo_quantize_axis0.argtypes = [vp, i64, i64, i32, vp, vp]
    L.mxo_quantize_axis0.restype = i32
    L.mxo_dequantize_bf16.argtypes = [vp, vp, i64, i64, i32, vp]
    L.mxo_dequantize_bf16.restype = i32
    L.mxo_block_matmul_f32b.argtypes = [vp, vp, i32, vp, i64, i64, i64, vp, vp, vp]
    L.mxo_block_matmul_f32b.restype = i32
    L.mxo_fold_scale.argtypes = [vp, i64, i32]
    L.mxo_fold_scale.restype = None
    L.mxo_fold_exponent.argtypes = [dbl]
    L.mxo_fold_exponent.restype = i32
    L.mxo_num_threads.argtypes = []
    L.mxo_num_threads.restype = i32
    L.mxo_set_num_threads.argtypes = [i32]
    L.mxo_set_num_threads.restype = None
    return L


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


class use_library:
    """Context manager: route this module's calls to another build of the
    oracle source (the pin suite uses it to check that planted mistakes in a
    copy of mx_oracle.c are caught)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = lib()
        _lib = _configure(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def code_bytes_per_row(fmt: int, cols: int) -> int:
    return cols // 2 if fmt == E2M1 else cols


def quantize(x: np.ndarray, fmt: int) -> tuple[np.ndarray, np.ndarray]:
    """x: float32 [rows, cols] -> (codes uint8 [rows, cb], scales uint8 [rows, cols/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x.reshape(1, -1)
    rows, cols = x.shape
    codes = np.zeros((rows, code_bytes_per_row(fmt, cols)), np.uint8)
    scales = np.zeros((rows, cols // BLOCK), np.uint8)
    rc = lib().mxo_quantize(_ptr(x), rows, cols, fmt, _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError(f"oracle quantize rejected shape/format (rc={rc})")
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray, cols: int, fmt: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows = scales.shape[0]
    y = np.zeros((rows, cols), np.float32)
    rc = lib().mxo_dequantize(_ptr(codes), _ptr(scales), rows, cols, fmt, _ptr(y))
    if rc:
        raise ValueError(f"oracle dequantize rejected shape/format (rc={rc})")
    return y


def block_matmul(a_codes, a_scales, a_fmt, b_codes, b_scales, b_fmt, M, N, K, c0):
    """C0 + A . Bt^T in binary64; returns (ref [M,N] f64, sabs [M,N] f64)."""
    a_codes = np.ascontiguousarray(a_codes, np.uint8)
    a_scales = np.ascontiguousarray(a_scales, np.uint8)
    b_codes = np.ascontiguousarray(b_codes, np.uint8)
    b_scales = np.ascontiguousarray(b_scales, np.uint8)
    c0 = np.ascontiguousarray(c0, np.float32)
    ref = np.zeros((M, N), np.float64)
    sabs = np.zeros((M, N), np.float64)
    rc = lib().mxo_block_matmul(_ptr(a_codes), _ptr(a_scales), a_fmt, _ptr(b_codes), _ptr(b_scales),
                                b_fmt, M, N, K, _ptr(c0), _ptr(ref), _ptr(sabs))
    if rc:
        raise ValueError("oracle block_matmul rejected shape/format")
    return ref, sabs


def block_matmul_entries(a_codes, a_scales, a_fmt, b_codes, b_scales, b_fmt, K,
                         a_row, b_row, c0):
    """Selected entries: entry i uses row a_row[i] of (a_codes, a_scales) and row
    b_row[i] of (b_codes, b_scales), starting from accumulator c0[i]."""
    a_codes = np.ascontiguousarray(a_codes, np.uint8)
    a_scales = np.ascontiguousarray(a_scales, np.uint8)
    b_codes = np.ascontiguousarray(b_codes, np.uint8)
    b_scales = np.ascontiguousarray(b_scales, np.uint8)
    a_row = np.ascontiguousarray(a_row, np.int64)
    b_row = np.ascontiguousarray(b_row, np.int64)
    c0 = np.ascontiguousarray(c0, np.float32)
    n = a_row.shape[0]
    ref = np.zeros(n, np.float64)
    sabs = np.zeros(n, np.float64)
    rc = lib().mxo_block_matmul_entries(_ptr(a_codes), _ptr(a_scales), a_fmt, _ptr(b_codes),
                                        _ptr(b_scales), b_fmt, K, _ptr(a_row), _ptr(b_row),
                                        _ptr(c0), n, _ptr(ref), _ptr(sabs))
    if rc:
        raise ValueError("oracle block_matmul_entries rejected shape/format")
    return ref, sabs


def quantize_axis0(x: np.ndarray, fmt: int) -> tuple[np.ndarray, np.ndarray]:
    """x: float32 [rows, cols], blocks of 32 rows down each column ->
    (codes uint8 [cols, cb(rows)], scales uint8 [cols, rows/32]): the layout of
    the transposed tensor."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    codes = np.zeros((cols, code_bytes_per_row(fmt, rows)), np.uint8)
    scales = np.zeros((cols, rows // BLOCK), np.uint8)
    rc = lib().mxo_quantize_axis0(_ptr(x), rows, cols, fmt, _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError(f"oracle quantize_axis0 rejected shape/format (rc={rc})")
    return codes, scales


def dequantize_bf16(codes: np.ndarray, scales: np.ndarray, cols: int, fmt: int) -> np.ndarray:
    """-> uint16 [rows, cols]: bfloat16 bit patterns."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    rows = scales.shape[0]
    y = np.zeros((rows, cols), np.uint16)
    rc = lib().mxo_dequantize_bf16(_ptr(codes), _ptr(scales), rows, cols, fmt, _ptr(y))
    if rc:
        raise ValueError(f"oracle dequantize_bf16 rejected shape/format (rc={rc})")
    return y


def block_matmul_f32b(a_codes, a_scales, a_fmt, B, M, N, K, c0):
    """C0 + deq(A) . B with B f32 [K, N] row-major; returns (ref, sabs) f64 [M, N]."""
    a_codes = np.ascontiguousarray(a_codes, np.uint8)
    a_scales = np.ascontiguousarray(a_scales, np.uint8)
    B = np.ascontiguousarray(B, np.float32)
    c0 = np.ascontiguousarray(c0, np.float32)
    ref = np.zeros((M, N), np.float64)
    sabs = np.zeros((M, N), np.float64)
    rc = lib().mxo_block_matmul_f32b(_ptr(a_codes), _ptr(a_scales), a_fmt, _ptr(B), M, N, K, _ptr(c0),
                                     _ptr(ref), _ptr(sabs))
    if rc:
        raise ValueError("oracle block_matmul_f32b rejected shape/format")
    return ref, sabs


def fold_scale(scales: np.ndarray, j: int) -> np.ndarray:
    """A copy of the scale bytes with the power-of-two factor 2^j folded in."""
    out = np.ascontiguousarray(scales, dtype=np.uint8).copy()
    lib().mxo_fold_scale(_ptr(out), out.size, int(j))
    return out


def fold_exponent(scalar: float):
    """j for a foldable scalar 2^j, else None."""
    j = lib().mxo_fold_exponent(float(scalar))
    return None if j == -1000 else j


def decode_element(fmt: int, code: int) -> float:
    return lib().mxo_decode_element(fmt, code)


def decode_scale(byte: int) -> float:
    return lib().mxo_decode_scale(byte)


def floor_log2(v: float) -> int:
    return lib().mxo_floor_log2(v)


def num_threads() -> int:
    return lib().mxo_num_threads()


def set_threads(n: int) -> None:
    """OpenMP thread count for later oracle calls."""
    lib().mxo_set_num_threads(int(n))
