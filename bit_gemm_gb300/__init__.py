"""Python binding of libmx, the GB300 (sm_103a) MX block-scaled library.

Every function mirrors one entry point of ``include/mx.h`` under the same
name and only marshals arguments: torch CUDA tensors in, raw device pointers
and sizes out, the stream taken from torch unless given.  Compute happens in
the CUDA kernels of ``libmx.so``; there is no CPU fallback, and importing this
package raises if the library has not been built.

Because the C ABI receives bare pointers, this layer checks what a pointer
cannot carry: that each tensor lives on the current CUDA device, is
contiguous, and holds at least the bytes the call will touch.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmx.so")

# enums of include/mx.h
MX_OK = 0
E2M1, E4M3FN = 1, 2
SCALE_E8M0 = 1
F32, BF16 = 1, 2
SCALES_ROWMAJOR, SCALES_MMA = 0, 1
BLOCK = 32

STATUS_NAMES = {0: "MX_OK", 1: "MX_ERR_NULL", 2: "MX_ERR_SHAPE", 3: "MX_ERR_UNSUPPORTED", 4: "MX_ERR_ALIGN",
                5: "MX_ERR_TIMEOUT", 6: "MX_ERR_CUDA", 7: "MX_ERR_NO_DEVICE"}


class MxError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()' "
            "or python bit_gemm_gb300/build.py)")
    L = ctypes.CDLL(LIB_PATH)
    i64, i32, u64, vp, cp = ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_char_p
    L.mx_codes_bytes.argtypes = [i32, i64, i64]
    L.mx_codes_bytes.restype = i64
    L.mx_scales_bytes.argtypes = [i32, i64, i64]
    L.mx_scales_bytes.restype = i64
    L.mx_quantize.argtypes = [vp, i32, i64, i64, i32, i32, i32, vp, vp, i32, vp]
    L.mx_quantize.restype = i32
    L.mx_dequantize.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, vp, vp]
    L.mx_dequantize.restype = i32
    L.mx_block_matmul.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, i64, i64, i64, vp, vp]
    L.mx_block_matmul.restype = i32
    L.mx_block_matmul_ws.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, i64, i64, i64, vp, vp, i64, vp]
    L.mx_block_matmul_ws.restype = i32
    L.mx_block_matmul_workspace_bytes.argtypes = [i32, i64, i64, i64]
    L.mx_block_matmul_workspace_bytes.restype = i64
    L.mx_block_matmul_static_ws.argtypes = [vp, vp, i32, vp, vp, i32, i32, i32, i32, i64, i64, i64, vp, vp]
    L.mx_block_matmul_static_ws.restype = i32
    L.mx_scales_relayout.argtypes = [vp, i32, i64, i64, vp, i32, vp]
    L.mx_scales_relayout.restype = i32
    L.mx_quantize_axis.argtypes = [vp, i32, i64, i64, i32, i32, i32, i32, vp, vp, i32, vp]
    L.mx_quantize_axis.restype = i32
    L.mx_dequantize_bf16.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, vp, vp]
    L.mx_dequantize_bf16.restype = i32
    L.mx_fold_scale.argtypes = [vp, i64, i64, i32, ctypes.c_double, vp]
    L.mx_fold_scale.restype = i32
    L.mx_block_matmul_act.argtypes = [vp, i32, i32, vp, vp, i32, i32, i32, i32, i64, i64, i64, vp, vp]
    L.mx_block_matmul_act.restype = i32
    L.mx_block_matmul_f32b.argtypes = [vp, vp, i32, i32, i32, i32, vp, i64, i64, i64, vp, vp]
    L.mx_block_matmul_f32b.restype = i32
    L.mx_measure_mma_rate.argtypes = [i32, i32, ctypes.POINTER(ctypes.c_double), vp]
    L.mx_measure_mma_rate.restype = i32
    L.mx_device_status.argtypes = [vp]
    L.mx_device_status.restype = i32
    L.mx_selftest_wait_timeout.argtypes = [u64, vp]
    L.mx_selftest_wait_timeout.restype = i32
    L.mx_status_string.argtypes = [i32]
    L.mx_status_string.restype = cp
    L.mx_last_error_detail.argtypes = []
    L.mx_last_error_detail.restype = cp
    return L


lib = _load()


def _check(status: int) -> None:
    if status != MX_OK:
        raise MxError(status, lib.mx_last_error_detail().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_ptr(t: torch.Tensor, name: str, min_bytes: int) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not the current device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    nbytes = t.numel() * t.element_size()
    if nbytes < min_bytes:
        raise ValueError(f"{name} holds {nbytes} bytes, the call needs {min_bytes}")
    return t.data_ptr()


def mx_codes_bytes(fmt: int, rows: int, cols: int) -> int:
    return lib.mx_codes_bytes(fmt, rows, cols)


def mx_scales_bytes(layout: int, rows: int, cols: int) -> int:
    return lib.mx_scales_bytes(layout, rows, cols)


def mx_status_string(status: int) -> str:
    return lib.mx_status_string(status).decode()


def mx_quantize(x: torch.Tensor, fmt: int, codes: torch.Tensor, scales: torch.Tensor,
                scale_layout: int = SCALES_ROWMAJOR, stream=None, block_size: int = BLOCK,
                scale_type: int = SCALE_E8M0) -> None:
    """quantize_block over a [rows, cols] f32/bf16 tensor into (codes, scales)."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D [rows, cols]")
    rows, cols = x.shape
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(x.dtype)
    if dt is None:
        raise ValueError(f"x dtype {x.dtype} (f32 or bf16 only)")
    if rows * cols == 0:
        return
    cb, sb = mx_codes_bytes(fmt, rows, cols), mx_scales_bytes(scale_layout, rows, cols)
    if cb < 0 or sb < 0:
        _check(lib.mx_quantize(None, dt, rows, cols, fmt, block_size, scale_type, None, None, scale_layout, None))
    _check(lib.mx_quantize(_dev_ptr(x, "x", 0), dt, rows, cols, fmt, block_size, scale_type,
                           _dev_ptr(codes, "codes", cb), _dev_ptr(scales, "scales", sb), scale_layout,
                           _stream(stream)))


def mx_dequantize(codes: torch.Tensor, scales: torch.Tensor, rows: int, cols: int, fmt: int, y: torch.Tensor,
                  scale_layout: int = SCALES_ROWMAJOR, stream=None, block_size: int = BLOCK,
                  scale_type: int = SCALE_E8M0) -> None:
    """dequantize_block: (codes, scales) -> y, an f32 [rows, cols] tensor."""
    if rows * cols == 0:
        return
    if y.dtype != torch.float32:
        raise ValueError("y must be float32")
    cb, sb = mx_codes_bytes(fmt, rows, cols), mx_scales_bytes(scale_layout, rows, cols)
    if cb < 0 or sb < 0:
        _check(lib.mx_dequantize(None, None, rows, cols, fmt, block_size, scale_type, scale_layout, None, None))
    _check(lib.mx_dequantize(_dev_ptr(codes, "codes", cb), _dev_ptr(scales, "scales", sb), rows, cols, fmt,
                             block_size, scale_type, scale_layout, _dev_ptr(y, "y", rows * cols * 4),
                             _stream(stream)))


def mx_block_matmul(a_codes: torch.Tensor, a_scales: torch.Tensor, a_fmt: int,
                    b_codes: torch.Tensor, b_scales: torch.Tensor, b_fmt: int,
                    M: int, N: int, K: int, C: torch.Tensor, scale_layout: int = SCALES_MMA, stream=None,
                    block_size: int = BLOCK, scale_type: int = SCALE_E8M0) -> None:
    """C += A * B with A [M,K] and B given transposed as [N,K], both MX; C f32 [M,N] in place."""
    if M * N * K == 0:
        _check(lib.mx_block_matmul(None, None, a_fmt, None, None, b_fmt, scale_layout, block_size, scale_type,
                                   M, N, K, None, None))
        return
    if C.dtype != torch.float32:
        raise ValueError("C must be float32")
    ca, cb = mx_codes_bytes(a_fmt, M, K), mx_codes_bytes(b_fmt, N, K)
    sa, sb = mx_scales_bytes(scale_layout, M, K), mx_scales_bytes(scale_layout, N, K)
    if min(ca, cb, sa, sb) < 0:
        _check(lib.mx_block_matmul(None, None, a_fmt, None, None, b_fmt, scale_layout, block_size, scale_type,
                                   M, N, K, None, None))
    _check(lib.mx_block_matmul(_dev_ptr(a_codes, "a_codes", ca), _dev_ptr(a_scales, "a_scales", sa), a_fmt,
                               _dev_ptr(b_codes, "b_codes", cb), _dev_ptr(b_scales, "b_scales", sb), b_fmt,
                               scale_layout, block_size, scale_type, M, N, K,
                               _dev_ptr(C, "C", M * N * 4), _stream(stream)))


def mx_block_matmul_workspace_bytes(scale_layout: int, M: int, N: int, K: int) -> int:
    return int(lib.mx_block_matmul_workspace_bytes(scale_layout, M, N, K))


def alloc_workspace(M: int, N: int, K: int, scale_layout: int = SCALES_ROWMAJOR) -> torch.Tensor | None:
    """A device buffer (caller-owned, from torch) for mx_block_matmul_ws; None when none is needed."""
    n = mx_block_matmul_workspace_bytes(scale_layout, M, N, K)
    if n < 0:
        raise ValueError("invalid layout or shape for a block_matmul workspace")
    return torch.empty(n, dtype=torch.uint8, device="cuda") if n > 0 else None


def mx_block_matmul_ws(a_codes: torch.Tensor, a_scales: torch.Tensor, a_fmt: int,
                       b_codes: torch.Tensor, b_scales: torch.Tensor, b_fmt: int,
                       M: int, N: int, K: int, C: torch.Tensor, workspace: torch.Tensor | None,
                       scale_layout: int = SCALES_ROWMAJOR, stream=None,
                       block_size: int = BLOCK, scale_type: int = SCALE_E8M0) -> None:
    """mx_block_matmul with a caller-owned workspace: row-major scales are
    rewritten into it in the tensor-core layout before the product."""
    need = mx_block_matmul_workspace_bytes(scale_layout, M, N, K) if min(M, N, K) >= 0 else 0
    ws = _dev_ptr(workspace, "workspace", max(need, 0)) if (workspace is not None and need > 0) else None
    nws = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if M * N * K == 0:
        _check(lib.mx_block_matmul_ws(None, None, a_fmt, None, None, b_fmt, scale_layout, block_size, scale_type,
                                      M, N, K, None, ws, nws, None))
        return
    if C.dtype != torch.float32:
        raise ValueError("C must be float32")
    ca, cb = mx_codes_bytes(a_fmt, M, K), mx_codes_bytes(b_fmt, N, K)
    sa, sb = mx_scales_bytes(scale_layout, M, K), mx_scales_bytes(scale_layout, N, K)
    if min(ca, cb, sa, sb) < 0:
        _check(lib.mx_block_matmul_ws(None, None, a_fmt, None, None, b_fmt, scale_layout, block_size, scale_type,
                                      M, N, K, None, ws, nws, None))
    _check(lib.mx_block_matmul_ws(_dev_ptr(a_codes, "a_codes", ca), _dev_ptr(a_scales, "a_scales", sa), a_fmt,
                                  _dev_ptr(b_codes, "b_codes", cb), _dev_ptr(b_scales, "b_scales", sb), b_fmt,
                                  scale_layout, block_size, scale_type, M, N, K,
                                  _dev_ptr(C, "C", M * N * 4), ws, nws, _stream(stream)))


def mx_quantize_axis(x: torch.Tensor, axis: int, fmt: int, codes: torch.Tensor, scales: torch.Tensor,
                     scale_layout: int = SCALES_ROWMAJOR, stream=None, block_size: int = BLOCK,
                     scale_type: int = SCALE_E8M0) -> None:
    """quantize_block of a [rows, cols] tensor along `axis`; axis 0 writes the
    layout of the [cols, rows] transpose (the N x K operand of mx_block_matmul)."""
    if x.dim() != 2:
        raise ValueError("x must be 2-D [rows, cols]")
    rows, cols = x.shape
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(x.dtype)
    if dt is None:
        raise ValueError(f"x dtype {x.dtype} (f32 or bf16 only)")
    if rows * cols == 0:
        return
    o_rows, o_cols = (cols, rows) if axis == 0 else (rows, cols)
    cb, sb = mx_codes_bytes(fmt, o_rows, o_cols), mx_scales_bytes(scale_layout, o_rows, o_cols)
    if cb < 0 or sb < 0 or axis not in (0, 1):
        _check(lib.mx_quantize_axis(None, dt, rows, cols, axis, fmt, block_size, scale_type, None, None,
                                    scale_layout, None))
    _check(lib.mx_quantize_axis(_dev_ptr(x, "x", 0), dt, rows, cols, axis, fmt, block_size, scale_type,
                                _dev_ptr(codes, "codes", cb), _dev_ptr(scales, "scales", sb), scale_layout,
                                _stream(stream)))


def mx_dequantize_bf16(codes: torch.Tensor, scales: torch.Tensor, rows: int, cols: int, fmt: int,
                       y: torch.Tensor, scale_layout: int = SCALES_ROWMAJOR, stream=None, block_size: int = BLOCK,
                       scale_type: int = SCALE_E8M0) -> None:
    """dequantize_block to bfloat16: (codes, scales) -> y, a bf16 [rows, cols] tensor."""
    if rows * cols == 0:
        return
    if y.dtype != torch.bfloat16:
        raise ValueError("y must be bfloat16")
    cb, sb = mx_codes_bytes(fmt, rows, cols), mx_scales_bytes(scale_layout, rows, cols)
    if cb < 0 or sb < 0:
        _check(lib.mx_dequantize_bf16(None, None, rows, cols, fmt, block_size, scale_type, scale_layout, None,
                                      None))
    _check(lib.mx_dequantize_bf16(_dev_ptr(codes, "codes", cb), _dev_ptr(scales, "scales", sb), rows, cols,
                                  fmt, block_size, scale_type, scale_layout, _dev_ptr(y, "y", rows * cols * 2),
                                  _stream(stream)))


def mx_fold_scale(scales: torch.Tensor, rows: int, cols: int, scalar: float,
                  scale_layout: int = SCALES_ROWMAJOR, stream=None) -> None:
    """fold_scale: multiply the MX tensor with these scales by a power-of-two scalar, in place."""
    sb = mx_scales_bytes(scale_layout, rows, cols)
    if sb < 0 or rows * cols == 0:
        _check(lib.mx_fold_scale(None, rows, cols, scale_layout, float(scalar), None))
        return
    _check(lib.mx_fold_scale(_dev_ptr(scales, "scales", sb), rows, cols, scale_layout, float(scalar),
                             _stream(stream)))


def mx_block_matmul_act(a: torch.Tensor, a_fmt: int, b_codes: torch.Tensor, b_scales: torch.Tensor, b_fmt: int,
                        N: int, C: torch.Tensor, stream=None, block_size: int = BLOCK,
                        scale_type: int = SCALE_E8M0) -> None:
    """C += quantize(a) * B with a f32/bf16 [M, K] quantized inside the GEMM (M <= 64); B given as [N, K]
    codes with MX_SCALES_MMA scales; C f32 [M, N] in place."""
    if a.dim() != 2:
        raise ValueError("a must be 2-D [M, K]")
    M, K = a.shape
    dt = {torch.float32: F32, torch.bfloat16: BF16}.get(a.dtype)
    if dt is None:
        raise ValueError(f"a dtype {a.dtype} (f32 or bf16 only)")
    if M * N * K == 0:
        _check(lib.mx_block_matmul_act(None, dt, a_fmt, None, None, b_fmt, SCALES_MMA, block_size, scale_type,
                                       M, N, K, None, None))
        return
    if C.dtype != torch.float32:
        raise ValueError("C must be float32")
    cb, sb = mx_codes_bytes(b_fmt, N, K), mx_scales_bytes(SCALES_MMA, N, K)
    if cb < 0 or sb < 0:
        _check(lib.mx_block_matmul_act(None, dt, a_fmt, None, None, b_fmt, SCALES_MMA, block_size, scale_type,
                                       M, N, K, None, None))
    _check(lib.mx_block_matmul_act(_dev_ptr(a, "a", 0), dt, a_fmt, _dev_ptr(b_codes, "b_codes", cb),
                                   _dev_ptr(b_scales, "b_scales", sb), b_fmt, SCALES_MMA, block_size, scale_type,
                                   M, N, K, _dev_ptr(C, "C", M * N * 4), _stream(stream)))


def mx_block_matmul_f32b(a_codes: torch.Tensor, a_scales: torch.Tensor, a_fmt: int, B: torch.Tensor, M: int,
                         C: torch.Tensor, scale_layout: int = SCALES_ROWMAJOR, stream=None, block_size: int = BLOCK,
                         scale_type: int = SCALE_E8M0) -> None:
    """C += dequantize(A) * B with A [M, K] codes/scales and B f32 [K, N] row-major; C f32 [M, N] in place."""
    if B.dim() != 2:
        raise ValueError("B must be 2-D [K, N]")
    K, N = B.shape
    if M * N * K == 0:
        _check(lib.mx_block_matmul_f32b(None, None, a_fmt, scale_layout, block_size, scale_type, None, M, N, K,
                                        None, None))
        return
    if B.dtype != torch.float32 or C.dtype != torch.float32:
        raise ValueError("B and C must be float32")
    cb, sb = mx_codes_bytes(a_fmt, M, K), mx_scales_bytes(scale_layout, M, K)
    if cb < 0 or sb < 0:
        _check(lib.mx_block_matmul_f32b(None, None, a_fmt, scale_layout, block_size, scale_type, None, M, N, K,
                                        None, None))
    _check(lib.mx_block_matmul_f32b(_dev_ptr(a_codes, "a_codes", cb), _dev_ptr(a_scales, "a_scales", sb), a_fmt,
                                    scale_layout, block_size, scale_type, _dev_ptr(B, "B", K * N * 4), M, N, K,
                                    _dev_ptr(C, "C", M * N * 4), _stream(stream)))


def mx_measure_mma_rate(fmt: int, iters: int = 20000, stream=None) -> float:
    """Measured block-scaled MMA rate (TFLOP/s, all SMs) for E4M3FN (kind::mxf8f6f4) or E2M1 (kind::mxf4)."""
    out = ctypes.c_double(0.0)
    _check(lib.mx_measure_mma_rate(fmt, iters, ctypes.byref(out), _stream(stream)))
    return out.value


def mx_scales_relayout(src: torch.Tensor, src_layout: int, rows: int, cols: int, dst: torch.Tensor,
                       dst_layout: int, stream=None) -> None:
    s, d = mx_scales_bytes(src_layout, rows, cols), mx_scales_bytes(dst_layout, rows, cols)
    if rows * cols == 0:
        return
    if s < 0 or d < 0:
        _check(lib.mx_scales_relayout(None, src_layout, rows, cols, None, dst_layout, None))
    _check(lib.mx_scales_relayout(_dev_ptr(src, "src", s), src_layout, rows, cols, _dev_ptr(dst, "dst", d),
                                  dst_layout, _stream(stream)))


def mx_device_status(stream=None) -> None:
    """Synchronize the stream; raise MxError on a kernel timeout or CUDA error."""
    _check(lib.mx_device_status(_stream(stream)))


def mx_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(lib.mx_selftest_wait_timeout(int(limit_ns), _stream(stream)))


# ---------------------------------------------------------------- helpers

def alloc_codes(rows: int, cols: int, fmt: int, device=None) -> torch.Tensor:
    n = mx_codes_bytes(fmt, rows, cols)
    if n < 0:
        raise ValueError("bad format or shape")
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device or "cuda")


def alloc_scales(rows: int, cols: int, layout: int = SCALES_ROWMAJOR, device=None) -> torch.Tensor:
    n = mx_scales_bytes(layout, rows, cols)
    if n < 0:
        raise ValueError("bad layout or shape")
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device or "cuda")
