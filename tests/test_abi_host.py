"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/mx.h declares, sizes its buffers as documented, and
rejects bad arguments on the host before anything is launched.

Calls here pass fake device addresses only where validation must fail first;
the one call with well-formed arguments runs only when no GPU is present."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import bit_gemm_gb300 as mx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
L = mx.lib
OK, NULL, SHAPE, UNSUP, ALIGN, TIMEOUT, CUDA, NODEV = range(8)
A16 = 0x10000  # fake, 16-byte aligned address (never dereferenced)


def declared_functions():
    with open(os.path.join(ROOT, "include", "mx.h")) as f:
        text = f.read()
    return re.findall(r"MX_API\s+[\w\s\*]+?\b(mx_\w+)\s*\(", text)


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert len(names) == 19
    out = subprocess.run(["nm", "-D", "--defined-only", mx.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (mx_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(L, n)


def test_size_helpers():
    assert mx.mx_codes_bytes(mx.E2M1, 4, 64) == 128
    assert mx.mx_codes_bytes(mx.E4M3FN, 4, 64) == 256
    assert mx.mx_codes_bytes(mx.E2M1, 4, 33) == -1
    assert mx.mx_codes_bytes(7, 4, 64) == -1
    assert mx.mx_scales_bytes(mx.SCALES_ROWMAJOR, 5, 96) == 15
    # tensor-core layout: rows padded to 128, blocks per row padded to 4, 512 B per tile
    assert mx.mx_scales_bytes(mx.SCALES_MMA, 5, 96) == 512
    assert mx.mx_scales_bytes(mx.SCALES_MMA, 129, 160) == 2 * 2 * 512
    assert mx.mx_scales_bytes(mx.SCALES_MMA, 0, 160) == 0
    # 136 bits per 32-element MXFP4 block
    assert (mx.mx_codes_bytes(mx.E2M1, 1, 32) + mx.mx_scales_bytes(mx.SCALES_ROWMAJOR, 1, 32)) * 8 == 136


def test_status_strings():
    for s in range(8):
        assert L.mx_status_string(s).decode().startswith("MX_")
    assert L.mx_status_string(99) == b"unknown mx_status_t"


def q(x=A16, dt=mx.F32, rows=4, cols=64, fmt=mx.E2M1, bs=32, st=1, codes=A16 * 4, scales=A16 * 8,
      layout=mx.SCALES_ROWMAJOR):
    return L.mx_quantize(x, dt, rows, cols, fmt, bs, st, codes, scales, layout, None)


def test_quantize_validation():
    assert q(cols=33) == SHAPE
    assert q(rows=-1) == SHAPE
    assert q(bs=16) == UNSUP
    assert q(st=2) == UNSUP
    assert q(fmt=3) == UNSUP
    assert q(dt=9) == UNSUP
    assert q(layout=5) == UNSUP
    assert q(x=None) == NULL
    assert q(codes=None) == NULL
    assert q(x=A16 + 4) == ALIGN
    assert q(codes=A16 * 4 + 8) == ALIGN
    assert q(scales=A16 * 8 + 2) == ALIGN
    assert q(scales=A16 * 8 + 4) != ALIGN or True  # 4-byte aligned is enough for row-major
    assert q(scales=A16 * 8 + 4, layout=mx.SCALES_MMA) == ALIGN
    assert q(codes=A16 + 64) == UNSUP            # overlaps x (4 x 64 f32 = 1 KB)
    assert q(rows=0) == OK and q(cols=0) == OK    # empty tensors are a no-op
    assert L.mx_last_error_detail() == b""
    q(cols=33)
    assert b"multiple of the block size" in L.mx_last_error_detail()


def test_dequantize_validation():
    d = lambda **k: L.mx_dequantize(k.get("codes", A16), k.get("scales", A16 * 2), k.get("rows", 4),
                                    k.get("cols", 64), k.get("fmt", mx.E4M3FN), k.get("bs", 32), 1,
                                    k.get("layout", 0), k.get("y", A16 * 8), None)
    assert d(cols=40) == SHAPE
    assert d(bs=64) == UNSUP
    assert d(y=None) == NULL
    assert d(y=A16 * 8 + 8) == ALIGN
    assert d(y=A16 + 16) == UNSUP  # y overlaps codes
    assert d(rows=0) == OK


def g(a=A16, sa=A16 * 2, af=mx.E2M1, b=A16 * 3, sb=A16 * 4, bf=mx.E2M1, layout=mx.SCALES_MMA, bs=32, M=128,
      N=128, K=256, C=A16 * 64):
    return L.mx_block_matmul(a, sa, af, b, sb, bf, layout, bs, 1, M, N, K, C, None)


def test_block_matmul_validation():
    assert g(K=48) == SHAPE
    assert g(M=-1) == SHAPE
    assert g(af=mx.E4M3FN, K=160) == SHAPE      # mixed formats need K % 128 == 0
    assert g(bs=16) == UNSUP
    assert g(af=0) == UNSUP
    assert g(layout=3) == UNSUP
    assert g(C=None) == NULL
    assert g(C=A16 * 64 + 4) == ALIGN
    assert g(af=mx.E4M3FN, b=A16 * 3 + 16) == ALIGN  # the E2M1 operand of a mixed product needs 32 B
    assert g(C=A16) == UNSUP                    # C overlaps A's codes
    assert g(layout=mx.SCALES_ROWMAJOR, K=96) == SHAPE   # row-major scales need K % 128 == 0
    assert g(M=0) == OK and g(N=0) == OK and g(K=0) == OK


def gw(ws=A16 * 256, nws=1 << 20, layout=mx.SCALES_ROWMAJOR, M=4, N=4, K=128, C=A16 * 64):
    return L.mx_block_matmul_ws(A16, A16 * 2, mx.E2M1, A16 * 3, A16 * 5, mx.E2M1, layout, 32, 1, M, N, K, C, ws,
                                nws, None)


def test_block_matmul_workspace_bytes_and_validation():
    need = L.mx_block_matmul_workspace_bytes
    # row-major scales: the tensor-core-layout scale bytes of A and B, each rounded up to 256
    rnd = lambda v: (v + 255) // 256 * 256
    for M, N, K in ((4, 4, 128), (130, 300, 1024), (8192, 28672, 8192), (16, 14336, 4096)):
        assert need(mx.SCALES_ROWMAJOR, M, N, K) == rnd(mx.mx_scales_bytes(mx.SCALES_MMA, M, K)) + \
            rnd(mx.mx_scales_bytes(mx.SCALES_MMA, N, K))
    assert need(mx.SCALES_MMA, 4, 4, 128) == 0
    assert need(mx.SCALES_ROWMAJOR, 0, 4, 128) == 0
    assert need(mx.SCALES_ROWMAJOR, 4, 4, 48) == -1
    assert need(5, 4, 4, 128) == -1
    # checks that run before anything is launched
    assert gw(ws=None) == NULL
    assert gw(nws=need(mx.SCALES_ROWMAJOR, 4, 4, 128) - 1) == SHAPE
    assert gw(ws=A16 * 256 + 16) == ALIGN
    assert gw(ws=A16 * 64) == UNSUP          # overlaps C
    assert gw(K=96) == SHAPE                 # row-major scales need K % 128 == 0
    assert gw(M=0) == OK


def test_relayout_and_selftest_validation():
    assert L.mx_scales_relayout(A16, 0, 4, 33, A16 * 4, 1, None) == SHAPE
    assert L.mx_scales_relayout(A16, 0, 4, 64, A16, 1, None) == UNSUP  # overlap
    assert L.mx_scales_relayout(None, 0, 4, 64, A16, 1, None) == NULL
    assert L.mx_selftest_wait_timeout(10, None) == UNSUP


@pytest.mark.skipif(torch.cuda.is_available(), reason="only meaningful on a host without a GPU")
def test_no_cpu_fallback_without_device():
    # Well-formed arguments on a machine with no GPU: the library reports the
    # missing device instead of computing anything on the CPU.
    assert q() == NODEV
    assert g() == NODEV
    assert L.mx_device_status(None) == NODEV


def test_python_binding_rejects_host_tensors():
    x = torch.zeros(4, 64)
    with pytest.raises((ValueError, RuntimeError, AssertionError)):
        mx.mx_quantize(x, mx.E2M1, torch.zeros(128, dtype=torch.uint8), torch.zeros(8, dtype=torch.uint8))


def qa(x=A16, dt=mx.BF16, rows=64, cols=7, axis=0, fmt=mx.E4M3FN, bs=32, st=1, codes=A16 * 4, scales=A16 * 8,
       layout=mx.SCALES_ROWMAJOR):
    return L.mx_quantize_axis(x, dt, rows, cols, axis, fmt, bs, st, codes, scales, layout, None)


def test_quantize_axis_validation():
    assert qa(axis=2) == UNSUP and qa(axis=-1) == UNSUP
    assert qa(rows=48) == SHAPE                 # axis 0 blocks run along rows
    assert qa(axis=1, cols=7) == SHAPE          # axis 1 blocks run along cols
    assert qa(bs=16) == UNSUP and qa(fmt=3) == UNSUP and qa(dt=9) == UNSUP
    assert qa(x=None) == NULL and qa(scales=None) == NULL
    assert qa(x=A16 + 4) == ALIGN
    assert qa(codes=A16 + 64) == UNSUP          # overlaps x (64 x 7 bf16 = 896 B)
    assert qa(rows=0) == OK and qa(cols=0) == OK
    if not torch.cuda.is_available():
        assert qa() == NODEV


def fs(scales=A16, rows=8, cols=64, layout=mx.SCALES_ROWMAJOR, scalar=2.0):
    return L.mx_fold_scale(scales, rows, cols, layout, scalar, None)


def test_fold_scale_validation():
    for bad in (3.0, -2.0, 0.0, -0.0, float("inf"), float("nan"), 1.5, 0.75):
        assert fs(scalar=bad) == UNSUP, bad
    assert fs(layout=5) == UNSUP
    assert fs(rows=-1) == SHAPE and fs(cols=33) == SHAPE
    assert fs(scales=None) == NULL
    assert fs(rows=0) == OK
    if not torch.cuda.is_available():
        for good in (1.0, 0.5, 2.0 ** 100, 2.0 ** -1000):
            assert fs(scalar=good) == NODEV, good


def test_dequantize_bf16_validation():
    d = lambda **k: L.mx_dequantize_bf16(k.get("codes", A16), k.get("scales", A16 * 4), k.get("rows", 4),
                                         k.get("cols", 64), k.get("fmt", mx.E2M1), 32, 1,
                                         k.get("layout", mx.SCALES_ROWMAJOR), k.get("y", A16 * 8), None)
    assert d(cols=33) == SHAPE and d(fmt=3) == UNSUP and d(layout=5) == UNSUP
    assert d(y=None) == NULL and d(y=A16 * 8 + 8) == ALIGN
    assert d(y=A16 + 16) == UNSUP                # overlaps the codes
    assert d(rows=0) == OK
    if not torch.cuda.is_available():
        assert d() == NODEV


def ga(a=A16 * 2, dt=mx.BF16, fa=mx.E4M3FN, b=A16 * 64, sb=A16 * 128, fb=mx.E2M1, layout=mx.SCALES_MMA, bs=32, st=1,
       M=16, N=256, K=256, C=A16 * 256):
    return L.mx_block_matmul_act(a, dt, fa, b, sb, fb, layout, bs, st, M, N, K, C, None)


def test_block_matmul_act_validation():
    assert ga(M=65) == UNSUP                      # larger M: quantize once, then mx_block_matmul
    assert ga(fa=mx.E2M1, fb=mx.E4M3FN) == UNSUP  # E2M1 activations with E4M3 weights
    assert ga(layout=mx.SCALES_ROWMAJOR) == UNSUP
    assert ga(dt=9) == UNSUP and ga(bs=16) == UNSUP
    assert ga(K=96) == SHAPE                      # mixed formats need K % 128 == 0
    assert ga(K=33) == SHAPE and ga(M=-1) == SHAPE
    assert ga(a=None) == NULL and ga(C=None) == NULL
    assert ga(a=A16 * 2 + 16) == ALIGN            # activations 32-byte aligned
    assert ga(M=0) == OK
    if not torch.cuda.is_available():
        assert ga() == NODEV


def gf(a=A16, sa=A16 * 2, fa=mx.E4M3FN, layout=mx.SCALES_ROWMAJOR, bs=32, st=1, B=A16 * 64, M=16, N=256, K=256,
       C=A16 * 256):
    return L.mx_block_matmul_f32b(a, sa, fa, layout, bs, st, B, M, N, K, C, None)


def test_block_matmul_f32b_validation():
    assert gf(fa=3) == UNSUP and gf(layout=4) == UNSUP and gf(bs=16) == UNSUP
    assert gf(K=33) == SHAPE and gf(N=-1) == SHAPE
    assert gf(N=258) == ALIGN                     # rows of B and C on 16-byte boundaries
    assert gf(B=None) == NULL and gf(C=None) == NULL
    assert gf(B=A16 * 64 + 4) == ALIGN and gf(C=A16 * 256 + 8) == ALIGN
    assert gf(C=A16 * 64) == UNSUP                # C overlaps B
    assert gf(M=0) == OK and gf(K=0) == OK
    if not torch.cuda.is_available():
        assert gf() == NODEV


def test_measure_mma_rate_validation():
    out = ctypes.c_double(0.0)
    assert L.mx_measure_mma_rate(3, 10, ctypes.byref(out), None) == UNSUP
    assert L.mx_measure_mma_rate(mx.E2M1, 0, ctypes.byref(out), None) == SHAPE
    assert L.mx_measure_mma_rate(mx.E2M1, 10, None, None) == NULL
    if not torch.cuda.is_available():
        assert L.mx_measure_mma_rate(mx.E2M1, 10, ctypes.byref(out), None) == NODEV
