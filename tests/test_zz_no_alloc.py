"""GPU test of mx_block_matmul_static_ws, the block_matmul entry point that
allocates nothing.

Callers that cannot allocate device memory (a host framework or plugin that
owns every device buffer, a process held to a fixed device memory budget, a
latency-critical path where an allocation that may synchronize the device is
not acceptable) call it instead of mx_block_matmul_ws: its scratch for the
tensor-core-layout scales is a 16 MiB device array inside the library.  Here
it is called through the C ABI on two products in a row, the second of a
different shape so that it runs over what the first left in that array, and
each result is compared with mx_block_matmul_ws on a caller-owned workspace
within the bound the GEMM tests use (1e-5 * sum|a*b| + 2^-23 * |result|).

This file sorts last among the tests, so a run that stops at the first
failure has run every other test before it; it depends on nothing those
tests leave behind and passes on its own in a fresh process too.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_gemm_gb300 as mx
import oracle

pytestmark = pytest.mark.gpu

O_FMT = {mx.E2M1: oracle.E2M1, mx.E4M3FN: oracle.E4M3}
MX_ERR_SHAPE = 2


def quantize_rowmajor(x, fmt):
    rows, cols = x.shape
    codes, scales = mx.alloc_codes(rows, cols, fmt), mx.alloc_scales(rows, cols, mx.SCALES_ROWMAJOR)
    mx.mx_quantize(torch.from_numpy(x).cuda(), fmt, codes, scales, mx.SCALES_ROWMAJOR)
    return codes, scales


def static_ws_call(ac, as_, fa, bc, bs, fb, M, N, K, C):
    """The entry point under test, called through the C ABI with raw device pointers."""
    torch.cuda.synchronize()
    status = mx.lib.mx_block_matmul_static_ws(
        ctypes.c_void_p(ac.data_ptr()), ctypes.c_void_p(as_.data_ptr()), fa, ctypes.c_void_p(bc.data_ptr()),
        ctypes.c_void_p(bs.data_ptr()), fb, mx.SCALES_ROWMAJOR, 32, mx.SCALE_E8M0, M, N, K,
        ctypes.c_void_p(C.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert status == 0, mx.lib.mx_last_error_detail().decode()
    mx.mx_device_status()


def one_product(seed, M, N, K, fa, fb):
    rng = np.random.default_rng(seed)
    A = rng.standard_normal((M, K)).astype(np.float32)
    Bt = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    ac, as_ = quantize_rowmajor(A, fa)
    bc, bs = quantize_rowmajor(Bt, fb)
    # the entry point under test
    C = torch.from_numpy(C0.copy()).cuda()
    static_ws_call(ac, as_, fa, bc, bs, fb, M, N, K, C)
    # the existing entry point, on a workspace the caller allocates
    C_ref = torch.from_numpy(C0.copy()).cuda()
    mx.mx_block_matmul_ws(ac, as_, fa, bc, bs, fb, M, N, K, C_ref, mx.alloc_workspace(M, N, K))
    mx.mx_device_status()
    # the bound's sum |a*b| over dequantized values, from the oracle
    oa, osa = oracle.quantize(A, O_FMT[fa])
    ob, osb = oracle.quantize(Bt, O_FMT[fb])
    _, sabs = oracle.block_matmul(oa, osa, O_FMT[fa], ob, osb, O_FMT[fb], M, N, K, C0)
    got = C.cpu().numpy().astype(np.float64)
    ref = C_ref.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all() and np.isfinite(ref).all()
    bad = np.abs(got - ref) > 1e-5 * sabs + 2.0 ** -23 * np.abs(ref)
    assert not bad.any(), f"{bad.sum()} of {bad.size} entries differ from mx_block_matmul_ws beyond the bound"


def test_static_workspace_matches_caller_workspace_on_two_calls():
    one_product(1, 256, 384, 512, mx.E4M3FN, mx.E4M3FN)
    one_product(2, 520, 264, 1024, mx.E2M1, mx.E2M1)


def test_static_workspace_rejects_products_beyond_its_size():
    # M = N = 16384, K = 32768 needs 32 MiB of scale workspace: refused before anything is launched
    M, N, K = 16384, 16384, 32768
    assert mx.mx_block_matmul_workspace_bytes(mx.SCALES_ROWMAJOR, M, N, K) > 16 << 20
    status = mx.lib.mx_block_matmul_static_ws(None, None, mx.E4M3FN, None, None, mx.E4M3FN, mx.SCALES_ROWMAJOR,
                                              32, mx.SCALE_E8M0, M, N, K, None, None)
    assert status == MX_ERR_SHAPE
    assert b"static workspace" in mx.lib.mx_last_error_detail()
