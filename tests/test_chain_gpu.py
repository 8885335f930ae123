"""Dependent calls back to back on one stream, with no host synchronization
between them.  Every kernel may start its set-up while the previous one
drains (programmatic dependent launch) and must not touch global memory
before the previous kernel's writes are visible; a chain whose every step
reads what the step before wrote checks that, bit for bit, against the same
steps run one at a time."""
import numpy as np
import pytest
import torch

import bit_gemm_gb300 as mx
from gpu_util import to_np

pytestmark = pytest.mark.gpu


def test_quantize_dequantize_chain():
    # x -> q -> deq -> q -> deq ... : each quantize reads the previous dequantize's output
    g = torch.Generator(device="cuda").manual_seed(1)
    rows, cols = 512, 1024
    x = torch.randn(rows, cols, device="cuda", generator=g) * 3
    codes = [mx.alloc_codes(rows, cols, mx.E4M3FN) for _ in range(2)]
    scales = [mx.alloc_scales(rows, cols) for _ in range(2)]
    ys = [torch.empty(rows, cols, device="cuda") for _ in range(2)]
    steps = 24
    cur = x
    for i in range(steps):
        c, s, y = codes[i & 1], scales[i & 1], ys[i & 1]
        mx.mx_quantize(cur, mx.E4M3FN, c, s)
        mx.mx_dequantize(c, s, rows, cols, mx.E4M3FN, y)
        cur = y * 1.0 if i % 5 == 4 else y  # an occasional torch kernel in between
    torch.cuda.synchronize()
    got = to_np(cur)
    # the same steps, synchronizing after every call
    ref = x
    for i in range(steps):
        c, s = mx.alloc_codes(rows, cols, mx.E4M3FN), mx.alloc_scales(rows, cols)
        y = torch.empty(rows, cols, device="cuda")
        mx.mx_quantize(ref, mx.E4M3FN, c, s)
        torch.cuda.synchronize()
        mx.mx_dequantize(c, s, rows, cols, mx.E4M3FN, y)
        torch.cuda.synchronize()
        ref = y
    mx.mx_device_status()
    assert np.array_equal(got.view(np.uint32), to_np(ref).view(np.uint32))


def test_quantize_gemm_chain_accumulates():
    # C += A_i * W for several freshly quantized A_i, no syncs: every GEMM
    # reads the codes the quantize before it wrote and the C the GEMM before it wrote
    g = torch.Generator(device="cuda").manual_seed(2)
    M, N, K = 16, 1024, 1024
    W = torch.randn(N, K, device="cuda", generator=g) * 0.05
    wc, ws = mx.alloc_codes(N, K, mx.E2M1), mx.alloc_scales(N, K, mx.SCALES_MMA)
    mx.mx_quantize(W, mx.E2M1, wc, ws, mx.SCALES_MMA)
    As = [torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16) for _ in range(6)]
    ac, as_ = mx.alloc_codes(M, K, mx.E4M3FN), mx.alloc_scales(M, K, mx.SCALES_MMA)
    C = torch.zeros(M, N, device="cuda")
    for A in As:
        mx.mx_quantize(A, mx.E4M3FN, ac, as_, mx.SCALES_MMA)
        mx.mx_block_matmul(ac, as_, mx.E4M3FN, wc, ws, mx.E2M1, M, N, K, C, mx.SCALES_MMA)
    torch.cuda.synchronize()
    Cref = torch.zeros(M, N, device="cuda")
    for A in As:
        c2, s2 = mx.alloc_codes(M, K, mx.E4M3FN), mx.alloc_scales(M, K, mx.SCALES_MMA)
        mx.mx_quantize(A, mx.E4M3FN, c2, s2, mx.SCALES_MMA)
        torch.cuda.synchronize()
        mx.mx_block_matmul(c2, s2, mx.E4M3FN, wc, ws, mx.E2M1, M, N, K, Cref, mx.SCALES_MMA)
        torch.cuda.synchronize()
    mx.mx_device_status()
    # the reductions into C may add partial sums in another order: compare to f32 rounding
    assert torch.allclose(C, Cref, rtol=1e-5, atol=1e-5)
