"""GPU parity of mx_block_matmul_ws: block_matmul on operands whose scales are
in the public row-major layout, through a caller-owned workspace.

The workspace receives both operands' scales in the tensor-core layout and the
product then runs on them, so the tests check (1) the workspace's scale bytes
against the tensor-core layout computed on the host from the oracle's scales
(padding zero), and (2) C against the binary64 oracle within the stated
bound, as for mx_block_matmul on the same operands quantized straight into
the tensor-core layout (also checked; where K is split over CTAs the partial
sums reach C in arrival order, so the two agree within the bound, not
always bit for bit).
"""
import numpy as np
import pytest
import torch

import bit_gemm_gb300 as mx
import oracle
from gpu_util import rowmajor_to_mma, to_np
from test_gemm_gpu import O_FMT, check, gpu_quant, host_f32, randn

pytestmark = pytest.mark.gpu


def gathers_scales(M, N, K, fa, fb):
    """Decode shapes, which mx_block_matmul_ws runs on the row-major scales directly."""
    k_stage = 256 if (fa == mx.E2M1 and fb == mx.E2M1) else 128
    return M <= 64 and N > M and -(-M // 16) * 16 <= 32 and K % (2 * k_stage) == 0


def run_ws(A, Bt, fa, fb, C0, canary=True):
    M, K = A.shape
    N = Bt.shape[0]
    ac, as_ = gpu_quant(A, fa, mx.SCALES_ROWMAJOR)
    bc, bs = gpu_quant(Bt, fb, mx.SCALES_ROWMAJOR)
    need = mx.mx_block_matmul_workspace_bytes(mx.SCALES_ROWMAJOR, M, N, K)
    # canary bytes after the workspace: the call writes only what it declares
    ws_full = torch.full((need + 512,), 0xA5, dtype=torch.uint8, device="cuda")
    ws = ws_full[:need]
    C = torch.from_numpy(np.ascontiguousarray(C0, np.float32)).cuda()
    mx.mx_block_matmul_ws(ac, as_, fa, bc, bs, fb, M, N, K, C, ws)
    mx.mx_device_status()
    if canary:
        assert (to_np(ws_full[need:]) == 0xA5).all(), "bytes past the workspace were written"
    oa, osa = oracle.quantize(host_f32(A), O_FMT[fa])
    ob, osb = oracle.quantize(host_f32(Bt), O_FMT[fb])
    w = to_np(ws)
    if gathers_scales(M, N, K, fa, fb):
        # (1') decode shapes read the row-major scales in the product: the
        # workspace is left as it was
        assert (w == 0xA5).all(), "decode shapes leave the workspace untouched"
    else:
        # (1) the workspace holds both operands' scales in the tensor-core layout
        nb = K // 32
        sa_mma = rowmajor_to_mma(osa, M, nb)
        sb_mma = rowmajor_to_mma(osb, N, nb)
        off_b = (sa_mma.size + 255) // 256 * 256
        assert np.array_equal(w[:sa_mma.size], sa_mma), "A scales in the workspace"
        assert np.array_equal(w[off_b:off_b + sb_mma.size], sb_mma), "B scales in the workspace"
    # (2) the product against the oracle
    ref, sabs = oracle.block_matmul(oa, osa, O_FMT[fa], ob, osb, O_FMT[fb], M, N, K, C0)
    check(to_np(C), ref, sabs, C0, f"ws {M}x{N}x{K} {fa}x{fb}")
    # the same product on tensor-core-layout scales meets the same bound
    ac2, as2 = gpu_quant(A, fa, mx.SCALES_MMA)
    bc2, bs2 = gpu_quant(Bt, fb, mx.SCALES_MMA)
    C2 = torch.from_numpy(np.ascontiguousarray(C0, np.float32)).cuda()
    mx.mx_block_matmul(ac2, as2, fa, bc2, bs2, fb, M, N, K, C2, mx.SCALES_MMA)
    mx.mx_device_status()
    check(to_np(C2), ref, sabs, C0, f"tensor-core layout {M}x{N}x{K} {fa}x{fb}")
    return to_np(C)


@pytest.mark.parametrize("M,N,K,fa,fb", [
    (128, 128, 256, mx.E2M1, mx.E2M1),        # one tile
    (130, 260, 384, mx.E4M3FN, mx.E4M3FN),     # ragged rows and columns, one-CTA tiles
    (200, 72, 512, mx.E4M3FN, mx.E2M1),        # mixed formats
    (520, 776, 1024, mx.E2M1, mx.E2M1),       # CTA pairs, ragged
    (640, 520, 2048, mx.E4M3FN, mx.E4M3FN),    # CTA pairs, two K atoms per stage
    (16, 1040, 4096, mx.E4M3FN, mx.E2M1),      # decode shape: the product gathers the scales itself
    (32, 520, 1024, mx.E2M1, mx.E2M1),        # decode shape, FP4, 32 activation rows
    (48, 300, 1024, mx.E4M3FN, mx.E4M3FN),     # 48 rows: relayout, then the product
    (5, 300, 128, mx.E4M3FN, mx.E4M3FN),       # fewer rows than a scale tile
])
def test_rowmajor_through_workspace(M, N, K, fa, fb):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = randn(rng, (M, K))
    Bt = randn(rng, (N, K), 0.05)
    C0 = randn(rng, (M, N))
    run_ws(A, Bt, fa, fb, C0)


def test_workspace_contents_do_not_matter_and_calls_repeat():
    # two calls in a row on one workspace (the first leaves its bytes behind)
    rng = np.random.default_rng(11)
    M, N, K = 260, 384, 512
    A, Bt, C0 = randn(rng, (M, K)), randn(rng, (N, K)), np.zeros((M, N), np.float32)
    ac, as_ = gpu_quant(A, mx.E4M3FN, mx.SCALES_ROWMAJOR)
    bc, bs = gpu_quant(Bt, mx.E4M3FN, mx.SCALES_ROWMAJOR)
    ws = mx.alloc_workspace(M, N, K)
    ws.fill_(0xFF)  # NaN scales if the relayout left any byte unwritten
    C = torch.zeros(M, N, device="cuda")
    mx.mx_block_matmul_ws(ac, as_, mx.E4M3FN, bc, bs, mx.E4M3FN, M, N, K, C, ws)
    mx.mx_block_matmul_ws(ac, as_, mx.E4M3FN, bc, bs, mx.E4M3FN, M, N, K, C, ws)
    mx.mx_device_status()
    oa, osa = oracle.quantize(A, oracle.E4M3)
    ob, osb = oracle.quantize(Bt, oracle.E4M3)
    ref, sabs = oracle.block_matmul(oa, osa, oracle.E4M3, ob, osb, oracle.E4M3, M, N, K, C0)
    check(to_np(C), 2 * ref, 2 * sabs, C0, "two calls")


def test_tensor_core_layout_needs_no_workspace():
    rng = np.random.default_rng(3)
    M, N, K = 130, 140, 256
    A, Bt, C0 = randn(rng, (M, K)), randn(rng, (N, K)), randn(rng, (M, N))
    ac, as_ = gpu_quant(A, mx.E2M1, mx.SCALES_MMA)
    bc, bs = gpu_quant(Bt, mx.E2M1, mx.SCALES_MMA)
    assert mx.mx_block_matmul_workspace_bytes(mx.SCALES_MMA, M, N, K) == 0
    C = torch.from_numpy(C0.copy()).cuda()
    mx.mx_block_matmul_ws(ac, as_, mx.E2M1, bc, bs, mx.E2M1, M, N, K, C, None, mx.SCALES_MMA)
    mx.mx_device_status()
    oa, osa = oracle.quantize(A, oracle.E2M1)
    ob, osb = oracle.quantize(Bt, oracle.E2M1)
    ref, sabs = oracle.block_matmul(oa, osa, oracle.E2M1, ob, osb, oracle.E2M1, M, N, K, C0)
    check(to_np(C), ref, sabs, C0, "tensor-core layout through the workspace entry point")


def test_nan_scale_reaches_outputs_through_workspace():
    # a 0xFF scale in the row-major input survives the relayout and poisons its row
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 256
    A, Bt = randn(rng, (M, K)), randn(rng, (N, K))
    ac, as_ = gpu_quant(A, mx.E4M3FN, mx.SCALES_ROWMAJOR)
    bc, bs = gpu_quant(Bt, mx.E4M3FN, mx.SCALES_ROWMAJOR)
    as_.view(M, K // 32)[7, 3] = 0xFF
    ws = mx.alloc_workspace(M, N, K)
    C = torch.zeros(M, N, device="cuda")
    mx.mx_block_matmul_ws(ac, as_, mx.E4M3FN, bc, bs, mx.E4M3FN, M, N, K, C, ws)
    mx.mx_device_status()
    c = to_np(C)
    assert np.isnan(c[7]).all()
    assert not np.isnan(np.delete(c, 7, axis=0)).any()
