"""GPU parity of mx_block_matmul_act (activations quantized inside the GEMM)
against the CPU oracle, which quantizes the same f32/bf16 activations itself
and forms C0 + sum_k deqA * deqB in binary64; tolerance as for
mx_block_matmul.  On single-stage shapes the result must also equal, bit for
bit, quantize-then-GEMM through mx_quantize and mx_block_matmul: the two
kernels then do the same MMA arithmetic, so any difference would be a
difference in the codes or scales the kernel produced."""
import numpy as np
import pytest
import torch

import bit_gemm_gb300 as mx
import oracle
import workloads
from gpu_util import to_np

pytestmark = pytest.mark.gpu

O_FMT = {mx.E2M1: oracle.E2M1, mx.E4M3FN: oracle.E4M3}
REL = 1e-5


def check(got, ref, sabs, c0, where):
    got = np.asarray(got, np.float64)
    nan_ref = np.isnan(ref)
    assert np.isnan(got[nan_ref]).all(), f"{where}: NaN expected"
    inf_ref = np.isinf(ref)
    assert (got[inf_ref] == ref[inf_ref]).all(), f"{where}: infinity expected"
    ok = ~(nan_ref | inf_ref)
    err = np.abs(got[ok] - ref[ok])
    tol = REL * sabs[ok] + np.abs(ref[ok]) * 2.0 ** -23
    zero = sabs[ok] == 0
    # a NaN or an infinity where the reference is finite fails too
    bad = ~(err <= tol) | (zero & (got[ok] != np.asarray(c0, np.float64)[ok]))
    assert not bad.any(), f"{where}: {bad.sum()} of {bad.size} entries outside tolerance"


def weights(Bt: np.ndarray, fb: int):
    N, K = Bt.shape
    bc, bs = mx.alloc_codes(N, K, fb), mx.alloc_scales(N, K, mx.SCALES_MMA)
    mx.mx_quantize(torch.from_numpy(Bt).cuda(), fb, bc, bs, mx.SCALES_MMA)
    return bc, bs


def fused_vs_oracle(A: torch.Tensor, Bt: np.ndarray, fa: int, fb: int, C0: np.ndarray):
    M, K = A.shape
    N = Bt.shape[0]
    bc, bs = weights(Bt, fb)
    C = torch.from_numpy(np.ascontiguousarray(C0, np.float32)).cuda()
    mx.mx_block_matmul_act(A.cuda(), fa, bc, bs, fb, N, C)
    mx.mx_device_status()
    oa, osa = oracle.quantize(A.float().numpy(), O_FMT[fa])
    ob, osb = oracle.quantize(Bt, O_FMT[fb])
    ref, sabs = oracle.block_matmul(oa, osa, O_FMT[fa], ob, osb, O_FMT[fb], M, N, K, C0)
    check(to_np(C), ref, sabs, C0, f"{M}x{N}x{K} {fa}x{fb} {A.dtype}")
    return to_np(C)


def randn(rng, shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


def test_workload3_decode_fused():
    w = workloads.make(3)
    fused_vs_oracle(w["A"], w["W"], mx.E4M3FN, mx.E2M1, w["C0"])


@pytest.mark.parametrize("M,N,K,fa,fb,dtype", [
    (1, 260, 256, mx.E4M3FN, mx.E4M3FN, torch.float32),
    (5, 300, 384, mx.E2M1, mx.E2M1, torch.bfloat16),      # FP4 stages of 256: the second is half
    (33, 998, 512, mx.E4M3FN, mx.E2M1, torch.bfloat16),   # N % 4 != 0: per-element epilogue
    (64, 512, 8192, mx.E4M3FN, mx.E4M3FN, torch.bfloat16),  # K over eight launches (8 resident stages)
    (16, 256, 8192, mx.E4M3FN, mx.E2M1, torch.float32),   # K over two launches (32 resident stages)
    (48, 130, 160, mx.E2M1, mx.E2M1, torch.float32),      # K shorter than one FP4 stage
    (20, 1024, 2048, mx.E2M1, mx.E2M1, torch.bfloat16),   # split along K across CTAs
])
def test_fused_shapes(M, N, K, fa, fb, dtype):
    rng = np.random.default_rng(M * 13 + N * 7 + K)
    A = torch.from_numpy(randn(rng, (M, K)) * np.float32(2.0) ** rng.integers(-8, 8, (M, 1)).astype(np.float32))
    fused_vs_oracle(A.to(dtype), randn(rng, (N, K), 0.05), fa, fb, randn(rng, (M, N)))


def test_fused_special_values():
    # zero rows, a NaN (its block's scale 0xFF poisons its products), subnormals
    rng = np.random.default_rng(31)
    M, N, K = 8, 256, 256
    A = randn(rng, (M, K))
    A[1] = 0.0
    A[2, 40] = np.nan
    A[3] = np.float32(2.0 ** -140) * np.arange(K, dtype=np.float32)
    A[4, :32] = -0.0
    fused_vs_oracle(torch.from_numpy(A), randn(rng, (N, K)), mx.E4M3FN, mx.E4M3FN, np.zeros((M, N), np.float32))


@pytest.mark.parametrize("fa,fb,dtype", [(mx.E4M3FN, mx.E2M1, torch.bfloat16), (mx.E4M3FN, mx.E4M3FN, torch.float32),
                                         (mx.E2M1, mx.E2M1, torch.bfloat16)])
@pytest.mark.parametrize("M,N", [(16, 128), (7, 384), (64, 256)])
def test_fused_equals_quantize_then_gemm_bitwise(fa, fb, dtype, M, N):
    rng = np.random.default_rng(M + N)
    K = 256 if fa == mx.E2M1 else 128  # one stage: both kernels run the same four MMAs per tile
    A = torch.from_numpy(randn(rng, (M, K)) * np.float32(3.0)).to(dtype)
    bc, bs = weights(randn(rng, (N, K)), fb)
    C0 = randn(rng, (M, N))
    C1 = torch.from_numpy(C0).cuda()
    mx.mx_block_matmul_act(A.cuda(), fa, bc, bs, fb, N, C1)
    ac, as_ = mx.alloc_codes(M, K, fa), mx.alloc_scales(M, K, mx.SCALES_MMA)
    mx.mx_quantize(A.cuda(), fa, ac, as_, mx.SCALES_MMA)
    C2 = torch.from_numpy(C0).cuda()
    mx.mx_block_matmul(ac, as_, fa, bc, bs, fb, M, N, K, C2, mx.SCALES_MMA)
    mx.mx_device_status()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))


# ------------------------------------------- bf16 activations streamed by stage
# Up to 16 bf16 rows with K a whole number of two-atom stages (256 elements for
# E4M3FN activations, 512 for E2M1): the activations are quantized stage by
# stage into the kernel's ring.  Everything else takes the resident path above.

@pytest.mark.parametrize("M,N,K,fa,fb", [
    (1, 130, 256, mx.E4M3FN, mx.E4M3FN),       # one stage, one real row
    (5, 1000, 1024, mx.E4M3FN, mx.E2M1),       # ragged weight tiles, split along K
    (16, 2052, 768, mx.E4M3FN, mx.E4M3FN),     # three stages
    (16, 1030, 512, mx.E4M3FN, mx.E2M1),       # N % 4 != 0: per-element epilogue
    (9, 384, 4096, mx.E2M1, mx.E2M1),          # packed FP4 stages of 512
    (16, 19500, 256, mx.E4M3FN, mx.E4M3FN),    # more tiles than SMs: whole tiles
])
def test_streamed_shapes(M, N, K, fa, fb):
    rng = np.random.default_rng(M * 7 + N + K)
    A = torch.from_numpy(randn(rng, (M, K)) * np.float32(2.0) ** rng.integers(-6, 6, (M, 1)).astype(np.float32))
    fused_vs_oracle(A.to(torch.bfloat16), randn(rng, (N, K), 0.05), fa, fb, randn(rng, (M, N)))


@pytest.mark.parametrize("M,N,K,fa,fb", [
    (16, 1000, 768, mx.E4M3FN, mx.E2M1),       # three stages
    (3, 384, 512, mx.E4M3FN, mx.E4M3FN),       # two stages
    (16, 512, 1024, mx.E2M1, mx.E2M1),         # two FP4 stages
    (16, 19500, 256, mx.E4M3FN, mx.E4M3FN),    # more tiles than SMs
])
def test_streamed_equals_quantize_then_gemm_bitwise(M, N, K, fa, fb):
    # same MMAs, same schedule as mx_quantize + mx_block_matmul: equal bit for
    # bit on shapes whose tiles each stay on one CTA (fewer than four stages,
    # or more tiles than SMs); split along K, partial sums meet in C through
    # reduce-adds in whatever order they land, so only the tolerance holds
    rng = np.random.default_rng(M + N + K)
    A = torch.from_numpy(randn(rng, (M, K)) * np.float32(3.0)).to(torch.bfloat16)
    bc, bs = weights(randn(rng, (N, K)), fb)
    C0 = randn(rng, (M, N))
    C1 = torch.from_numpy(C0).cuda()
    mx.mx_block_matmul_act(A.cuda(), fa, bc, bs, fb, N, C1)
    ac, as_ = mx.alloc_codes(M, K, fa), mx.alloc_scales(M, K, mx.SCALES_MMA)
    mx.mx_quantize(A.cuda(), fa, ac, as_, mx.SCALES_MMA)
    C2 = torch.from_numpy(C0).cuda()
    mx.mx_block_matmul(ac, as_, fa, bc, bs, fb, M, N, K, C2, mx.SCALES_MMA)
    mx.mx_device_status()
    assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))


def test_streamed_special_values():
    # bf16: zero rows, a NaN and an infinity (their blocks' scales 0xFF poison
    # their products), subnormals, negative zeros
    rng = np.random.default_rng(37)
    M, N, K = 16, 256, 512
    A = randn(rng, (M, K))
    A[1] = 0.0
    A[2, 40] = np.nan
    A[5, 300] = -np.inf
    A[3] = np.float32(2.0 ** -130) * np.arange(K, dtype=np.float32)
    A[4, :32] = -0.0
    fused_vs_oracle(torch.from_numpy(A).to(torch.bfloat16), randn(rng, (N, K)), mx.E4M3FN, mx.E2M1,
                    np.zeros((M, N), np.float32))
