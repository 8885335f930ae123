"""GPU parity of mx_block_matmul_f32b (C += dequantize(A) * B with B a plain
f32 K x N matrix) against the CPU oracle, which forms C0 + sum_k deqA * B in
binary64 from the same codes and scales.  Tolerance as for the MX product:
|C - ref| <= 1e-5 * sum |deqA * b| (plus half an f32 ulp of the result), and
an output with an all-zero sum must equal C0 exactly."""
import numpy as np
import pytest
import torch

import bit_gemm_gb300 as mx
import oracle
import workloads
from gpu_util import rowmajor_to_mma, to_np

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


def run(codes, scales, fmt, B, C0, layout=mx.SCALES_ROWMAJOR):
    """codes/scales: oracle (row-major) arrays; returns C from the GPU."""
    M = scales.shape[0]
    K = B.shape[0]
    s = rowmajor_to_mma(scales, M, K // 32) if layout == mx.SCALES_MMA else scales
    C = torch.from_numpy(np.ascontiguousarray(C0, np.float32)).cuda()
    mx.mx_block_matmul_f32b(torch.from_numpy(np.ascontiguousarray(codes)).cuda(),
                            torch.from_numpy(np.ascontiguousarray(s)).cuda(), fmt,
                            torch.from_numpy(np.ascontiguousarray(B, np.float32)).cuda(), M, C, layout)
    mx.mx_device_status()
    return to_np(C)


def randn(rng, shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
@pytest.mark.parametrize("M,N,K", [
    (1, 4, 32),          # one unit; the second 256-column box wholly past N is not loaded
    (5, 260, 96),        # ragged rows and a part of the second box
    (16, 512, 4096),     # one tile, K split over many CTAs
    (17, 1028, 256),     # two row tiles (one row in the second), three column tiles
    (40, 2048, 1024),
    (64, 516, 2048),
])
def test_shapes(fmt, layout, M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = randn(rng, (M, K)) * np.float32(2.0) ** rng.integers(-6, 6, (M, 1)).astype(np.float32)
    B = randn(rng, (K, N), 0.1)
    C0 = randn(rng, (M, N))
    codes, scales = oracle.quantize(A, O_FMT[fmt])
    got = run(codes, scales, fmt, B, C0, layout)
    ref, sabs = oracle.block_matmul_f32b(codes, scales, O_FMT[fmt], B, M, N, K, C0)
    check(got, ref, sabs, C0, f"{M}x{N}x{K} fmt {fmt} layout {layout}")


def test_many_units_per_cta():
    # more units than SMs many times over, tiles split at arbitrary K steps
    rng = np.random.default_rng(2)
    M, N, K = 200, 3000, 1536
    A = randn(rng, (M, K))
    B = randn(rng, (K, N))
    C0 = np.zeros((M, N), np.float32)
    codes, scales = oracle.quantize(A, oracle.E4M3)
    got = run(codes, scales, mx.E4M3FN, B, C0)
    ref, sabs = oracle.block_matmul_f32b(codes, scales, oracle.E4M3, B, M, N, K, C0)
    check(got, ref, sabs, C0, "200x3000x1536")


def test_special_values():
    # a 0xFF scale poisons its block's products (NaN in the outputs that use it);
    # an all-zero row leaves its outputs equal to C0; inf in B times a zero code
    # is NaN on both sides; subnormal-scale blocks stay exact enough
    rng = np.random.default_rng(5)
    M, N, K = 8, 256, 256
    A = randn(rng, (M, K))
    A[1] = 0.0
    codes, scales = oracle.quantize(A, oracle.E4M3)
    scales[2, 3] = 0xFF
    B = randn(rng, (K, N))
    B[200, 7] = np.inf
    C0 = randn(rng, (M, N))
    got = run(codes, scales, mx.E4M3FN, B, C0)
    ref, sabs = oracle.block_matmul_f32b(codes, scales, oracle.E4M3, B, M, N, K, C0)
    assert np.isnan(got[2]).all()
    assert np.isnan(got[1, 7])  # zero code times inf
    check(got, ref, sabs, C0, "special values")


def test_every_code_value():
    # B = identity (K x K): C = C0 + deq(A) exactly, every code at scales around 127
    K = 256
    rng = np.random.default_rng(9)
    for fmt, ncode in ((mx.E2M1, 16), (mx.E4M3FN, 256)):
        M = 32
        cu = (np.arange(M * K) % ncode).astype(np.uint8).reshape(M, K)
        if fmt == mx.E4M3FN:
            cu[(cu & 0x7F) == 0x7F] = 0x11  # NaN codes are covered by the oracle's pins
            codes = cu
        else:
            codes = (cu[:, 0::2] | (cu[:, 1::2] << 4)).astype(np.uint8)
        scales = rng.integers(120, 135, (M, K // 32)).astype(np.uint8)
        B = np.eye(K, dtype=np.float32)
        got = run(codes, scales, fmt, B, np.zeros((M, K), np.float32))
        want = oracle.dequantize(codes, scales, K, O_FMT[fmt])
        assert np.array_equal(got, want)


def test_workload6_decode_f32b():
    w = workloads.make(6)
    M, N, K = w["M"], w["N"], w["K"]
    codes = mx.alloc_codes(M, K, mx.E4M3FN)
    scales = mx.alloc_scales(M, K)
    mx.mx_quantize(w["A"].cuda(), mx.E4M3FN, codes, scales)
    B = torch.from_numpy(w["B"]).cuda()
    C = torch.from_numpy(w["C0"]).cuda()
    mx.mx_block_matmul_f32b(codes, scales, mx.E4M3FN, B, M, C)
    mx.mx_device_status()
    oc, os_ = oracle.quantize(w["A"].float().numpy(), oracle.E4M3)
    assert np.array_equal(to_np(codes).reshape(oc.shape), oc)
    ref, sabs = oracle.block_matmul_f32b(oc, os_, oracle.E4M3, w["B"], M, N, K, w["C0"])
    check(to_np(C), ref, sabs, w["C0"], "workload 6")
