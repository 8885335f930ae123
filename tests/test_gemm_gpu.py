"""GPU parity of mx_block_matmul against the CPU oracle.

The oracle quantizes the same seeded f32/bf16 inputs itself (never the GPU's
codes) and forms C0 + sum_k deqA*deqB in binary64.  The bound is the stated
one, |gpu - oracle| <= 1e-5 * sum_k |deqA*deqB|, plus one binary32 rounding of
the output itself (an f32 result cannot be closer than that); an entry whose
products are all zero must equal C0 exactly, and a NaN in the oracle must be a
NaN on the GPU.  At full size the check runs on sampled rows, columns and
entries, each computed by the oracle one by one."""
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


def gpu_quant(x, fmt, layout=mx.SCALES_MMA):
    x = torch.as_tensor(x)
    rows, cols = x.shape
    codes, scales = mx.alloc_codes(rows, cols, fmt), mx.alloc_scales(rows, cols, layout)
    mx.mx_quantize(x.cuda(), fmt, codes, scales, layout)
    return codes, scales


def host_f32(x):
    return x.float().numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float32)


def check(got, ref, sabs, c0, where=""):
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
    if bad.any():
        i = np.flatnonzero(bad)[:8]
        ratio = got[ok][i] / np.where(ref[ok][i] == 0, 1, ref[ok][i])
        raise AssertionError(f"{where}: {bad.sum()} of {bad.size} outside tolerance; got {got[ok][i]}, "
                             f"ref {ref[ok][i]}, sabs {sabs[ok][i]}, ratio {ratio}")


def run_full(A, Bt, fa, fb, C0, layout=mx.SCALES_MMA, repeat=1):
    """GEMM of host inputs on the GPU, checked against the full oracle product."""
    M, K = A.shape
    N = Bt.shape[0]
    ac, as_ = gpu_quant(A, fa, layout)
    bc, bs = gpu_quant(Bt, fb, layout)
    C = torch.from_numpy(np.ascontiguousarray(C0, np.float32)).cuda()
    for _ in range(repeat):
        mx.mx_block_matmul(ac, as_, fa, bc, bs, fb, M, N, K, C, layout)
    mx.mx_device_status()
    oa, osa = oracle.quantize(host_f32(A), O_FMT[fa])
    ob, osb = oracle.quantize(host_f32(Bt), O_FMT[fb])
    ref, sabs = oracle.block_matmul(oa, osa, O_FMT[fa], ob, osb, O_FMT[fb], M, N, K, C0)
    if repeat > 1:
        ref = C0.astype(np.float64) + repeat * (ref - C0.astype(np.float64))
        sabs = repeat * sabs
    check(to_np(C), ref, sabs, C0, f"{M}x{N}x{K} {fa}x{fb}")
    return to_np(C), ref


def randn(rng, shape, std=1.0):
    return (rng.standard_normal(shape) * std).astype(np.float32)


# --------------------------------------------------------- small and exact

def test_workload1_mxfp4_128():
    w = workloads.make(1)
    run_full(w["A"], w["Bt"], mx.E2M1, mx.E2M1, w["C0"])


@pytest.mark.parametrize("fa,fb", [(mx.E4M3FN, mx.E4M3FN), (mx.E2M1, mx.E2M1), (mx.E4M3FN, mx.E2M1),
                                   (mx.E2M1, mx.E4M3FN)])
def test_format_pairs_one_tile(fa, fb):
    rng = np.random.default_rng(21)
    A, Bt = randn(rng, (128, 256)), randn(rng, (128, 256))
    run_full(A, Bt, fa, fb, randn(rng, (128, 128)))


@pytest.mark.parametrize("fa,fb", [(mx.E4M3FN, mx.E4M3FN), (mx.E2M1, mx.E2M1)])
def test_integer_valued_product_is_exact(fa, fb):
    # grid values with all scales 2^0: every partial sum is a small dyadic
    # number, so f32 accumulation is exact and the result must equal the oracle.
    rng = np.random.default_rng(22)
    g = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    A = rng.choice(g, (128, 256)) * rng.choice([-1, 1], (128, 256)).astype(np.float32)
    Bt = rng.choice(g, (256, 256)) * rng.choice([-1, 1], (256, 256)).astype(np.float32)
    A[:, 0], Bt[:, 0] = 6.0 if fa == mx.E2M1 else 4.0, 6.0 if fb == mx.E2M1 else 4.0
    C0 = rng.integers(-4, 4, (128, 256)).astype(np.float32)
    got, ref = run_full(A.astype(np.float32), Bt.astype(np.float32), fa, fb, C0)
    assert np.array_equal(got.astype(np.float64), ref)


def test_accumulates_into_c_in_place():
    w = workloads.make(1)
    rng = np.random.default_rng(23)
    run_full(w["A"], w["Bt"], mx.E2M1, mx.E2M1, randn(rng, (128, 128)), repeat=2)


def test_nan_scale_reaches_its_row():
    rng = np.random.default_rng(24)
    A, Bt = randn(rng, (128, 128)), randn(rng, (128, 128))
    A[5, 40] = np.nan  # the block of row 5 holding k = 40 gets scale 0xFF
    run_full(A, Bt, mx.E4M3FN, mx.E4M3FN, np.zeros((128, 128), np.float32))


# ------------------------------------------------------------ ragged shapes

@pytest.mark.parametrize("M,N,K,fa,fb", [
    (200, 300, 160, mx.E4M3FN, mx.E4M3FN),   # ragged M, N and K (a partial last stage)
    (200, 300, 96, mx.E2M1, mx.E2M1),        # K shorter than one stage
    (130, 130, 128, mx.E4M3FN, mx.E2M1),     # N % 4 != 0: per-element epilogue
    (1, 260, 256, mx.E2M1, mx.E2M1),         # single row, swapped operands
    (64, 1000, 512, mx.E4M3FN, mx.E4M3FN),   # swapped, 64 rows
    (48, 384, 384, mx.E2M1, mx.E4M3FN),      # swapped, mixed
    (256, 512, 8192, mx.E4M3FN, mx.E4M3FN),  # few tiles, long K: split along K across CTAs
    (300, 520, 32, mx.E4M3FN, mx.E4M3FN),    # a single 32-element block
])
def test_ragged_shapes(M, N, K, fa, fb):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    run_full(randn(rng, (M, K)), randn(rng, (N, K)), fa, fb, randn(rng, (M, N)))


# ------------------------------------------------ 256 x 256 tiles on CTA pairs

@pytest.mark.parametrize("M,N,K,fa,fb", [
    (512, 512, 1024, mx.E4M3FN, mx.E4M3FN),
    (300, 600, 416, mx.E2M1, mx.E2M1),       # ragged K with an odd count of 4-block scale groups
    (260, 1000, 384, mx.E4M3FN, mx.E2M1),    # the odd CTA's A rows mostly past M
    (520, 260, 1152, mx.E2M1, mx.E4M3FN),    # the odd CTA's B rows mostly past N (mixed: K % 128 == 0)
    (129, 129, 64, mx.E4M3FN, mx.E4M3FN),    # N % 4 != 0 (per-element epilogue), K shorter than a stage
    (1024, 768, 2048, mx.E2M1, mx.E2M1),     # few tiles, K split across pairs
    (2048, 2048, 256, mx.E4M3FN, mx.E4M3FN), # several tiles per pair
])
def test_pair_tiles(M, N, K, fa, fb):
    rng = np.random.default_rng(M * 5 + N * 11 + K)
    run_full(randn(rng, (M, K)), randn(rng, (N, K)), fa, fb, randn(rng, (M, N)))


# ---------------------------------------- two K atoms per pipeline stage

@pytest.mark.parametrize("M,N,K,fa,fb", [
    (32, 1000, 512, mx.E4M3FN, mx.E2M1),     # decode-shaped, MMA N = 32, mixed formats
    (5, 1300, 1024, mx.E2M1, mx.E2M1),       # decode-shaped, packed FP4 atoms of 256 elements
    (17, 2052, 768, mx.E4M3FN, mx.E4M3FN),   # MMA N = 32 with 17 real rows, ragged weight tiles
    (16, 1030, 512, mx.E4M3FN, mx.E4M3FN),   # N % 4 != 0: the per-element epilogue
    (2560, 2048, 1024, mx.E4M3FN, mx.E4M3FN),  # pairs: 80 tiles on 76 pairs, the last 4 split along K
])
def test_two_atom_stages(M, N, K, fa, fb):
    rng = np.random.default_rng(M * 3 + N + K)
    run_full(randn(rng, (M, K)), randn(rng, (N, K)), fa, fb, randn(rng, (M, N)))


# ------------------------------------------------------ row-major scales

@pytest.mark.parametrize("M,N,K,fa,fb", [
    (128, 128, 256, mx.E2M1, mx.E2M1),
    (200, 300, 384, mx.E4M3FN, mx.E4M3FN),   # ragged M and N: scale rows past the end read as zero
    (130, 512, 128, mx.E4M3FN, mx.E2M1),
    (16, 1024, 512, mx.E4M3FN, mx.E2M1),     # swapped operands, two K atoms per stage
    (16, 1040, 4096, mx.E4M3FN, mx.E2M1),    # decode shape, ragged weight rows, split along K
    (5, 300, 1024, mx.E4M3FN, mx.E4M3FN),    # fewer activation rows than a scale tile
    (32, 264, 1024, mx.E2M1, mx.E2M1),       # FP4, two scale groups per atom, 32 activation rows
    (48, 520, 1024, mx.E2M1, mx.E4M3FN),     # 48 activation rows: one-atom stages
    (256, 512, 8192, mx.E2M1, mx.E2M1),      # split along K across CTAs
])
def test_row_major_scales(M, N, K, fa, fb):
    rng = np.random.default_rng(M + 2 * N + 3 * K)
    run_full(randn(rng, (M, K)), randn(rng, (N, K)), fa, fb, randn(rng, (M, N)), layout=mx.SCALES_ROWMAJOR)


# ------------------------------------------------------- workload 3 (decode)

def test_workload3_decode_full():
    w = workloads.make(3)
    run_full(w["A"], w["W"], mx.E4M3FN, mx.E2M1, w["C0"])


def test_workload3_decode_full_row_major_scales():
    # the public scale layout, gathered by the producer lanes (two K atoms per stage)
    w = workloads.make(3)
    run_full(w["A"], w["W"], mx.E4M3FN, mx.E2M1, w["C0"], layout=mx.SCALES_ROWMAJOR)


# --------------------------------------------- workloads 4 and 5, sampled

def sampled_check(A, Bt, fa, fb, C0, seed, n_rows=64, n_cols=64, n_rand=4096):
    M, K = A.shape
    N = Bt.shape[0]
    ac, as_ = gpu_quant(A, fa)
    bc, bs = gpu_quant(Bt, fb)
    C = torch.from_numpy(C0).cuda()
    mx.mx_block_matmul(ac, as_, fa, bc, bs, fb, M, N, K, C, mx.SCALES_MMA)
    mx.mx_device_status()
    rng = np.random.default_rng(seed)
    rows = rng.choice(M, n_rows, replace=False)
    cols = rng.choice(N, n_cols, replace=False)
    em = np.concatenate([np.repeat(rows, 32), rng.integers(0, M, n_cols * 32), rng.integers(0, M, n_rand)])
    en = np.concatenate([rng.integers(0, N, n_rows * 32), np.repeat(cols, 32), rng.integers(0, N, n_rand)])
    um, im = np.unique(em, return_inverse=True)
    un, in_ = np.unique(en, return_inverse=True)
    Ah, Bh = host_f32(A[torch.from_numpy(um)] if isinstance(A, torch.Tensor) else A[um]), host_f32(Bt[un])
    oa, osa = oracle.quantize(Ah, O_FMT[fa])
    ob, osb = oracle.quantize(Bh, O_FMT[fb])
    c0 = C0[em, en]
    ref, sabs = oracle.block_matmul_entries(oa, osa, O_FMT[fa], ob, osb, O_FMT[fb], K, im, in_, c0)
    got = to_np(C)[em, en]
    check(got, ref, sabs, c0, "sampled")


def test_workload4_square_mxfp8_sampled():
    w = workloads.make(4)
    sampled_check(w["A"], w["Bt"], mx.E4M3FN, mx.E4M3FN, w["C0"], seed=4)


def test_workload5_prefill_mxfp4_sampled():
    w = workloads.make(5)
    sampled_check(w["A"], w["W"], mx.E2M1, mx.E2M1, w["C0"], seed=5)


def test_measure_mma_rate():
    # the tensor pipe on shared-memory operands: somewhere between a quarter of
    # and twice the nominal dense rates (4.5 PF FP8, 13.5 PF FP4)
    f8 = mx.mx_measure_mma_rate(mx.E4M3FN, 2000)
    f4 = mx.mx_measure_mma_rate(mx.E2M1, 2000)
    mx.mx_device_status()
    assert 1000 < f8 < 9000, f8
    assert 2000 < f4 < 27000, f4
    assert f4 > 1.5 * f8
