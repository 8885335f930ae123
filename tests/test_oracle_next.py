"""Pins for the oracle's functions beyond the three core ops: quantize along
the first axis, dequantize to bfloat16, the product with an f32 right-hand
operand, and fold_scale.  Each is checked against something other than itself:
a mathematical identity evaluated through separately pinned oracle functions
and numpy / torch library routines, closed forms, and literal values."""
import numpy as np
import pytest
import torch

import oracle

FMTS = [oracle.E2M1, oracle.E4M3]


def rand(rng, shape, spread=20):
    """Normal values with per-row power-of-two spreads, a few zeros, negatives
    and exact grid values."""
    x = rng.standard_normal(shape).astype(np.float32)
    x *= np.float32(2.0) ** rng.integers(-spread, spread, (shape[0], 1)).astype(np.float32)
    x.flat[rng.integers(0, x.size, max(1, x.size // 50))] = 0.0
    return x


# --------------------------------------------------------------- block axis 0

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("rows,cols", [(32, 1), (64, 33), (96, 7), (128, 130), (256, 3)])
def test_axis0_is_quantize_of_the_transpose(fmt, rows, cols):
    # [Dialect] "The block axis": blocks run along the reduction axis; for a
    # K x N operand that is axis 0, i.e. the rows of its transpose.
    rng = np.random.default_rng(rows * 1000 + cols)
    x = rand(rng, (rows, cols))
    c0, s0 = oracle.quantize_axis0(x, fmt)
    c1, s1 = oracle.quantize(np.ascontiguousarray(x.T), fmt)
    assert np.array_equal(c0, c1) and np.array_equal(s0, s1)


def test_axis0_literal_column():
    # one column whose 32-element block is 6 at the top and 0.5 elsewhere, E2M1:
    # amax 6 -> e = 2 - 2 = 0 -> scale 127; codes 7 (6.0) and 1 (0.5)
    x = np.zeros((32, 3), np.float32)
    x[:, 1] = 0.5
    x[0, 1] = 6.0
    codes, scales = oracle.quantize_axis0(x, oracle.E2M1)
    assert scales.shape == (3, 1) and scales[1, 0] == 127 and scales[0, 0] == 127
    assert codes[1, 0] == 0x17 and (codes[1, 1:] == 0x11).all()
    assert (codes[0] == 0).all() and (codes[2] == 0).all()


def test_axis0_rejects_partial_blocks():
    with pytest.raises(ValueError):
        oracle.quantize_axis0(np.zeros((48, 4), np.float32), oracle.E4M3)


# -------------------------------------------------------- dequantize to bf16

@pytest.mark.parametrize("fmt", FMTS)
def test_dequantize_bf16_every_code_and_scale(fmt):
    # the exact value (pinned f32 dequantize) rounded by torch's f32 -> bfloat16
    # conversion (round to nearest, ties to even)
    ncodes = 16 if fmt == oracle.E2M1 else 256
    codes_u = np.repeat(np.arange(ncodes, dtype=np.uint8), 256)
    scales = np.tile(np.arange(256, dtype=np.uint8), ncodes)
    rows = codes_u.size
    cols = 32
    cu = np.repeat(codes_u[:, None], cols, axis=1)
    codes = (cu[:, 0::2] | (cu[:, 1::2] << 4)).astype(np.uint8) if fmt == oracle.E2M1 else cu
    s = scales[:, None]
    y32 = oracle.dequantize(codes, s, cols, fmt)
    want = torch.from_numpy(y32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.dequantize_bf16(codes, s, cols, fmt)
    nan_w = np.isnan(y32)
    got_f = (got.astype(np.uint32) << 16).view(np.float32)
    assert np.isnan(got_f[nan_w]).all()
    assert np.array_equal(got[~nan_w], want[~nan_w])


def test_dequantize_bf16_literals():
    # E4M3 448 x 2^127 overflows to +inf; 2^-9 x 2^-127 = 2^-136 is below half the
    # smallest bfloat16 subnormal (2^-133) and rounds to +0; 1.125 x 2^0 needs 4
    # significant bits and is exact
    codes = np.array([[0x7E] * 32, [0x01] * 32, [0x39] * 32], np.uint8)
    scales = np.array([[254], [0], [127]], np.uint8)
    y = oracle.dequantize_bf16(codes, scales, 32, oracle.E4M3)
    assert (y[0] == 0x7F80).all() and (y[1] == 0x0000).all() and (y[2] == 0x3F90).all()


# ------------------------------------------------------------ f32 right operand

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,N,K", [(3, 5, 32), (17, 9, 96), (64, 33, 256)])
def test_f32b_matches_numpy(fmt, M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A = rand(rng, (M, K), 8)
    B = rand(rng, (K, N), 8)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    ac, as_ = oracle.quantize(A, fmt)
    deqA = oracle.dequantize(ac, as_, K, fmt).astype(np.float64)
    ref, sabs = oracle.block_matmul_f32b(ac, as_, fmt, B, M, N, K, C0)
    want = C0.astype(np.float64) + deqA @ B.astype(np.float64)
    assert np.all(np.abs(ref - want) <= 1e-13 * (sabs + np.abs(C0)))
    assert np.allclose(sabs, np.abs(deqA) @ np.abs(B.astype(np.float64)), rtol=1e-13, atol=0)


def test_f32b_equals_mx_product_when_b_is_representable():
    # B drawn from the E2M1 grid with a 6 in every 32-block of each column, so
    # quantizing B along K is exact (scale 127): the two products then sum the
    # same exact terms in the same order
    rng = np.random.default_rng(5)
    M, N, K = 20, 12, 128
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    B = rng.choice(grid, (K, N)) * rng.choice([-1, 1], (K, N)).astype(np.float32)
    B[0::32, :] = 6.0
    A = rand(rng, (M, K), 6)
    C0 = rng.standard_normal((M, N)).astype(np.float32)
    ac, as_ = oracle.quantize(A, oracle.E4M3)
    bc, bs = oracle.quantize_axis0(B, oracle.E2M1)
    assert (bs == 127).all()
    r1, s1 = oracle.block_matmul_f32b(ac, as_, oracle.E4M3, B, M, N, K, C0)
    r2, s2 = oracle.block_matmul(ac, as_, oracle.E4M3, bc, bs, oracle.E2M1, M, N, K, C0)
    assert np.array_equal(r1, r2) and np.array_equal(s1, s2)


# ---------------------------------------------------------------- fold_scale

@pytest.mark.parametrize("fmt", FMTS)
def test_fold_scale_multiplies_by_power_of_two(fmt):
    rng = np.random.default_rng(11)
    rows, cols = 64, 256
    codes = rng.integers(0, 256, (rows, cols if fmt == oracle.E4M3 else cols // 2), dtype=np.uint8)
    scales = rng.integers(60, 190, (rows, cols // 32), dtype=np.uint8)
    y = oracle.dequantize(codes, scales, cols, fmt)
    for j in (-40, -7, -1, 0, 1, 9, 60):
        yj = oracle.dequantize(codes, oracle.fold_scale(scales, j), cols, fmt)
        with np.errstate(over="ignore"):  # values beyond binary32 become inf on both sides
            want = np.ldexp(y.astype(np.float64), j).astype(np.float32)
        same = (yj == want) | (np.isnan(yj) & np.isnan(want))
        assert same.all(), j


def test_fold_scale_saturates_and_keeps_nan():
    s = np.array([0, 1, 3, 127, 250, 254, 255], np.uint8)
    assert list(oracle.fold_scale(s, 10)) == [10, 11, 13, 137, 254, 254, 255]
    assert list(oracle.fold_scale(s, -10)) == [0, 0, 0, 117, 240, 244, 255]
    assert list(oracle.fold_scale(s, 300)) == [254, 254, 254, 254, 254, 254, 255]


def test_fold_exponent():
    assert oracle.fold_exponent(1.0) == 0
    assert oracle.fold_exponent(0.125) == -3
    assert oracle.fold_exponent(2.0 ** 100) == 100
    assert oracle.fold_exponent(2.0 ** -140) == -140
    for bad in (3.0, -2.0, 0.0, -0.0, float("inf"), float("nan"), 1.5, 0.75):
        assert oracle.fold_exponent(bad) is None, bad
