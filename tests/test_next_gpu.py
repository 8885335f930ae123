"""GPU parity of the entry points beyond the three core ops, against the CPU
oracle: quantize along the first axis (mx_quantize_axis), dequantize to
bfloat16 (mx_dequantize_bf16) and fold_scale (mx_fold_scale).  Codes, scales
and bfloat16 outputs are compared bit for bit."""
import numpy as np
import pytest
import torch

import bit_gemm_gb300 as mx
import oracle
from gpu_util import mma_padding_mask, mma_to_rowmajor, rowmajor_to_mma, to_np

pytestmark = pytest.mark.gpu

O_FMT = {mx.E2M1: oracle.E2M1, mx.E4M3FN: oracle.E4M3}
GUARD = 256


def rand(rng, shape, spread=25):
    x = rng.standard_normal(shape).astype(np.float32)
    x *= np.float32(2.0) ** rng.integers(-spread, spread, (1, shape[1])).astype(np.float32)
    x.flat[rng.integers(0, x.size, max(1, x.size // 64))] = 0.0
    x.flat[rng.integers(0, x.size, max(1, x.size // 64))] = -0.0
    return x


def axis0_gpu(x: torch.Tensor, fmt: int, layout: int, codes_offset: int = 0):
    """codes_offset: start the codes this many bytes into their buffer (16 puts
    them on a 16- but not a 32-byte boundary, which the register kernel for
    bf16 input does not take)."""
    rows, cols = x.shape
    cb, sb = mx.mx_codes_bytes(fmt, cols, rows), mx.mx_scales_bytes(layout, cols, rows)
    codes_buf = torch.full((codes_offset + cb + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    codes = codes_buf[codes_offset:]
    scales = torch.full((sb + GUARD,), 0x5A, dtype=torch.uint8, device="cuda")
    mx.mx_quantize_axis(x.cuda(), 0, fmt, codes, scales, layout)
    mx.mx_device_status()
    c, s = to_np(codes_buf), to_np(scales)
    assert (c[:codes_offset] == 0xA5).all(), "wrote before the codes"
    c = c[codes_offset:]
    assert (c[cb:] == 0xA5).all() and (s[sb:] == 0x5A).all(), "wrote past the end"
    return c[:cb], s[:sb]


def check_axis0(x: torch.Tensor, fmt: int, layout: int, codes_offset: int = 0):
    rows, cols = x.shape
    codes, scales = axis0_gpu(x, fmt, layout, codes_offset)
    oc, os_ = oracle.quantize_axis0(x.float().numpy(), O_FMT[fmt])
    assert np.array_equal(codes.reshape(oc.shape), oc), "codes differ from the oracle"
    nb = rows // 32
    if layout == mx.SCALES_MMA:
        assert np.array_equal(mma_to_rowmajor(scales, cols, nb), os_)
        assert (scales[mma_padding_mask(cols, nb)] == 0).all()
    else:
        assert np.array_equal(scales.reshape(os_.shape), os_)


# --------------------------------------------------------------- block axis 0

@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
def test_axis0_shapes(fmt, dtype, layout):
    rng = np.random.default_rng(3)
    # odd and even column counts (bf16 takes two columns per load when even),
    # row counts that leave 1..3 blocks in a thread's last group of four
    for rows, cols in [(32, 1), (64, 7), (96, 130), (160, 33), (256, 256), (4096, 16)]:
        x = torch.from_numpy(rand(rng, (rows, cols))).to(dtype)
        check_axis0(x, fmt, layout)


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
def test_axis0_tiled_shapes(fmt, dtype, layout):
    # rows of 16-byte multiples: f32 takes the shared-memory tile kernel, bf16
    # the register kernel (four columns per lane when the column count is a
    # multiple of 4, else two); ragged last column tiles (264, 520, 1000
    # columns), one block row, many units per CTA
    rng = np.random.default_rng(13)
    for rows, cols in [(32, 8), (64, 264), (96, 520), (1024, 1000), (2048, 4096)]:
        x = torch.from_numpy(rand(rng, (rows, cols))).to(dtype)
        check_axis0(x, fmt, layout)


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
def test_axis0_bf16_codes_off_32_bytes(fmt, layout):
    # bf16 input with codes on a 16- but not a 32-byte boundary takes the
    # shared-memory tile kernel instead of the register one
    rng = np.random.default_rng(17)
    for rows, cols in [(64, 264), (1024, 1000)]:
        x = torch.from_numpy(rand(rng, (rows, cols))).to(torch.bfloat16)
        check_axis0(x, fmt, layout, codes_offset=16)


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
def test_axis0_every_bf16_pattern_at_every_scale(fmt):
    # the exhaustive bf16 ladder of the last-axis tests, transposed: each
    # column is one block sequence, so axis-0 blocks are the ladder's blocks
    from test_quant_gpu import _bf16_ladder
    x = _bf16_ladder(0)
    nblk = x.shape[0]
    x = x[: (nblk // 8) * 8]  # whole tiles of 8 columns x 32 rows keep the transpose simple
    xt = x.reshape(-1, 8, 32).permute(0, 2, 1).reshape(-1, 32, 8)  # [groups, 32 rows, 8 cols]
    xt = xt.permute(1, 0, 2).reshape(32, -1).contiguous()           # 32 rows x (8 * groups) cols
    check_axis0(xt, fmt, mx.SCALES_ROWMAJOR)


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
def test_axis1_is_mx_quantize(fmt):
    rng = np.random.default_rng(4)
    x = torch.from_numpy(rand(rng, (64, 256))).cuda()
    c1, s1 = mx.alloc_codes(64, 256, fmt), mx.alloc_scales(64, 256)
    c2, s2 = mx.alloc_codes(64, 256, fmt), mx.alloc_scales(64, 256)
    mx.mx_quantize(x, fmt, c1, s1)
    mx.mx_quantize_axis(x, 1, fmt, c2, s2)
    mx.mx_device_status()
    assert torch.equal(c1, c2) and torch.equal(s1, s2)


def test_axis0_result_is_a_gemm_operand():
    # workload-1 shape: B is K x N; quantized along K (axis 0) it is the N x K
    # operand directly, with no transpose on the host
    rng = np.random.default_rng(6)
    M, N, K = 128, 128, 256
    A = rand(rng, (M, K), 4)
    B = rand(rng, (K, N), 4)
    C0 = np.zeros((M, N), np.float32)
    ac, as_ = mx.alloc_codes(M, K, mx.E2M1), mx.alloc_scales(M, K, mx.SCALES_MMA)
    bc, bs = mx.alloc_codes(N, K, mx.E2M1), mx.alloc_scales(N, K, mx.SCALES_MMA)
    mx.mx_quantize(torch.from_numpy(A).cuda(), mx.E2M1, ac, as_, mx.SCALES_MMA)
    mx.mx_quantize_axis(torch.from_numpy(B).cuda(), 0, mx.E2M1, bc, bs, mx.SCALES_MMA)
    C = torch.from_numpy(C0).cuda()
    mx.mx_block_matmul(ac, as_, mx.E2M1, bc, bs, mx.E2M1, M, N, K, C, mx.SCALES_MMA)
    mx.mx_device_status()
    oa, osa = oracle.quantize(A, oracle.E2M1)
    ob, osb = oracle.quantize_axis0(B, oracle.E2M1)
    ref, sabs = oracle.block_matmul(oa, osa, oracle.E2M1, ob, osb, oracle.E2M1, M, N, K, C0)
    err = np.abs(to_np(C).astype(np.float64) - ref)
    assert (err <= 1e-5 * sabs + np.abs(ref) * 2.0 ** -23).all()


# ------------------------------------------------------------ bf16 dequantize

@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
def test_dequantize_bf16_every_code_and_scale(fmt, layout):
    ncodes = 16 if fmt == mx.E2M1 else 256
    rows, cols = ncodes * 256, 64
    cu = np.repeat(np.arange(ncodes, dtype=np.uint8), 256)[:, None].repeat(cols, axis=1)
    cu[:, 1::2] = np.roll(cu[:, 1::2], 5, axis=0)
    s = np.tile(np.arange(256, dtype=np.uint8), ncodes)[:, None].repeat(2, axis=1)
    s[:, 1] = np.roll(s[:, 1], 3)
    codes = (cu[:, 0::2] | (cu[:, 1::2] << 4)).astype(np.uint8) if fmt == mx.E2M1 else cu
    s_dev = torch.from_numpy(rowmajor_to_mma(s, rows, 2) if layout == mx.SCALES_MMA else s.copy()).cuda()
    ybuf = torch.full((rows * cols + 64,), 7.0, dtype=torch.bfloat16, device="cuda")
    y = ybuf[:rows * cols]
    mx.mx_dequantize_bf16(torch.from_numpy(np.ascontiguousarray(codes)).cuda(), s_dev, rows, cols, fmt, y, layout)
    mx.mx_device_status()
    got = to_np(ybuf.view(torch.int16)).view(np.uint16)
    assert (got[rows * cols:] == 0x40E0).all(), "wrote past the end of y"  # 7.0 in bf16
    want = oracle.dequantize_bf16(codes, s, cols, O_FMT[fmt]).reshape(-1)
    got = got[:rows * cols]
    nan_w = (want & 0x7FFF) > 0x7F80
    assert ((got[nan_w] & 0x7FFF) > 0x7F80).all()
    assert np.array_equal(got[~nan_w], want[~nan_w])


def test_dequantize_bf16_roundtrip_workload2():
    import workloads
    w = workloads.make(2)
    x = w["x"]
    rows, cols = x.shape
    codes, scales = mx.alloc_codes(rows, cols, mx.E4M3FN), mx.alloc_scales(rows, cols)
    mx.mx_quantize(x.cuda(), mx.E4M3FN, codes, scales)
    y = torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")
    mx.mx_dequantize_bf16(codes, scales, rows, cols, mx.E4M3FN, y)
    mx.mx_device_status()
    want = oracle.dequantize_bf16(to_np(codes).reshape(rows, cols), to_np(scales).reshape(rows, -1), cols,
                                  oracle.E4M3)
    assert np.array_equal(to_np(y.view(torch.int16)).view(np.uint16), want)


# ----------------------------------------------------------------- fold_scale

@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
@pytest.mark.parametrize("scalar", [2.0 ** -40, 0.5, 1.0, 2.0, 2.0 ** 60, 2.0 ** 300, 2.0 ** -300])
def test_fold_scale_matches_oracle(layout, scalar):
    rng = np.random.default_rng(8)
    rows, cols = 130, 224
    nb = cols // 32
    s = rng.integers(0, 256, (rows, nb), dtype=np.uint8)
    s[rng.integers(0, rows, 10), rng.integers(0, nb, 10)] = 0xFF
    s_dev = torch.from_numpy(rowmajor_to_mma(s, rows, nb) if layout == mx.SCALES_MMA else s.copy()).cuda()
    mx.mx_fold_scale(s_dev, rows, cols, scalar, layout)
    mx.mx_device_status()
    got = to_np(s_dev)
    want = oracle.fold_scale(s, oracle.fold_exponent(scalar))
    if layout == mx.SCALES_MMA:
        assert (got[mma_padding_mask(rows, nb)] == 0).all(), "padding must stay 0"
        got = mma_to_rowmajor(got, rows, nb)
    assert np.array_equal(got.reshape(rows, nb), want)


def test_fold_scale_scales_the_values():
    # unsaturated bytes: the dequantized tensor is multiplied by the scalar exactly
    rng = np.random.default_rng(9)
    rows, cols = 64, 256
    x = torch.from_numpy(rng.standard_normal((rows, cols)).astype(np.float32)).cuda()
    codes, scales = mx.alloc_codes(rows, cols, mx.E4M3FN), mx.alloc_scales(rows, cols)
    mx.mx_quantize(x, mx.E4M3FN, codes, scales)
    y0 = torch.empty(rows, cols, device="cuda")
    mx.mx_dequantize(codes, scales, rows, cols, mx.E4M3FN, y0)
    mx.mx_fold_scale(scales, rows, cols, 2.0 ** -9)
    y1 = torch.empty(rows, cols, device="cuda")
    mx.mx_dequantize(codes, scales, rows, cols, mx.E4M3FN, y1)
    mx.mx_device_status()
    assert torch.equal(y1, y0 * 2.0 ** -9)


def test_fold_scale_rejects_non_powers_of_two():
    s = mx.alloc_scales(4, 64)
    for bad in (3.0, -2.0, 0.0):
        with pytest.raises(mx.MxError):
            mx.mx_fold_scale(s, 4, 64, bad)
