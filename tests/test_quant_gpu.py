"""GPU parity of mx_quantize / mx_dequantize / mx_scales_relayout against the
CPU oracle: codes, scales and dequantized values bit-exact, through the C ABI.

Workload inputs come from the seeded generators (``workloads``); expected
values come from the oracle only."""
import numpy as np
import pytest
import torch

import bit_gemm_gb300 as mx
import oracle
import workloads
from gpu_util import (mma_padding_mask, mma_to_rowmajor, same_f32_bits, to_np, unpack_e2m1)

pytestmark = pytest.mark.gpu

O_FMT = {mx.E2M1: oracle.E2M1, mx.E4M3FN: oracle.E4M3}
GUARD = 256  # canary bytes after every output


def gpu_quantize(x: torch.Tensor, fmt: int, layout: int):
    """Quantize on the GPU into canary-guarded buffers; returns numpy (codes, scales)."""
    rows, cols = x.shape
    cb, sb = mx.mx_codes_bytes(fmt, rows, cols), mx.mx_scales_bytes(layout, rows, cols)
    codes = torch.full((cb + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    scales = torch.full((sb + GUARD,), 0x5A, dtype=torch.uint8, device="cuda")
    mx.mx_quantize(x.cuda(), fmt, codes, scales, layout)
    mx.mx_device_status()
    c, s = to_np(codes), to_np(scales)
    assert (c[cb:] == 0xA5).all(), "quantize wrote past the end of codes"
    assert (s[sb:] == 0x5A).all(), "quantize wrote past the end of scales"
    return c[:cb], s[:sb]


def check_quantize(x_cpu: torch.Tensor, fmt: int, layout: int):
    rows, cols = x_cpu.shape
    nb = cols // 32
    codes, scales = gpu_quantize(x_cpu, fmt, layout)
    oc, os_ = oracle.quantize(x_cpu.float().numpy(), O_FMT[fmt])
    assert np.array_equal(codes.reshape(oc.shape), oc), "codes differ from the oracle"
    if layout == mx.SCALES_MMA:
        assert np.array_equal(mma_to_rowmajor(scales, rows, nb), os_), "scales differ from the oracle"
        assert (scales[mma_padding_mask(rows, nb)] == 0).all(), "layout padding must be written as 0"
    else:
        assert np.array_equal(scales.reshape(os_.shape), os_), "scales differ from the oracle"
    return codes, scales, oc, os_


# ----------------------------------------------------------------- workloads

@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
def test_workload1_f32_to_mxfp4(layout):
    w = workloads.make(1)
    for name in ("A", "Bt"):
        check_quantize(torch.from_numpy(w[name]), mx.E2M1, layout)


def test_workload2_bf16_to_mxfp8_full_size_and_nan_blocks():
    w = workloads.make(2)
    x = w["x"]
    rows, cols = x.shape
    codes, scales, oc, os_ = check_quantize(x, mx.E4M3FN, mx.SCALES_ROWMAJOR)
    # the injected structures are present
    flat_s = os_.reshape(-1)
    assert (flat_s[w["zero_blocks"]] == 127).all()
    assert (flat_s[w["tiny_blocks"]] == 0).all()          # clip at -127
    sub = oc.reshape(-1, 32)[w["subnormal_blocks"]]
    assert ((sub[:, 1:] & 0x78) == 0).any()                # E4M3 subnormal codes appear
    # NaN poisoning: 64 blocks get scale 0xFF before dequantize
    s_bad = scales.copy().reshape(-1)
    s_bad[w["nan_blocks"]] = 0xFF
    y = torch.empty(rows, cols, dtype=torch.float32, device="cuda")
    mx.mx_dequantize(torch.from_numpy(codes).cuda(), torch.from_numpy(s_bad).cuda(), rows, cols, mx.E4M3FN, y)
    mx.mx_device_status()
    yo = oracle.dequantize(oc, s_bad.reshape(os_.shape), cols, oracle.E4M3)
    yg = to_np(y)
    assert same_f32_bits(yg, yo).all()
    assert np.isnan(yg.reshape(-1, 32)[w["nan_blocks"]]).all()
    assert np.isnan(yg).reshape(-1, 32).all(axis=1).sum() == 64


def test_workload3_and_5_activation_quantize():
    w3 = workloads.make(3)
    check_quantize(w3["A"], mx.E4M3FN, mx.SCALES_MMA)
    w5 = workloads.make(5, scale=1 / 16)
    check_quantize(w5["A"], mx.E2M1, mx.SCALES_MMA)


# ---------------------------------------------------------------- edge cases

SHAPES = [(1, 32), (3, 96), (127, 160), (129, 224), (128, 4096), (300, 32 * 7)]


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
def test_shapes_dtypes_layouts(fmt, dtype, layout):
    rng = np.random.default_rng(100)
    for rows, cols in SHAPES:
        x = rng.standard_normal((rows, cols)).astype(np.float32) * np.float32(2.0) ** rng.integers(
            -30, 30, (rows, 1)).astype(np.float32)
        check_quantize(torch.from_numpy(x).to(dtype), fmt, layout)


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_special_values(fmt, dtype):
    rows, cols = 10, 64
    x = np.zeros((rows, cols), np.float32)
    x[1, :32] = -0.0
    x[1, 40] = -0.0
    x[2, 3] = np.nan
    x[3, 40] = np.inf
    x[4, :] = -np.inf
    x[5, :] = np.float32(2.0 ** -149) * np.arange(cols, dtype=np.float32)   # f32 subnormals
    x[6, :] = np.float32(3.0e38) * np.linspace(-1, 1, cols, dtype=np.float32)
    x[7, :] = -np.float32(1e-3)
    x[8, :] = np.float32(2.0 ** -133) * np.arange(-32, 32, dtype=np.float32)  # bf16 subnormals
    x[9, 1::2] = -0.0
    x[9, 0::2] = -np.float32(2.0 ** -140)  # rounds to zero, keeps its sign
    x[9, 32] = 1.0
    xt = torch.from_numpy(x).to(dtype)
    codes, scales, oc, os_ = check_quantize(xt, fmt, mx.SCALES_ROWMAJOR)
    assert os_[2, 0] == 0xFF and os_[3, 1] == 0xFF and os_[4, 0] == 0xFF and os_[0, 0] == 127


def _bf16_ladder(anchor_mantissa: int) -> torch.Tensor:
    """Blocks [anchor, v1..v31]: for the anchor 2^E (times 1 + m/128) of every
    bf16 binade E, subnormal ones included, the v run through every bf16 bit
    pattern of magnitude <= the anchor's, both signs (the last block of each
    anchor is padded with +0)."""
    out = []
    for E in range(-133, 128):
        a = ((E + 127) << 7 | anchor_mantissa) if E >= -126 else (1 << (E + 133))
        pats = np.arange(0, a + 1, dtype=np.uint16)
        pats = np.concatenate([pats, pats | 0x8000])
        nblk = -(-len(pats) // 31)
        flat = np.zeros(nblk * 31, np.uint16)
        flat[:len(pats)] = pats
        blk = np.empty((nblk, 32), np.uint16)
        blk[:, 0] = a
        blk[:, 1:] = flat.reshape(nblk, 31)
        out.append(blk)
    return torch.from_numpy(np.concatenate(out).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("anchor_mantissa", [0, 0x7F])
def test_exhaustive_bf16_elements_at_every_scale(fmt, anchor_mantissa):
    """Every bf16 element pattern below the block maximum, at every scale a
    bf16 block can take (the maximum 2^E or (2 - 2^-7) 2^E for every E,
    subnormal maxima included, which also drives the scale into its -127
    clip): codes and scales equal the oracle's, byte for byte."""
    x = _bf16_ladder(anchor_mantissa)
    check_quantize(x, fmt, mx.SCALES_ROWMAJOR)


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
def test_bf16_only_16_byte_aligned(fmt, layout):
    """Input and codes that are 16- but not 32-byte aligned take the
    four-threads-per-block path; results are the same."""
    rng = np.random.default_rng(7)
    rows, cols = 130, 256
    x = torch.from_numpy(rng.standard_normal((rows, cols)).astype(np.float32)).to(torch.bfloat16)
    big = torch.zeros(rows * cols + 8, dtype=torch.bfloat16, device="cuda")
    xs = big[8:].view(rows, cols)
    xs.copy_(x.cuda())
    cb, sb = mx.mx_codes_bytes(fmt, rows, cols), mx.mx_scales_bytes(layout, rows, cols)
    cbuf = torch.full((cb + 16 + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    codes = cbuf[16:16 + cb]
    scales = torch.full((sb,), 0x5A, dtype=torch.uint8, device="cuda")
    assert xs.data_ptr() % 32 == 16 and codes.data_ptr() % 32 == 16
    mx.mx_quantize(xs, fmt, codes, scales, layout)
    mx.mx_device_status()
    oc, os_ = oracle.quantize(x.float().numpy(), O_FMT[fmt])
    c, s = to_np(cbuf), to_np(scales)
    assert (c[:16] == 0xA5).all() and (c[16 + cb:] == 0xA5).all()
    assert np.array_equal(c[16:16 + cb].reshape(oc.shape), oc)
    got_s = mma_to_rowmajor(s, rows, cols // 32) if layout == mx.SCALES_MMA else s.reshape(os_.shape)
    assert np.array_equal(got_s, os_)


def test_empty_is_noop():
    x = torch.zeros(0, 64, device="cuda")
    mx.mx_quantize(x, mx.E2M1, torch.zeros(1, dtype=torch.uint8, device="cuda"),
                   torch.zeros(1, dtype=torch.uint8, device="cuda"))
    mx.mx_device_status()


# ----------------------------------------------------- exhaustive rounding

def _transitions(v: torch.Tensor) -> np.ndarray:
    return to_np(torch.nonzero(v[1:] != v[:-1]).flatten() + 1)


@pytest.mark.parametrize("fmt,anchor,top_bits", [(mx.E2M1, 4.0, 0x41000000), (mx.E4M3FN, 256.0, 0x44000000)])
def test_exhaustive_element_rounding(fmt, anchor, top_bits):
    """Every binary32 y in [0, 8) (E2M1) or [0, 512) (E4M3FN), placed in blocks
    whose maximum pins the scale exponent e = 0, goes through the GPU kernel.
    The GPU code sequence is reduced to its change points; the oracle is then
    evaluated at every change point and the element just before it.  The oracle
    (nearest point of a sorted grid, lower index on ties) is a non-decreasing
    function of y, so agreeing at both ends of every constant run means
    agreeing at every y."""
    n = top_bits
    per = 31
    nblk = (n + per - 1) // per
    x = torch.full((nblk, 32), anchor, dtype=torch.float32, device="cuda")
    bits = torch.arange(nblk * per, dtype=torch.int64, device="cuda").clamp_(max=n - 1).to(torch.int32)
    x[:, 1:] = bits.view(nblk, per).view(torch.float32)
    codes = mx.alloc_codes(nblk, 32, fmt)
    scales = mx.alloc_scales(nblk, 32)
    mx.mx_quantize(x, fmt, codes, scales)
    mx.mx_device_status()
    del x
    assert bool((scales == 127).all())
    if fmt == mx.E2M1:
        c = codes.view(nblk, 16)
        full = torch.stack([c & 0xF, c >> 4], dim=2).view(nblk, 32)
    else:
        full = codes.view(nblk, 32)
    seq = full[:, 1:].reshape(-1)[:n]
    t = _transitions(seq)
    assert 0 < len(t) < 200
    pts = sorted(set([0, n - 1] + list(t) + list(t - 1)))
    ys = np.array(pts, np.uint32).view(np.float32)
    blocks = np.full((len(ys), 32), anchor, np.float32)
    blocks[:, 1] = ys
    oc, os_ = oracle.quantize(blocks, O_FMT[fmt])
    ocodes = unpack_e2m1(oc)[:, 1] if fmt == mx.E2M1 else oc[:, 1]
    gcodes = to_np(seq[torch.tensor(pts, device="cuda")])
    assert (os_ == 127).all()
    assert np.array_equal(gcodes, ocodes), [(hex(p), int(g), int(o)) for p, g, o in zip(pts, gcodes, ocodes) if g != o][:10]


@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
def test_exhaustive_scale_selection(fmt):
    """Every positive finite binary32 v as the only nonzero element (element 0)
    of a block: the GPU's (scale byte, code of v) pairs, in increasing v, are
    reduced to change points and checked against the oracle there.  The
    oracle's scale is non-decreasing in v and, for a fixed scale, so is the code
    of v, so agreement at both ends of every run is agreement everywhere."""
    total = 0x7F800000
    chunk = 1 << 26
    prev_pair = None
    checked = []
    for start in range(1, total, chunk):
        cnt = min(chunk, total - start)
        x = torch.zeros(cnt, 32, dtype=torch.float32, device="cuda")
        x[:, 0] = torch.arange(start, start + cnt, dtype=torch.int64, device="cuda").to(torch.int32).view(torch.float32)
        codes = mx.alloc_codes(cnt, 32, fmt)
        scales = mx.alloc_scales(cnt, 32)
        mx.mx_quantize(x, fmt, codes, scales)
        mx.mx_device_status()
        del x
        c0 = (codes.view(cnt, 16)[:, 0] & 0xF) if fmt == mx.E2M1 else codes.view(cnt, 32)[:, 0]
        pair = scales.to(torch.int32) * 256 + c0.to(torch.int32)
        t = _transitions(pair)
        idx = sorted(set([0, cnt - 1] + list(t) + list(t - 1)))
        vals = to_np(pair[torch.tensor(idx, device="cuda")])
        checked += [(start + i, int(v)) for i, v in zip(idx, vals)]
        if prev_pair is not None and prev_pair != int(vals[0]):
            checked.append((start - 1, prev_pair))
        prev_pair = int(to_np(pair[-1:])[0])
    bits = np.array([b for b, _ in checked], np.uint32)
    blocks = np.zeros((len(bits), 32), np.float32)
    blocks[:, 0] = bits.view(np.float32)
    oc, os_ = oracle.quantize(blocks, O_FMT[fmt])
    oc0 = (oc[:, 0] & 0xF) if fmt == mx.E2M1 else oc[:, 0]
    expect = os_[:, 0].astype(np.int64) * 256 + oc0
    got = np.array([v for _, v in checked], np.int64)
    assert np.array_equal(got, expect)


# ---------------------------------------------------------------- dequantize

@pytest.mark.parametrize("fmt", [mx.E2M1, mx.E4M3FN])
@pytest.mark.parametrize("layout", [mx.SCALES_ROWMAJOR, mx.SCALES_MMA])
@pytest.mark.parametrize("y_off", [0, 4])  # y 32-byte aligned, or only 16-byte aligned
def test_dequantize_every_code_and_scale(fmt, layout, y_off):
    ncodes = 16 if fmt == mx.E2M1 else 256
    rows, cols = ncodes * 256, 32
    cu = np.repeat(np.arange(ncodes, dtype=np.uint8), 256)[:, None].repeat(32, axis=1)
    cu[:, 1::2] = np.roll(cu[:, 1::2], 7, axis=0)  # vary the odd elements too
    s = np.tile(np.arange(256, dtype=np.uint8), ncodes)[:, None]
    codes = (cu[:, 0::2] | (cu[:, 1::2] << 4)).astype(np.uint8) if fmt == mx.E2M1 else cu
    if layout == mx.SCALES_MMA:
        from gpu_util import rowmajor_to_mma
        s_dev = torch.from_numpy(rowmajor_to_mma(s, rows, 1)).cuda()
    else:
        s_dev = torch.from_numpy(s.copy()).cuda()
    ybuf = torch.full((rows * cols + 64,), 7.0, dtype=torch.float32, device="cuda")
    y = ybuf[y_off:y_off + rows * cols]
    mx.mx_dequantize(torch.from_numpy(np.ascontiguousarray(codes)).cuda(), s_dev, rows, cols, fmt, y, layout)
    mx.mx_device_status()
    yg = to_np(ybuf)
    assert (yg[:y_off] == 7.0).all() and (yg[y_off + rows * cols:] == 7.0).all(), "dequantize wrote outside y"
    yo = oracle.dequantize(codes, s, cols, O_FMT[fmt])
    assert same_f32_bits(yg[y_off:y_off + rows * cols].reshape(rows, cols), yo).all()


def test_dequantize_roundtrip_workload1():
    w = workloads.make(1)
    A = torch.from_numpy(w["A"]).cuda()
    codes, scales = mx.alloc_codes(128, 256, mx.E2M1), mx.alloc_scales(128, 256)
    mx.mx_quantize(A, mx.E2M1, codes, scales)
    y = torch.empty(128, 256, device="cuda")
    mx.mx_dequantize(codes, scales, 128, 256, mx.E2M1, y)
    mx.mx_device_status()
    oc, os_ = oracle.quantize(w["A"], oracle.E2M1)
    assert same_f32_bits(to_np(y), oracle.dequantize(oc, os_, 256, oracle.E2M1)).all()


# ------------------------------------------------------------------ relayout

@pytest.mark.parametrize("rows,cols", [(1, 32), (130, 160), (256, 4096), (16, 4096)])
def test_relayout_both_ways(rows, cols):
    nb = cols // 32
    rng = np.random.default_rng(rows + cols)
    s = rng.integers(0, 256, (rows, nb)).astype(np.uint8)
    src = torch.from_numpy(s).cuda()
    mma = torch.full((mx.mx_scales_bytes(mx.SCALES_MMA, rows, cols),), 0xEE, dtype=torch.uint8, device="cuda")
    mx.mx_scales_relayout(src, mx.SCALES_ROWMAJOR, rows, cols, mma, mx.SCALES_MMA)
    back = torch.empty(rows * nb, dtype=torch.uint8, device="cuda")
    mx.mx_scales_relayout(mma, mx.SCALES_MMA, rows, cols, back, mx.SCALES_ROWMAJOR)
    mx.mx_device_status()
    m = to_np(mma)
    assert np.array_equal(mma_to_rowmajor(m, rows, nb), s)
    assert (m[mma_padding_mask(rows, nb)] == 0).all()
    assert np.array_equal(to_np(back).reshape(rows, nb), s)
