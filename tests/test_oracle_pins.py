"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- a value the pages print (tests/golden/), a library decode
routine, exact rational arithmetic, or a closed form -- chosen so that a
plausible slip (a wrong bias or emax, a tie broken the other way, a swapped
nibble, a dropped sign, a transposed operand) fails at least one of them.

Sources: "A Dialect Is a Set of Co-Designed Decisions: Designing for MX
Quantization in MLIR" ("The four ops", "The block axis") and "Bit Layout"
("The E2M1 element", "The E8M0 shared scale", "Block structure and packing",
"Reference encode and decode").
"""
import math
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from golden_facts import e2m1_magnitudes, facts

E2M1, E4M3 = oracle.E2M1, oracle.E4M3
F = facts()


# ---------------------------------------------------------------- helpers ---

def f32_bits(v):
    return struct.unpack("<I", struct.pack("<f", v))[0]


def bits_f32(b):
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def e4m3_grid_torch():
    """Nonnegative finite E4M3FN magnitudes for codes 0..126, decoded by torch."""
    codes = torch.arange(0, 127, dtype=torch.uint8)
    return [float(v) for v in codes.view(torch.float8_e4m3fn).float().tolist()]


def grid(fmt):
    return e2m1_magnitudes() if fmt == E2M1 else e4m3_grid_torch()


def emax(fmt):
    # E2M1: printed on the page; E4M3: the binade of its largest finite value
    # (448 = 1.75 * 2^8), taken from the torch decode.
    if fmt == E2M1:
        return F["e2m1_emax"]
    return math.floor(math.log2(max(e4m3_grid_torch())))


def exact_floor_log2(q: Fraction) -> int:
    """floor(log2 q) for rational q > 0, by exact comparison with powers of 2."""
    e = q.numerator.bit_length() - q.denominator.bit_length()
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    return e


def brute_quantize_block(xs, fmt):
    """The pages' definition evaluated in exact rationals: argmin over the grid,
    first (lower) index on ties.  xs: 32 binary32-representable floats."""
    g = [Fraction(v) for v in grid(fmt)]
    sign = 0x8 if fmt == E2M1 else 0x80
    fx = [Fraction(v) for v in xs]
    amax = max(abs(v) for v in fx)
    if amax == 0:
        return [0] * 32, F["zero_block_scale"]
    e = exact_floor_log2(amax) - emax(fmt)
    e = max(F["scale_clip_low"], min(F["scale_clip_high"], e))
    codes = []
    for v in fx:
        y = abs(v) / Fraction(2) ** e
        idx = min(range(len(g)), key=lambda j: (abs(y - g[j]), j))
        codes.append(idx | (sign if v < 0 else 0))
    return codes, e + F["e8m0_bias"]


def unpack(codes_row, fmt, cols):
    if fmt == E4M3:
        return list(codes_row[:cols])
    out = []
    for b in codes_row[: cols // 2]:
        out.append(int(b) & 0xF)
        out.append(int(b) >> 4)
    return out


def check_blocks_against_brute(x, fmt):
    x = np.asarray(x, np.float32).reshape(-1, 32)
    codes, scales = oracle.quantize(x, fmt)
    for r in range(x.shape[0]):
        exp_codes, exp_scale = brute_quantize_block([float(v) for v in x[r]], fmt)
        got = unpack(codes[r], fmt, 32)
        assert int(scales[r, 0]) == exp_scale, (r, x[r], scales[r, 0], exp_scale)
        assert got == exp_codes, (r, x[r], got, exp_codes)


# ------------------------------------------------------ element formats -----

def test_e2m1_decode_matches_page_table():
    table = e2m1_magnitudes()
    assert len(table) == 8
    for code in range(16):
        expect = table[code & 7] * (-1.0 if code & 8 else 1.0)
        got = oracle.decode_element(E2M1, code)
        assert got == expect and math.copysign(1, got) == math.copysign(1, expect), code


def test_e2m1_decode_matches_bit_formula():
    # "The E2M1 element": normal (-1)^S 2^(E-1) (1 + M/2); subnormal (E=0) (-1)^S 0.5 M.
    bias = F["e2m1_exponent_bias"]
    for code in range(16):
        S, E, M = code >> 3, (code >> 1) & 3, code & 1
        mag = 2.0 ** (E - bias) * (1 + M / 2) if E > 0 else 0.5 * M
        assert oracle.decode_element(E2M1, code) == (-mag if S else mag)


def test_e4m3_decode_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float()
    for code in range(256):
        got, exp = oracle.decode_element(E4M3, code), float(ref[code])
        if math.isnan(exp):
            assert math.isnan(got), code
        else:
            assert got == exp and math.copysign(1, got) == math.copysign(1, exp), code


def test_e8m0_decode_matches_torch_and_page():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).float()
    for b in range(256):
        got = oracle.decode_scale(b)
        if b == F["e8m0_nan_byte"]:
            assert math.isnan(got) and math.isnan(float(ref[b]))
        else:
            assert got == 2.0 ** (b - F["e8m0_bias"]) == float(ref[b]), b


def test_floor_log2_matches_bit_extraction():
    rng = np.random.default_rng(1)
    vals = [bits_f32(b) for b in rng.integers(1, 0x7F800000, 20000)]
    vals += [bits_f32(1 << i) for i in range(23)]                  # subnormal leading bits
    vals += [bits_f32((1 << i) | ((1 << i) - 1)) for i in range(23)]
    vals += [2.0 ** k for k in range(-126, 128)] + [np.nextafter(np.float32(2.0 ** k), np.float32(0)) for k in range(-125, 128)]
    for v in vals:
        b = f32_bits(float(v))
        fe, mant = (b >> 23) & 0xFF, b & 0x7FFFFF
        expect = fe - 127 if fe else mant.bit_length() - 1 - 149
        assert oracle.floor_log2(float(v)) == expect, (v, hex(b))


def test_floor_log2_is_exact_not_rounded_log2():
    # A float32 log2 rounds up just below a power of two; the exact reading does not.
    v = float(np.float32(2047.9999))
    assert float(np.floor(np.log2(np.float32(v)))) == 11.0
    assert oracle.floor_log2(v) == 10


# ------------------------------------------------------------- quantize -----

def test_zero_block_gives_zero_codes_and_scale_127():
    for fmt in (E2M1, E4M3):
        for x in (np.zeros((1, 32), np.float32), -np.zeros((1, 32), np.float32)):
            codes, scales = oracle.quantize(x, fmt)
            assert scales.tolist() == [[F["zero_block_scale"]]]
            assert (codes == F["zero_block_code"]).all()


def test_nonfinite_block_is_poisoned():
    for fmt in (E2M1, E4M3):
        for bad in (np.nan, np.inf, -np.inf):
            x = np.ones((2, 32), np.float32)
            x[0, 5] = bad
            codes, scales = oracle.quantize(x, fmt)
            assert scales[0, 0] == 0xFF and (codes[0] == 0).all()
            assert scales[1, 0] != 0xFF


def test_low_nibble_holds_element_zero():
    # element 0 -> code 1 (0.5), element 1 -> code 7 (6.0); amax 6 gives e = 0.
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 0.5, 6.0
    codes, scales = oracle.quantize(x, E2M1)
    assert scales[0, 0] == 127
    assert codes[0, 0] == (7 << 4) | 1
    assert F["low_nibble_element"] == 0


def test_tie_rule_lower_magnitude():
    # Midpoints of the E2M1 grid (e = 0 via the anchor 4.0): each goes to the lower point.
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 4.0
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    x[0, 1:8] = mids
    codes, _ = oracle.quantize(x, E2M1)
    got = unpack(codes[0], E2M1, 32)[1:8]
    assert got == [0, 1, 2, 3, 4, 5, 6]
    # Round-to-nearest-even would send 0.75 -> 1.0, 1.75 -> 2.0, 3.5 -> 4.0.
    # E4M3, e = 0 via the anchor 256: 1.1875 lies halfway between 1.125 and 1.25.
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 256.0, 1.1875
    codes, _ = oracle.quantize(x, E4M3)
    assert oracle.decode_element(E4M3, int(codes[0, 1])) == 1.125
    assert torch.tensor([1.1875]).to(torch.float8_e4m3fn).float().item() == 1.25


def _midpoint_inputs(fmt):
    g = grid(fmt)
    anchor = 4.0 if fmt == E2M1 else 256.0
    top = 2.0 ** (emax(fmt) + 1)
    pts = []
    for a, b in zip(g[:-1], g[1:]):
        m = np.float32((a + b) / 2)
        pts += [np.nextafter(m, np.float32(0)), m, np.nextafter(m, np.float32(np.inf))]
    pts += [g[-1], np.nextafter(np.float32(g[-1]), np.float32(np.inf)),
            (g[-1] + top) / 2, np.nextafter(np.float32(top), np.float32(0))]
    vals = np.array(pts, np.float32)
    vals = np.concatenate([vals, -vals])
    n = (len(vals) + 30) // 31
    x = np.zeros((n, 32), np.float32)
    x[:, 0] = anchor
    flat = x[:, 1:].reshape(-1)
    flat[: len(vals)] = vals
    x[:, 1:] = flat.reshape(n, 31)
    return x


@pytest.mark.parametrize("fmt", [E2M1, E4M3])
def test_rounding_at_every_midpoint_against_exact_argmin(fmt):
    check_blocks_against_brute(_midpoint_inputs(fmt), fmt)


@pytest.mark.parametrize("fmt", [E2M1, E4M3])
def test_random_blocks_against_exact_argmin(fmt):
    rng = np.random.default_rng(7)
    blocks = []
    for k in list(range(-150, 128, 9)) + [0, 1, -1]:
        v = rng.standard_normal(32) * 2.0 ** k
        blocks.append(np.clip(v, -3e38, 3e38))
    t = rng.standard_t(3, size=(16, 32))
    blocks += list(t)
    sub = rng.integers(1, 1 << 23, size=(4, 32)).astype(np.uint32).view(np.float32)  # subnormals
    blocks += list(sub * rng.choice([-1, 1], size=(4, 32)))
    x = np.array(blocks, np.float32)
    check_blocks_against_brute(x, fmt)


def test_tiny_shapes_against_exact_argmin():
    rng = np.random.default_rng(11)
    for fmt in (E2M1, E4M3):
        for shape in ((1, 32), (2, 64), (3, 96)):
            x = (rng.standard_normal(shape) * 3).astype(np.float32)
            codes, scales = oracle.quantize(x, fmt)
            for r in range(shape[0]):
                row = unpack(codes[r], fmt, shape[1])
                for b in range(shape[1] // 32):
                    ec, es = brute_quantize_block([float(v) for v in x[r, 32 * b: 32 * b + 32]], fmt)
                    assert row[32 * b: 32 * b + 32] == ec
                    assert scales[r, b] == es


def test_scale_clip_low_and_subnormal_codes():
    # amax 2^-130 -> e = -132 (E2M1) is clipped to -127: scale byte 0.
    x = np.full((1, 32), 2.0 ** -130, np.float32)
    _, s = oracle.quantize(x, E2M1)
    assert s[0, 0] == 0
    # E4M3 block with one element at 1.0 and the rest far below: e = -8, so
    # 2^-16 becomes y = 2^-8 = 2 * 2^-9, an E4M3 subnormal (code 2).
    x = np.full((1, 32), 2.0 ** -16, np.float32)
    x[0, 0] = 1.0
    c, s = oracle.quantize(x, E4M3)
    assert s[0, 0] == 127 - 8 and c[0, 1] == 2 and c[0, 0] == 0x78   # 1.0 * 2^8 = 256: exponent field 15
    assert oracle.decode_element(E4M3, int(c[0, 0])) * 2.0 ** -8 == 1.0


def test_saturation_band_maps_to_largest_code():
    for fmt, anchor, top in ((E2M1, 4.0, 8.0), (E4M3, 256.0, 512.0)):
        gmax = max(grid(fmt))
        x = np.zeros((1, 32), np.float32)
        x[0, 0] = anchor
        x[0, 1:4] = [np.nextafter(np.float32(gmax), np.float32(top)), (gmax + top) / 2,
                     np.nextafter(np.float32(top), np.float32(0))]
        c, _ = oracle.quantize(x, fmt)
        for code in unpack(c[0], fmt, 32)[1:4]:
            assert oracle.decode_element(fmt, code) == gmax


def test_negative_values_and_signed_zero():
    x = np.zeros((1, 32), np.float32)
    x[0, :4] = [-6.0, -0.1, -0.0, 0.1]
    c, s = oracle.quantize(x, E2M1)
    row = unpack(c[0], E2M1, 32)
    assert s[0, 0] == 127
    assert row[:4] == [0xF, 0x8, 0x0, 0x0]  # -0.1 rounds to zero but keeps its sign bit


# ----------------------------------------------------------- dequantize -----

@pytest.mark.parametrize("fmt", [E2M1, E4M3])
def test_dequantize_every_code_every_scale(fmt):
    ncodes = 16 if fmt == E2M1 else 256
    if fmt == E2M1:
        dec = [e2m1_magnitudes()[c & 7] * (-1.0 if c & 8 else 1.0) for c in range(16)]
    else:
        dec = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().tolist()
    rows = ncodes * 256
    cols = 32
    scales = np.zeros((rows, 1), np.uint8)
    codes_u = np.zeros((rows, cols), np.uint8)
    for c in range(ncodes):
        for s in range(256):
            r = c * 256 + s
            codes_u[r, :] = c
            scales[r, 0] = s
    if fmt == E2M1:
        codes = (codes_u[:, 0::2] | (codes_u[:, 1::2] << 4)).astype(np.uint8)
    else:
        codes = codes_u
    y = oracle.dequantize(codes, scales, cols, fmt)
    for c in range(ncodes):
        for s in range(256):
            r = c * 256 + s
            v = y[r]
            if s == F["e8m0_nan_byte"] or math.isnan(dec[c]):
                assert np.isnan(v).all(), (c, s)
                continue
            with np.errstate(over="ignore"):
                exp = np.float32(dec[c] * 2.0 ** (s - F["e8m0_bias"]))  # overflow -> inf
            assert (v.view(np.uint32) == np.full(32, exp, np.float32).view(np.uint32)).all(), (c, s, v[0], exp)


def test_nan_scale_poisons_whole_block():
    x = np.random.default_rng(3).standard_normal((2, 64)).astype(np.float32)
    for fmt in (E2M1, E4M3):
        c, s = oracle.quantize(x, fmt)
        s[1, 0] = 0xFF
        y = oracle.dequantize(c, s, 64, fmt)
        assert np.isnan(y[1, :32]).all()
        assert not np.isnan(y[1, 32:]).any() and not np.isnan(y[0]).any()


# --------------------------------------------------------- storage math -----

def test_storage_arithmetic():
    rows, cols = 8, 256
    x = np.random.default_rng(0).standard_normal((rows, cols)).astype(np.float32)
    c, s = oracle.quantize(x, E2M1)
    blocks = rows * cols // F["block_size"]
    bits = (c.nbytes + s.nbytes) * 8
    assert bits / blocks == F["bits_per_block"]
    assert bits / (rows * cols) == F["bits_per_element"]
    assert round(16 / (bits / (rows * cols)), 2) == F["reduction_vs_bf16"]


# ------------------------------------------------------- round-trip laws -----

@pytest.mark.parametrize("fmt", [E2M1, E4M3])
def test_roundtrip_grid_points_are_fixed(fmt):
    rng = np.random.default_rng(5)
    g = np.array(grid(fmt), np.float64)
    rows = []
    for _ in range(64):
        k = int(rng.integers(-100, 100))
        row = rng.choice(g, 32) * rng.choice([-1, 1], 32)
        row[0] = g[-1]  # pins e = k: amax = gmax * 2^k
        rows.append(row * 2.0 ** k)
    x = np.array(rows, np.float32)
    c, s = oracle.quantize(x, fmt)
    y = oracle.dequantize(c, s, 32, fmt)
    assert (y == x).all()


@pytest.mark.parametrize("fmt", [E2M1, E4M3])
def test_roundtrip_error_bound_and_idempotence(fmt):
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((256, 64)) * 2.0 ** rng.integers(-20, 20, (256, 1))).astype(np.float32)
    c, s = oracle.quantize(x, fmt)
    y = oracle.dequantize(c, s, 64, fmt)
    g = np.array(grid(fmt))
    gaps = np.diff(g)
    for r in range(x.shape[0]):
        for b in range(2):
            e = int(s[r, b]) - 127
            xs, ys = x[r, 32 * b:32 * b + 32].astype(np.float64), y[r, 32 * b:32 * b + 32].astype(np.float64)
            yv = np.abs(xs) / 2.0 ** e
            inside = yv <= g[-1]
            idx = np.clip(np.searchsorted(g, yv) - 1, 0, len(gaps) - 1)
            bound = gaps[idx] / 2 * 2.0 ** e
            assert (np.abs(ys - xs)[inside] <= bound[inside]).all()
    # Re-quantizing the dequantized tensor reproduces it (values; a negative
    # value that rounded to -0.0 re-quantizes to +0 because the sign rule is x < 0).
    c2, s2 = oracle.quantize(y, fmt)
    assert (s2 == s).all()
    assert (oracle.dequantize(c2, s2, 64, fmt) == y).all()


# ------------------------------------------------------------ block_matmul ---

def _decode_rows(codes, scales, fmt, K):
    """Decode with the page's table / torch's decode (independent of the oracle)."""
    tab = e2m1_magnitudes()
    e4 = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    out = np.zeros((codes.shape[0], K))
    for r in range(codes.shape[0]):
        u = unpack(codes[r], fmt, K)
        for k in range(K):
            v = (tab[u[k] & 7] * (-1 if u[k] & 8 else 1)) if fmt == E2M1 else e4[u[k]]
            out[r, k] = v * 2.0 ** (int(scales[r, k // 32]) - 127)
    return out


def _random_codes(rng, rows, K, fmt):
    if fmt == E2M1:
        return rng.integers(0, 256, (rows, K // 2)).astype(np.uint8)
    c = rng.integers(0, 256, (rows, K)).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x11  # keep NaN codes out of this test
    return c


def test_gemm_integer_case_is_exact():
    rng = np.random.default_rng(8)
    M, N, K = 5, 7, 96
    a = _random_codes(rng, M, K, E2M1)
    b = _random_codes(rng, N, K, E2M1)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    c0 = rng.integers(-8, 8, (M, N)).astype(np.float32)
    ref, sabs = oracle.block_matmul(a, sa, E2M1, b, sb, E2M1, M, N, K, c0)
    A, B = _decode_rows(a, sa, E2M1, K), _decode_rows(b, sb, E2M1, K)
    assert (ref == c0 + A @ B.T).all()
    assert (sabs == np.abs(A) @ np.abs(B).T).all()


@pytest.mark.parametrize("fa,fb", [(E2M1, E2M1), (E4M3, E4M3), (E4M3, E2M1), (E2M1, E4M3)])
def test_gemm_factored_block_sums(fa, fb):
    """The block-axis identity: per block, 2^(sa+sb) factors out of the sum of
    mantissa products.  Evaluated exactly with integer mantissas."""
    rng = np.random.default_rng(9)
    M, N, K = 4, 3, 128
    a, b = _random_codes(rng, M, K, fa), _random_codes(rng, N, K, fb)
    sa = rng.integers(100, 150, (M, K // 32)).astype(np.uint8)
    sb = rng.integers(100, 150, (N, K // 32)).astype(np.uint8)
    c0 = rng.standard_normal((M, N)).astype(np.float32)
    ref, sabs = oracle.block_matmul(a, sa, fa, b, sb, fb, M, N, K, c0)
    tab = e2m1_magnitudes()
    e4 = e4m3_grid_torch()

    def int_mant(fmt, code):  # (integer mantissa, power-of-two denominator exponent)
        if fmt == E2M1:
            return int(tab[code & 7] * 2) * (-1 if code & 8 else 1), 1
        return int(e4[code & 0x7F] * 512) * (-1 if code & 0x80 else 1), 9

    for m in range(M):
        ua = unpack(a[m], fa, K)
        for n in range(N):
            ub = unpack(b[n], fb, K)
            total = Fraction(float(c0[m, n]))
            tabs = Fraction(0)
            for blk in range(K // 32):
                s_int, s_abs = 0, 0
                for k in range(32 * blk, 32 * blk + 32):
                    ma, da = int_mant(fa, ua[k])
                    mb, db = int_mant(fb, ub[k])
                    s_int += ma * mb
                    s_abs += abs(ma * mb)
                scale = Fraction(2) ** (int(sa[m, blk]) + int(sb[n, blk]) - 254 - da - db)
                total += scale * s_int
                tabs += scale * s_abs
            assert abs(Fraction(sabs[m, n]) - tabs) <= Fraction(K) * Fraction(2) ** -52 * tabs
            assert abs(Fraction(ref[m, n]) - total) <= Fraction(K + 2) * Fraction(2) ** -52 * (tabs + abs(Fraction(float(c0[m, n])))), (m, n)


def test_gemm_single_block_closed_form():
    # K = 32: C = c0 + 2^(sa+sb-254) * <a_dec, b_dec>; with a = all 1.0 and b = codes
    # 0..15 repeated, <a,b> is the sum of the page's signed table over two periods.
    a = np.full((1, 16), 0x22, np.uint8)              # every nibble = 2 -> 1.0
    b = np.array([[(2 * i + 1) << 4 | (2 * i) for i in range(8)] * 2], np.uint8)
    sa, sb = np.array([[130]], np.uint8), np.array([[120]], np.uint8)
    ref, _ = oracle.block_matmul(a, sa, E2M1, b, sb, E2M1, 1, 1, 32, np.array([[0.25]], np.float32))
    tab = e2m1_magnitudes()
    dot = 2 * (sum(tab) - sum(tab))  # codes 0..7 positive, 8..15 their negatives
    assert ref[0, 0] == 0.25 + 2.0 ** (130 + 120 - 254) * dot == 0.25
    b2 = np.array([[(2 * i + 1) << 4 | (2 * i) for i in range(4)] * 4], np.uint8)  # codes 0..7 only
    ref2, _ = oracle.block_matmul(a, sa, E2M1, b2, sb, E2M1, 1, 1, 32, np.array([[0.25]], np.float32))
    assert ref2[0, 0] == 0.25 + 2.0 ** -4 * 4 * sum(tab)


def test_gemm_operand_orientation():
    # A row m and Bt row n must pair up: a rank-one check with distinct rows.
    M, N, K = 3, 2, 32
    a = np.zeros((M, K // 2), np.uint8)
    b = np.zeros((N, K // 2), np.uint8)
    a[:, 0] = [0x02, 0x04, 0x07]       # element 0 of each A row: 1.0, 2.0, 6.0
    b[:, 0] = [0x20, 0x30]             # element 1 of each Bt row: 1.0, 1.5 (element 0 is 0)
    b[:, 0] |= 0x02                    # element 0 of each Bt row: 1.0
    s1 = np.full((M, 1), 127, np.uint8)
    s2 = np.array([[127], [128]], np.uint8)
    ref, _ = oracle.block_matmul(a, s1, E2M1, b, s2, E2M1, M, N, K, np.zeros((M, N), np.float32))
    assert ref.tolist() == [[1.0, 2.0], [2.0, 4.0], [6.0, 12.0]]


def test_gemm_nan_scale_poisons_row():
    rng = np.random.default_rng(10)
    a = _random_codes(rng, 2, 64, E2M1)
    b = _random_codes(rng, 2, 64, E2M1)
    sa = np.full((2, 2), 127, np.uint8)
    sb = np.full((2, 2), 127, np.uint8)
    sa[1, 1] = 0xFF
    ref, _ = oracle.block_matmul(a, sa, E2M1, b, sb, E2M1, 2, 2, 64, np.zeros((2, 2), np.float32))
    assert np.isnan(ref[1]).all() and not np.isnan(ref[0]).any()


def test_gemm_entries_match_full():
    rng = np.random.default_rng(12)
    M, N, K = 6, 5, 64
    a, b = _random_codes(rng, M, K, E4M3), _random_codes(rng, N, K, E2M1)
    sa = rng.integers(110, 140, (M, 2)).astype(np.uint8)
    sb = rng.integers(110, 140, (N, 2)).astype(np.uint8)
    c0 = rng.standard_normal((M, N)).astype(np.float32)
    ref, sabs = oracle.block_matmul(a, sa, E4M3, b, sb, E2M1, M, N, K, c0)
    ms = np.array([0, 5, 3, 2]); ns = np.array([4, 0, 1, 2])
    r2, s2 = oracle.block_matmul_entries(a, sa, E4M3, b, sb, E2M1, K, ms, ns, c0[ms, ns])
    assert (r2 == ref[ms, ns]).all() and (s2 == sabs[ms, ns]).all()
