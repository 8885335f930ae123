"""Seeded synthetic inputs for the five MX workloads.

This module holds no MX arithmetic: it only draws tensors (numpy
``default_rng``) in the shapes, distributions and special structures of the
workloads, so that the CPU oracle and the GPU path can be fed the same bits.
bf16 tensors are made by rounding float32 draws to nearest-even with torch.

Workloads (each a dict of named host arrays; f32 as numpy float32, bf16 as a
CPU torch.bfloat16 tensor):

  1 ``mxfp4_roundtrip_128``: A f32 128x256 and B f32 256x128, N(0,1), 1% of
    the positions of each multiplied by 100; Bt = B transposed (N x K, so that
    B is blocked along its reduction axis); C0 f32 128x128 zeros.
  2 ``mxfp8_act_4096``: x bf16 4096x4096, N(0,1) with 1% of positions replaced
    by Student-t(3) draws; 64 all-zero blocks; 64 blocks of magnitude ~2^-130;
    64 blocks with one element 1.0 and the rest in 2^-20..2^-16; plus 64 block
    indices whose scale is set to 0xFF before dequantize (``nan_blocks``).
  3 ``decode_mixed_16x14336x4096``: A bf16 16x4096 N(0,1); W f32 14336x4096
    N(0, 0.02) with one element per row multiplied by 20; C0 f32 16x14336 N(0,1).
  4 ``square_mxfp8_8192``: A, Bt f32 8192x8192 N(0,1); C0 uniform[-1,1].
  5 ``prefill_mxfp4_8192x28672x8192``: A bf16 8192x8192 N(0,1) with 0.1% of
    positions multiplied by 100; W f32 28672x8192 N(0, 0.02); C0 zeros.
  6 ``decode_f32b_16x14336x4096``: the product with an unquantized f32 right
    operand: A bf16 16x4096 N(0,1) (quantized to MXFP8 before the product);
    B f32 4096x14336 (K x N, row-major) N(0, 0.02) with one element per column
    multiplied by 20 (the per-output-channel outliers of workload 3's W, drawn
    directly in the K x N orientation); C0 f32 16x14336 N(0,1).

``scale`` (0 < scale <= 1) shrinks the row counts of the large workloads for
quick runs; the full workloads use scale = 1.
"""
from __future__ import annotations

import numpy as np
import torch

NAMES = {
    1: "mxfp4_roundtrip_128",
    2: "mxfp8_act_4096",
    3: "decode_mixed_16x14336x4096",
    4: "square_mxfp8_8192",
    5: "prefill_mxfp4_8192x28672x8192",
    6: "decode_f32b_16x14336x4096",
}

BLOCK = 32


def _normal(rng, shape, std=1.0):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def _outliers(rng, x, frac, factor):
    n = x.size
    k = max(1, int(round(frac * n)))
    pos = rng.choice(n, size=k, replace=False)
    flat = x.reshape(-1)
    flat[pos] *= np.float32(factor)
    return x


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)


def _rows(n, scale):
    return max(1, int(n * scale))


def workload1(seed: int = 0):
    rng = np.random.default_rng(seed)
    A = _outliers(rng, _normal(rng, (128, 256)), 0.01, 100.0)
    B = _outliers(rng, _normal(rng, (256, 128)), 0.01, 100.0)
    return {"A": A, "B": B, "Bt": np.ascontiguousarray(B.T), "C0": np.zeros((128, 128), np.float32),
            "M": 128, "N": 128, "K": 256}


def workload2(seed: int = 0, scale: float = 1.0):
    rng = np.random.default_rng(seed)
    R, K = _rows(4096, scale), 4096
    x = _normal(rng, (R, K))
    n = x.size
    pos = rng.choice(n, size=max(1, int(round(0.01 * n))), replace=False)
    x.reshape(-1)[pos] = rng.standard_t(3, size=pos.size).astype(np.float32)
    nblk = n // BLOCK
    special = rng.choice(nblk, size=64 * 3, replace=False)
    zero_b, tiny_b, sub_b = special[:64], special[64:128], special[128:]
    xb = x.reshape(nblk, BLOCK)
    xb[zero_b] = 0.0
    xb[tiny_b] = (_normal(rng, (64, BLOCK)) * np.float32(2.0 ** -130)).astype(np.float32)
    mags = np.float32(2.0) ** rng.uniform(-20, -16, (64, BLOCK)).astype(np.float32)
    signs = rng.choice(np.array([-1, 1], np.float32), (64, BLOCK))
    xb[sub_b] = (mags * signs).astype(np.float32)
    xb[sub_b, 0] = 1.0
    nan_blocks = np.sort(rng.choice(nblk, size=64, replace=False))
    return {"x": _bf16(x), "rows": R, "cols": K, "nan_blocks": nan_blocks,
            "zero_blocks": np.sort(zero_b), "tiny_blocks": np.sort(tiny_b), "subnormal_blocks": np.sort(sub_b)}


def workload3(seed: int = 0, scale: float = 1.0):
    rng = np.random.default_rng(seed)
    M, N, K = 16, _rows(14336, scale), 4096
    A = _bf16(_normal(rng, (M, K)))
    W = _normal(rng, (N, K), 0.02)
    cols = rng.integers(0, K, N)
    W[np.arange(N), cols] *= np.float32(20.0)
    C0 = _normal(rng, (M, N))
    return {"A": A, "W": W, "C0": C0, "M": M, "N": N, "K": K}


def workload4(seed: int = 0, scale: float = 1.0):
    rng = np.random.default_rng(seed)
    M, N, K = _rows(8192, scale), _rows(8192, scale), 8192
    A = _normal(rng, (M, K))
    Bt = _normal(rng, (N, K))
    C0 = rng.uniform(-1.0, 1.0, (M, N)).astype(np.float32)
    return {"A": A, "Bt": Bt, "C0": C0, "M": M, "N": N, "K": K}


def workload5(seed: int = 0, scale: float = 1.0):
    rng = np.random.default_rng(seed)
    M, N, K = _rows(8192, scale), _rows(28672, scale), 8192
    A = _bf16(_outliers(rng, _normal(rng, (M, K)), 0.001, 100.0))
    W = _normal(rng, (N, K), 0.02)
    C0 = np.zeros((M, N), np.float32)
    return {"A": A, "W": W, "C0": C0, "M": M, "N": N, "K": K}


def workload6(seed: int = 0, scale: float = 1.0):
    rng = np.random.default_rng(seed)
    M, N, K = 16, _rows(14336, scale) // 4 * 4, 4096
    A = _bf16(_normal(rng, (M, K)))
    B = _normal(rng, (K, N), 0.02)
    rows = rng.integers(0, K, N)
    B[rows, np.arange(N)] *= np.float32(20.0)
    C0 = _normal(rng, (M, N))
    return {"A": A, "B": B, "C0": C0, "M": M, "N": N, "K": K}


def make(cfg: int, seed: int = 0, scale: float = 1.0):
    if cfg == 1:
        return workload1(seed)
    return {2: workload2, 3: workload3, 4: workload4, 5: workload5, 6: workload6}[cfg](seed, scale)
