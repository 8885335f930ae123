"""Helpers for the GPU parity tests: layout conversions and comparisons.

Nothing here computes MX arithmetic: the tensor-core scale layout is an index
permutation (its formula is documented in include/mx.h), and nibble unpacking
only splits bytes."""
import numpy as np
import torch


def mma_offsets(rows: int, nb: int) -> np.ndarray:
    """Byte offset of scale (r, j) in the tensor-core layout, as an [rows, nb] array."""
    nb4 = (nb + 3) // 4 * 4
    r = np.arange(rows, dtype=np.int64)[:, None]
    j = np.arange(nb, dtype=np.int64)[None, :]
    return ((r >> 7) * (nb4 >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3)


def mma_to_rowmajor(buf: np.ndarray, rows: int, nb: int) -> np.ndarray:
    return np.asarray(buf).reshape(-1)[mma_offsets(rows, nb)]


def mma_padding_mask(rows: int, nb: int) -> np.ndarray:
    """True at the bytes of the tensor-core layout that hold no real scale."""
    nb4 = (nb + 3) // 4 * 4
    r128 = (rows + 127) // 128 * 128
    size = r128 // 128 * (nb4 // 4) * 512
    mask = np.ones(size, bool)
    mask[mma_offsets(rows, nb).reshape(-1)] = False
    return mask


def rowmajor_to_mma(s: np.ndarray, rows: int, nb: int) -> np.ndarray:
    nb4 = (nb + 3) // 4 * 4
    r128 = (rows + 127) // 128 * 128
    out = np.zeros(r128 // 128 * (nb4 // 4) * 512, np.uint8)
    out[mma_offsets(rows, nb)] = np.asarray(s).reshape(rows, nb)
    return out


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def same_f32_bits(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Elementwise: identical bit patterns, or both NaN (any payload)."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    return (a.view(np.uint32) == b.view(np.uint32)) | (np.isnan(a) & np.isnan(b))


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()
