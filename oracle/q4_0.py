"""q4_0 codec, stated plainly (test infrastructure; see the package docstring).

Format (inferencelayer ``cuda_llm.rs``, ``Q4Dev`` and its doc comment): a ``[rows, cols]``
matrix is cut row-wise into blocks of 32 consecutive weights; each block has one f16 scale
``d`` and 16 bytes of 4-bit codes ``q``; the weight is ``(q - 8) * d``. Scales and codes are
separate arrays (``scales [rows][cols/32]``, ``quants [rows][cols/32][16]``).

Readings where the pages are silent (the quantiser ``quantize_q4_0`` itself is not shown):

* scale: ``d = f16_round_nearest_even(max|x| / 7)``, the division in f64;
* code: ``q = clamp(round_half_even(x / d), -7, 7) + 8`` in f64; a block with ``d == 0``
  gets ``q = 8`` everywhere. This keeps ``|x - (q - 8) d| <= d / 2`` for every weight whose
  block scale is a normal f16 (the bound the decode method relies on);
* nibble order: byte ``j`` (0..15) of a block holds element ``j`` in its low nibble and
  element ``j + 16`` in its high nibble;
* a non-finite weight, or a block whose scale overflows f16, is an error.
"""
from __future__ import annotations

import numpy as np

QK = 32  # weights per block


def f16_scale(amax: np.ndarray) -> np.ndarray:
    """Block scale d as an f16 array: nearest f16 to amax/7 (ties to even), from f64."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(over="ignore"):
        d = (amax / 7.0).astype(np.float16)  # IEEE round-to-nearest-even from double
    if not np.all(np.isfinite(d)):
        raise ValueError("q4_0: a block scale overflows f16")
    return d


def quantize(w) -> tuple[np.ndarray, np.ndarray]:
    """Quantise ``w [rows, cols]`` (cols % 32 == 0) to (scales u16 bits, quants u8)."""
    w = np.asarray(w)
    if w.ndim != 2 or w.shape[1] % QK != 0:
        raise ValueError("q4_0: need a 2-D matrix with cols % 32 == 0")
    x = w.astype(np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("q4_0: non-finite weight")
    rows, cols = x.shape
    blocks = x.reshape(rows, cols // QK, QK)
    amax = np.abs(blocks).max(axis=-1)
    d16 = f16_scale(amax)
    d = d16.astype(np.float64)[..., None]
    safe = np.where(d > 0.0, d, 1.0)
    q = np.clip(np.rint(blocks / safe), -7, 7) + 8          # np.rint rounds half to even
    q = np.where(d > 0.0, q, 8.0).astype(np.uint8)
    quants = (q[..., :16] | (q[..., 16:] << 4)).astype(np.uint8)
    return d16.view(np.uint16), quants


def codes(quants: np.ndarray) -> np.ndarray:
    """Unpack ``quants [..., 16]`` into the 32 codes of each block, in element order."""
    quants = np.asarray(quants, dtype=np.uint8)
    lo = quants & 0x0F
    hi = quants >> 4
    return np.concatenate([lo, hi], axis=-1)


def dequantize(scales: np.ndarray, quants: np.ndarray) -> np.ndarray:
    """``w[r, 32 j + e] = (q - 8) * d`` in f64, the f16 scale taken exactly."""
    scales = np.asarray(scales, dtype=np.uint16)
    d = scales.view(np.float16).astype(np.float64)
    q = codes(quants).astype(np.float64)
    w = (q - 8.0) * d[..., None]
    rows = w.shape[0]
    return w.reshape(rows, -1)
