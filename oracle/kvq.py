"""Quantised KV-cache rows: the q8_0 (keys) and q5_1 (values) codecs, stated plainly (test
infrastructure; see the package docstring).

Source: memra-engine ``qwen4exp_gpu.rs``, the quantised-cache storage items
(``q8_row_bytes`` / ``q5_row_bytes``, the ``Q8Q5`` store, and the host twins
``host_quant_q8_row``, ``host_deq_q8_rows``, ``host_quant_q5_row``, ``host_deq_q5_rows``,
which the page states are bit-identical to its device kernels). The page fixes the precision:
every step is an f32 operation, the f16 conversions round to nearest even.

A row of ``dim`` values is cut into blocks of 32 consecutive elements; a ragged last block is
padded with zeros, and the padding takes part in the block's statistics.

q8_0, 34 bytes per block: the f16 scale ``d`` (little-endian), then 32 signed 8-bit codes.
    amax = max |x|;  d = amax / 127;  id = 1 / d, or 0 when d == 0 or 1 / d is not finite;
    code = clamp(round_half_even(x * id), -127, 127);  stored d = f16(d).
    Decoded value: f32(stored d) * code (one f32 product, exact).

q5_1, 24 bytes per block: f16 ``d``, f16 ``m``, a 32-bit word whose bit l is bit 4 of code l,
then 16 bytes whose byte l holds the low four bits of code l (low nibble) and of code l + 16
(high nibble).
    mn = min x;  mx = max x;  d = (mx - mn) / 31;  id as for q8_0;
    code = clamp(round_half_even((x - mn) * id), 0, 31);  stored d = f16(d), m = f16(mn).
    Decoded value: fma(f32(d), code, f32(m)) rounded once to f32. (d * code is exact in f32:
    an 11-bit mantissa times a 5-bit integer, so the fma is one f32 addition.)

Inputs must be finite (the page's domain: projection outputs). Reading where the page is
silent: the sign of a zero block minimum (a -0 and a +0 both minimal) is not fixed by it; the
minimum is taken as ``min + 0`` in f32, so a zero minimum is stored as +0.
"""
from __future__ import annotations

import numpy as np

QK = 32
Q8_BLOCK_BYTES = 34
Q5_BLOCK_BYTES = 24


def q8_row_bytes(dim: int) -> int:
    return -(-dim // QK) * Q8_BLOCK_BYTES


def q5_row_bytes(dim: int) -> int:
    return -(-dim // QK) * Q5_BLOCK_BYTES


def _blocks(rows) -> np.ndarray:
    """[n, dim] f32 -> [n, nblk, 32] f32, the ragged tail padded with zeros."""
    x = np.asarray(rows, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("kvq: need a 2-D array of rows")
    if not np.all(np.isfinite(x)):
        raise ValueError("kvq: rows must be finite")
    n, dim = x.shape
    nblk = -(-dim // QK)
    pad = np.zeros((n, nblk * QK), dtype=np.float32)
    pad[:, :dim] = x
    return pad.reshape(n, nblk, QK)


def _inverse(d: np.ndarray) -> np.ndarray:
    """1 / d in f32; 0 where d == 0 or the reciprocal is not finite (a subnormal d)."""
    with np.errstate(divide="ignore", over="ignore"):
        inv = np.float32(1.0) / d
    return np.where((d != 0) & np.isfinite(inv), inv, np.float32(0.0)).astype(np.float32)


def _f16_bits(v: np.ndarray) -> np.ndarray:
    """f32 -> f16 (round to nearest even) as uint16 bit patterns."""
    with np.errstate(over="ignore"):
        h = np.asarray(v, dtype=np.float32).astype(np.float16)
    if not np.all(np.isfinite(h)):
        raise ValueError("kvq: a block scale or minimum overflows f16")
    return h.view(np.uint16)


def quantize_q8_0(rows) -> np.ndarray:
    """Rows [n, dim] -> bytes [n, q8_row_bytes(dim)]."""
    b = _blocks(rows)
    n, nblk, _ = b.shape
    amax = np.max(np.abs(b), axis=2)                       # exact
    d = (amax / np.float32(127.0)).astype(np.float32)
    inv = _inverse(d)
    prod = (b * inv[:, :, None]).astype(np.float32)        # one f32 product per element
    code = np.clip(np.rint(prod), -127, 127).astype(np.int8)   # rint: ties to even
    out = np.zeros((n, nblk, Q8_BLOCK_BYTES), dtype=np.uint8)
    db = _f16_bits(d)
    out[:, :, 0] = (db & 0xFF).astype(np.uint8)
    out[:, :, 1] = (db >> 8).astype(np.uint8)
    out[:, :, 2:] = code.view(np.uint8)
    return out.reshape(n, nblk * Q8_BLOCK_BYTES)


def dequantize_q8_0(data, dim: int) -> np.ndarray:
    """Bytes [n, q8_row_bytes(dim)] -> f32 rows [n, dim]."""
    raw = np.asarray(data, dtype=np.uint8)
    nblk = -(-dim // QK)
    blk = raw.reshape(raw.shape[0], nblk, Q8_BLOCK_BYTES)
    d = (blk[:, :, 0].astype(np.uint16) | (blk[:, :, 1].astype(np.uint16) << 8)).view(np.float16)
    code = blk[:, :, 2:].view(np.int8).astype(np.float32)
    vals = (d.astype(np.float32)[:, :, None] * code).astype(np.float32)
    return vals.reshape(raw.shape[0], nblk * QK)[:, :dim]


def quantize_q5_1(rows) -> np.ndarray:
    """Rows [n, dim] -> bytes [n, q5_row_bytes(dim)]."""
    b = _blocks(rows)
    n, nblk, _ = b.shape
    mn = (np.min(b, axis=2) + np.float32(0.0)).astype(np.float32)   # a zero minimum is stored as +0
    mx = np.max(b, axis=2)
    d = ((mx - mn).astype(np.float32) / np.float32(31.0)).astype(np.float32)
    inv = _inverse(d)
    diff = (b - mn[:, :, None]).astype(np.float32)        # one f32 subtraction
    prod = (diff * inv[:, :, None]).astype(np.float32)     # one f32 product
    code = np.clip(np.rint(prod), 0, 31).astype(np.uint32)
    qh = np.zeros((n, nblk), dtype=np.uint32)
    for l in range(QK):
        qh |= ((code[:, :, l] >> 4) & 1) << np.uint32(l)
    lo = (code & 0x0F).astype(np.uint8)
    nib = lo[:, :, :16] | (lo[:, :, 16:] << 4)
    out = np.zeros((n, nblk, Q5_BLOCK_BYTES), dtype=np.uint8)
    db, mb = _f16_bits(d), _f16_bits(mn)
    out[:, :, 0] = (db & 0xFF).astype(np.uint8)
    out[:, :, 1] = (db >> 8).astype(np.uint8)
    out[:, :, 2] = (mb & 0xFF).astype(np.uint8)
    out[:, :, 3] = (mb >> 8).astype(np.uint8)
    for k in range(4):
        out[:, :, 4 + k] = ((qh >> np.uint32(8 * k)) & 0xFF).astype(np.uint8)
    out[:, :, 8:] = nib
    return out.reshape(n, nblk * Q5_BLOCK_BYTES)


def q5_1_codes(data, dim: int) -> np.ndarray:
    """The 5-bit codes [n, nblk * 32] of q5_1 bytes (bit 4 from the high-bit word)."""
    raw = np.asarray(data, dtype=np.uint8)
    nblk = -(-dim // QK)
    blk = raw.reshape(raw.shape[0], nblk, Q5_BLOCK_BYTES)
    qh = np.zeros(blk.shape[:2], dtype=np.uint32)
    for k in range(4):
        qh |= blk[:, :, 4 + k].astype(np.uint32) << np.uint32(8 * k)
    nib = blk[:, :, 8:]
    lo = np.concatenate([nib & 0x0F, nib >> 4], axis=2).astype(np.uint32)   # elements 0..15, 16..31
    hi = (qh[:, :, None] >> np.arange(QK, dtype=np.uint32)[None, None, :]) & 1
    return (lo | (hi << 4)).reshape(raw.shape[0], nblk * QK)


def dequantize_q5_1(data, dim: int) -> np.ndarray:
    """Bytes [n, q5_row_bytes(dim)] -> f32 rows [n, dim]."""
    raw = np.asarray(data, dtype=np.uint8)
    nblk = -(-dim // QK)
    blk = raw.reshape(raw.shape[0], nblk, Q5_BLOCK_BYTES)
    d = (blk[:, :, 0].astype(np.uint16) | (blk[:, :, 1].astype(np.uint16) << 8)).view(np.float16)
    m = (blk[:, :, 2].astype(np.uint16) | (blk[:, :, 3].astype(np.uint16) << 8)).view(np.float16)
    code = q5_1_codes(raw, dim).reshape(raw.shape[0], nblk, QK).astype(np.float32)
    prod = d.astype(np.float32)[:, :, None] * code                     # exact in f32
    vals = (prod + m.astype(np.float32)[:, :, None]).astype(np.float32)  # the fma's one rounding
    return vals.reshape(raw.shape[0], nblk * QK)[:, :dim]


def paged_attention_q8k_q5v(q, k_codes, v_codes, head_dim, block_tables, lens, scale):
    """Paged GQA decode attention over a quantised pool: K rows q8_0, V rows q5_1.

    ``k_codes`` / ``v_codes``: uint8 [num_blocks, n_kv, 16, q8_row_bytes(hd)] /
    [..., q5_row_bytes(hd)], one quantised row per (block, kv head, slot). The rows are decoded
    as above and the attention is the plain f64 definition of ``oracle.ops.paged_attention``
    over the decoded pools.
    """
    from oracle import ops
    kc = np.asarray(k_codes, dtype=np.uint8)
    vc = np.asarray(v_codes, dtype=np.uint8)
    lead = kc.shape[:3]
    kp = dequantize_q8_0(kc.reshape(-1, kc.shape[-1]), head_dim).reshape(*lead, head_dim)
    vp = dequantize_q5_1(vc.reshape(-1, vc.shape[-1]), head_dim).reshape(*lead, head_dim)
    return ops.paged_attention(q, kp, vp, block_tables, lens, scale)
