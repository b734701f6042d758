"""Per-operation definitions in f64 (test infrastructure; see the package docstring).

Each function is the plain definition of one step of the decode path; none is blocked,
fused or reordered.
"""
from __future__ import annotations

import numpy as np


def gemv(w: np.ndarray, x: np.ndarray) -> np.ndarray:
    """``y[b, r] = sum_k w[r, k] x[b, k]`` (a dense matrix product, f64).

    The q4_0 GEMV of inferencelayer ``cuda_llm.rs`` (``CudaQwen3::gemv``) computes this with
    ``w`` the dequantised matrix.
    """
    w = np.asarray(w, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    return x @ w.T


def rmsnorm(v: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """``v / sqrt(mean(v^2) + eps) * w`` over the last axis.

    memra-engine ``qwen4exp_gpu.rs`` ``host_rms_norm`` (effective weights); the weight is
    the stored value itself (Qwen3 convention, inferencelayer ``Cfg``).
    """
    v = np.asarray(v, dtype=np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rope_angles(position: int, head_dim: int, theta: float) -> np.ndarray:
    """Angles ``position * theta^(-2i/head_dim)`` for i < head_dim/2 (f64).

    inferencelayer ``cuda_llm.rs`` ``rope_inv_freq`` (default rope type).
    """
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = np.power(float(theta), -(2.0 * i) / head_dim)
    return float(position) * inv_freq


def rope(v: np.ndarray, position: int, theta: float) -> np.ndarray:
    """NeoX split-half rotation of every head vector in ``v [..., head_dim]``.

    Pairs ``(i, i + head_dim/2)``: ``(a, b) -> (a cos - b sin, a sin + b cos)``
    (memra-engine ``qwen4exp_gpu.rs`` ``host_rope_at``).
    """
    v = np.asarray(v, dtype=np.float64)
    hd = v.shape[-1]
    half = hd // 2
    ang = rope_angles(position, hd, theta)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., :half], v[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def silu(z: np.ndarray) -> np.ndarray:
    """``z / (1 + exp(-z))``."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """``silu(gate) * up`` (the SwiGLU activation fed to the down projection)."""
    return silu(gate) * np.asarray(up, dtype=np.float64)


def softmax(s: np.ndarray) -> np.ndarray:
    """Softmax over the last axis (max-subtracted; mathematically the plain definition)."""
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def kv_head_of(h: int, n_heads: int, n_kv_heads: int) -> int:
    """GQA: query head h reads kv head ``h // (n_heads / n_kv_heads)``."""
    return h // (n_heads // n_kv_heads)


def gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Decode attention of one sequence over its whole (already causal) context.

    ``q [n_heads, hd]``, ``k, v [n_kv_heads, L, hd]`` ->
    ``o[h] = sum_t softmax_t(q_h . k_{g(h), t} * scale) v_{g(h), t}`` with ``g`` from
    :func:`kv_head_of`. ferrum-kernels ``cuda_decode.rs`` ``attention_paged``: every stored
    position up to and including the current token is attended (valid length = len + 1),
    scale = 1/sqrt(hd).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nh, nkv = q.shape[0], k.shape[0]
    out = np.empty_like(q)
    for h in range(nh):
        g = kv_head_of(h, nh, nkv)
        p = softmax(k[g] @ q[h] * scale)
        out[h] = p @ v[g]
    return out


def gather_paged(pool: np.ndarray, block_table, length: int) -> np.ndarray:
    """Logical ``[n_kv_heads, length, hd]`` view of a paged pool.

    ``pool [num_blocks, n_kv_heads, block_size, hd]``; position p lives in physical block
    ``block_table[p // block_size]``, slot ``p % block_size`` (ferrum-kernels
    ``cuda_decode.rs`` ``attention_paged`` / ``PagedSequenceKvState``).
    """
    pool = np.asarray(pool)
    bs = pool.shape[2]
    rows = []
    for p in range(length):
        rows.append(pool[int(block_table[p // bs]), :, p % bs, :])
    if not rows:
        return np.zeros((pool.shape[1], 0, pool.shape[3]), dtype=np.float64)
    return np.stack(rows, axis=1).astype(np.float64)


def paged_attention(q, k_pool, v_pool, block_tables, lens, scale: float) -> np.ndarray:
    """Batched paged decode attention: ``q [B, nh, hd]`` -> ``o [B, nh, hd]`` (f64)."""
    q = np.asarray(q)
    out = np.empty(q.shape, dtype=np.float64)
    for b in range(q.shape[0]):
        L = int(lens[b])
        if L < 1:
            raise ValueError("context length must be >= 1")
        k = gather_paged(k_pool, block_tables[b], L)
        v = gather_paged(v_pool, block_tables[b], L)
        out[b] = gqa_attention(q[b], k, v, scale)
    return out


def argmax_lowest(logits: np.ndarray) -> np.ndarray:
    """Greedy token: the index of the largest logit, the lowest index among equal maxima."""
    logits = np.asarray(logits)
    return np.argmax(logits, axis=-1)  # numpy returns the first occurrence of the maximum
