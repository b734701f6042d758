"""The decode step of a dense Qwen3-style model, in f64 (test infrastructure).

Dataflow (inferencelayer ``cuda_llm.rs``, ``CudaQwen3::step``; ferrum-kernels
``cuda_decode.rs``, ``decode_step``), per slot, at position ``p``:

1. ``x = embed[token]``
2. per layer: ``hn = rms(x) * attn_norm``; ``y = Wqkv hn``; split q | k | v per head;
   ``q_h = rope(rms(q_h) * q_norm, p)``, ``k_g = rope(rms(k_g) * k_norm, p)``; V as is;
   K and V are stored in the f16 cache at position p; ``o_h`` = attention of ``q_h`` over
   cache positions ``0..p`` of kv head ``h // (n_heads/n_kv_heads)``;
   ``x += Wo o``; ``hn = rms(x) * ffn_norm``; ``x += Wd (silu(Wg hn) * (Wu hn))``
3. ``logits = Wlm (rms(x) * final_norm)``; greedy ``token = argmax(logits)`` (lowest index
   on ties).

Two independent formulations are given: :func:`decode_step` (one position at a time over a
KV cache) and :func:`forward_full` (all positions at once, matrix form with a causal mask).
Prefill is sequential decode, as on the pages ("prefill runs as sequential decode"), so the
two must agree at every position.
"""
from __future__ import annotations

import numpy as np

from . import moe, ops
from .q4_0 import quantize, dequantize

LAYER_MATRICES = ("wqkv", "wo", "wgu", "wd")
MOE_MATRICES = ("wqkv", "wo", "w1", "w2")   # routed experts: w1 gate|up per expert, w2 down


def layer_matrices(cfg):
    return MOE_MATRICES if getattr(cfg, "num_experts", 0) else LAYER_MATRICES


class Q4Model:
    """A model whose linear weights are held as q4_0 codes (quantised by this oracle's codec).

    Matrices are dequantised to f64 when a step needs them (one at a time), so large shapes
    never hold a whole f64 model in memory.
    """

    def __init__(self, cfg, w: dict):
        self.cfg = cfg
        self.embed = np.asarray(w["embed"], dtype=np.float64)
        self.final_norm = np.asarray(w["final_norm"], dtype=np.float64)
        self.lm_head = quantize(w["lm_head"])
        self.layers = []
        for lw in w["layers"]:
            layer = {n: np.asarray(lw[n], dtype=np.float64)
                     for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm")}
            for n in layer_matrices(cfg):
                layer[n] = quantize(lw[n])
            if getattr(cfg, "num_experts", 0):
                layer["router"] = np.asarray(lw["router"], dtype=np.float64)
            self.layers.append(layer)

    @classmethod
    def from_codes(cls, cfg, layers: list, final_norm, lm_head, embed=None) -> "Q4Model":
        """A model from existing q4_0 arrays (``(scales u16 [rows][cols/32], quants u8
        [rows][cols/32][16])`` per matrix, the layout :func:`oracle.q4_0.quantize` returns),
        e.g. codes made by another implementation of the same codec. ``embed`` may be None
        when only :func:`decode_hidden` is used."""
        self = cls.__new__(cls)
        self.cfg = cfg
        self.embed = None if embed is None else np.asarray(embed, dtype=np.float64)
        self.final_norm = np.asarray(final_norm, dtype=np.float64)
        self.lm_head = lm_head
        self.layers = []
        for lw in layers:
            layer = {n: np.asarray(lw[n], dtype=np.float64) for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm")}
            for n in layer_matrices(cfg):
                layer[n] = lw[n]
            if getattr(cfg, "num_experts", 0):
                layer["router"] = np.asarray(lw["router"], dtype=np.float64)
            self.layers.append(layer)
        return self

    @staticmethod
    def dense(q4) -> np.ndarray:
        return dequantize(*q4)


KV_F16 = "f16"
KV_Q8_Q5 = "q8_0/q5_1"


class KVCache:
    """Per slot, per layer: K and V ``[n_kv_heads, capacity, head_dim]`` holding the values the
    cache stores: f16 (``kv="f16"``), or (``kv="q8_0/q5_1"``, memra-engine ``qwen4exp_gpu.rs``,
    the Q8Q5 quantised-cache store) each K row as the decoded q8_0 row and each V row as the
    decoded q5_1 row of its f32 value (``oracle.kvq``)."""

    def __init__(self, cfg, batch: int, capacity: int, kv: str = KV_F16):
        if kv not in (KV_F16, KV_Q8_Q5):
            raise ValueError("unknown KV format")
        self.cfg = cfg
        self.kv = kv
        shape = (batch, cfg.n_layers, cfg.n_kv_heads, capacity, cfg.head_dim)
        self.k = np.zeros(shape, dtype=np.float64)
        self.v = np.zeros(shape, dtype=np.float64)

    def stored(self, k_rows: np.ndarray, v_rows: np.ndarray):
        """The values the cache keeps for rows ``[..., head_dim]`` of K and V."""
        if self.kv == KV_F16:
            return _f16(k_rows), _f16(v_rows)
        from . import kvq
        hd = self.cfg.head_dim
        kr = np.asarray(k_rows, dtype=np.float64).astype(np.float32).reshape(-1, hd)
        vr = np.asarray(v_rows, dtype=np.float64).astype(np.float32).reshape(-1, hd)
        kd = kvq.dequantize_q8_0(kvq.quantize_q8_0(kr), hd).astype(np.float64)
        vd = kvq.dequantize_q5_1(kvq.quantize_q5_1(vr), hd).astype(np.float64)
        return kd.reshape(np.shape(k_rows)), vd.reshape(np.shape(v_rows))

    def preload(self, slot: int, k_ctx: np.ndarray, v_ctx: np.ndarray):
        """Pre-filled context ``[n_layers, n_kv, n_pos, hd]`` at positions 0..n_pos-1 (the f16
        cache keeps its values as f16; the quantised one quantises them)."""
        n = k_ctx.shape[2]
        kd, vd = self.stored(k_ctx, v_ctx)
        self.k[slot, :, :, :n] = kd
        self.v[slot, :, :, :n] = vd


def _f16(a: np.ndarray) -> np.ndarray:
    """The value an f16 cache stores for ``a`` (round to nearest even)."""
    return np.asarray(a, dtype=np.float64).astype(np.float16).astype(np.float64)


def _split_qkv(cfg, y: np.ndarray):
    nh, nkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    q = y[..., : nh * hd].reshape(y.shape[:-1] + (nh, hd))
    k = y[..., nh * hd:(nh + nkv) * hd].reshape(y.shape[:-1] + (nkv, hd))
    v = y[..., (nh + nkv) * hd:].reshape(y.shape[:-1] + (nkv, hd))
    return q, k, v


def decode_step(model: Q4Model, cache: KVCache, tokens, positions, act=None) -> np.ndarray:
    """One decode step for every slot; returns logits ``[B, vocab]`` (f64).

    ``tokens[b]`` sits at position ``positions[b]``; cache positions ``0..positions[b]-1``
    must already hold that slot's context. The step writes K and V of position
    ``positions[b]`` into the cache. ``act``: see :func:`decode_hidden`.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    act = _identity if act is None else act
    hf = decode_hidden(model, cache, model.embed[tokens], positions, act=act)
    return ops.gemv(model.dense(model.lm_head), act(hf))


def _identity(v):
    return v


def decode_hidden(model: Q4Model, cache: KVCache, x, positions, act=None) -> np.ndarray:
    """Steps 2 and the final RMSNorm of 3 for embedded tokens ``x`` ``[B, hidden]``: the
    normalised final hidden state ``[B, hidden]`` that the lm_head multiplies (f64).

    ``act`` (default: none) is applied to the input vector of every GEMV of the layers, for a
    GEMV that reads its activations in a quantised form (e.g. ``oracle.act8.absmax_dequant``,
    the int8 absmax form of inferencelayer ``cuda_llm.rs``); the lm_head's input is left to the
    caller."""
    cfg = model.cfg
    act = _identity if act is None else act
    positions = np.asarray(positions, dtype=np.int64)
    x = np.array(x, dtype=np.float64)                               # [B, hidden]
    B = x.shape[0]
    scale = 1.0 / np.sqrt(cfg.head_dim)
    for li, L in enumerate(model.layers):
        hn = ops.rmsnorm(x, L["attn_norm"], cfg.eps)
        y = ops.gemv(model.dense(L["wqkv"]), act(hn))
        q, k, v = _split_qkv(cfg, y)
        o = np.empty((B, cfg.n_heads, cfg.head_dim))
        for b in range(B):
            p = int(positions[b])
            qb = ops.rope(ops.rmsnorm(q[b], L["q_norm"], cfg.eps), p, cfg.rope_theta)
            kb = ops.rope(ops.rmsnorm(k[b], L["k_norm"], cfg.eps), p, cfg.rope_theta)
            cache.k[b, li, :, p], cache.v[b, li, :, p] = cache.stored(kb, v[b])
            o[b] = ops.gqa_attention(qb, cache.k[b, li, :, : p + 1],
                                     cache.v[b, li, :, : p + 1], scale)
        x = x + ops.gemv(model.dense(L["wo"]), act(o.reshape(B, -1)))
        hn = ops.rmsnorm(x, L["ffn_norm"], cfg.eps)
        if getattr(cfg, "num_experts", 0):
            for b in range(B):
                x[b] = x[b] + moe.moe_ffn(hn[b], L["router"], L["w1"], L["w2"], cfg)[0]
            continue
        gu = ops.gemv(model.dense(L["wgu"]), act(hn))
        a = ops.swiglu(gu[:, : cfg.intermediate], gu[:, cfg.intermediate:])
        x = x + ops.gemv(model.dense(L["wd"]), act(a))
    return ops.rmsnorm(x, model.final_norm, cfg.eps)


def logits_by_rows(lm_head, hf, rows_per_chunk: int = 8192) -> np.ndarray:
    """``W_lm hf`` for a q4_0 lm_head dequantised ``rows_per_chunk`` rows at a time (each
    logit is the same dot product as in :func:`decode_step`; only the memory differs):
    ``[B, vocab]`` f64."""
    scales, quants = lm_head
    rows = scales.shape[0]
    hf = np.asarray(hf, dtype=np.float64)
    out = np.empty((hf.shape[0], rows))
    for r0 in range(0, rows, rows_per_chunk):
        r1 = min(rows, r0 + rows_per_chunk)
        out[:, r0:r1] = ops.gemv(dequantize(scales[r0:r1], quants[r0:r1]), hf)
    return out


def forward_full(model: Q4Model, tokens, k_ctx=None, v_ctx=None) -> np.ndarray:
    """All positions of one sequence at once (matrix form, causal mask).

    ``tokens [T]`` occupy positions ``n0 .. n0+T-1`` after an optional pre-filled context
    ``k_ctx, v_ctx [n_layers, n_kv, n0, hd]``. Returns logits ``[T, vocab]``. Keys and values
    are rounded to f16 before use, as the f16 cache stores them.
    """
    cfg = model.cfg
    tokens = np.asarray(tokens, dtype=np.int64)
    T = tokens.shape[0]
    n0 = 0 if k_ctx is None else k_ctx.shape[2]
    nh, nkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    group = nh // nkv
    scale = 1.0 / np.sqrt(hd)
    pos = n0 + np.arange(T)
    # causal mask over [n0 + T] keys for each of the T queries
    key_pos = np.arange(n0 + T)
    mask = key_pos[None, :] <= pos[:, None]                          # [T, n0+T]
    x = model.embed[tokens].copy()                                   # [T, hidden]
    for li, L in enumerate(model.layers):
        hn = ops.rmsnorm(x, L["attn_norm"], cfg.eps)
        y = hn @ model.dense(L["wqkv"]).T                            # [T, qkv]
        q, k, v = _split_qkv(cfg, y)                                 # [T, heads, hd]
        q = ops.rmsnorm(q, L["q_norm"], cfg.eps)
        k = ops.rmsnorm(k, L["k_norm"], cfg.eps)
        q = np.stack([ops.rope(q[t], int(pos[t]), cfg.rope_theta) for t in range(T)])
        k = np.stack([ops.rope(k[t], int(pos[t]), cfg.rope_theta) for t in range(T)])
        K = _f16(k).transpose(1, 0, 2)                               # [nkv, T, hd]
        V = _f16(v).transpose(1, 0, 2)
        if n0:
            K = np.concatenate([np.asarray(k_ctx[li], np.float16).astype(np.float64), K], axis=1)
            V = np.concatenate([np.asarray(v_ctx[li], np.float16).astype(np.float64), V], axis=1)
        o = np.empty((T, nh, hd))
        for h in range(nh):
            g = h // group
            s = (q[:, h, :] @ K[g].T) * scale                        # [T, n0+T]
            s = np.where(mask, s, -np.inf)
            o[:, h, :] = ops.softmax(s) @ V[g]
        x = x + o.reshape(T, -1) @ model.dense(L["wo"]).T
        hn = ops.rmsnorm(x, L["ffn_norm"], cfg.eps)
        if getattr(cfg, "num_experts", 0):
            # every position routes on its own normalised input
            x = x + np.stack([moe.moe_ffn(hn[t], L["router"], L["w1"], L["w2"], cfg)[0] for t in range(T)])
            continue
        gu = hn @ model.dense(L["wgu"]).T
        x = x + ops.swiglu(gu[:, : cfg.intermediate], gu[:, cfg.intermediate:]) \
            @ model.dense(L["wd"]).T
    hf = ops.rmsnorm(x, model.final_norm, cfg.eps)
    return hf @ model.dense(model.lm_head).T


def greedy(logits: np.ndarray) -> np.ndarray:
    """Greedy next token per row (lowest index among equal maxima)."""
    return ops.argmax_lowest(logits)


def agreement_tolerance(top1: float) -> float:
    """Logit tolerance at a greedy step: 2e-2 absolute + 1e-2 relative to the top logit."""
    return 2e-2 + 1e-2 * abs(float(top1))


def greedy_must_agree(oracle_logits: np.ndarray) -> bool:
    """True where the oracle's top-2 margin exceeds the tolerance, so a tie flip is impossible."""
    row = np.asarray(oracle_logits, dtype=np.float64)
    i = int(np.argmax(row))
    rest = np.delete(row, i)
    margin = row[i] - (rest.max() if rest.size else -np.inf)
    return bool(margin > agreement_tolerance(row[i]))


def logits_close(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Element-wise logit parity: ``|got - want| <= 2e-2 + 1e-2 |want|``."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return np.abs(got - want) <= 2e-2 + 1e-2 * np.abs(want)
