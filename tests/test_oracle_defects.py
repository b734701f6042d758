"""Deliberate-defect gates: a plausible mistake planted in the oracle (on the CPU) must make
one of its pins fail. A pin that a wrong oracle also passes is no pin."""
import math

import numpy as np
import pytest

import ql_inputs
from oracle import decode, ops, q4_0

from test_oracle_q4_0 import load_golden


def golden_ok(quantize):
    for name, x, scale, qb in load_golden():
        s, q = quantize(x[None, :])
        if int(s[0, 0]) != scale or not np.array_equal(q[0, 0], qb):
            return False
    return True


def test_golden_accepts_the_oracle():
    assert golden_ok(q4_0.quantize)


def test_wrong_nibble_order_is_caught():
    def bad(w):
        s, q = q4_0.quantize(w)
        c = q4_0.codes(q)                      # element order
        q2 = (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)   # adjacent pairs
        return s, q2
    assert not golden_ok(bad)


def test_wrong_scale_rule_is_caught():
    def bad(w):  # d = max|x| / 8 (a plausible alternative) instead of / 7
        x = np.asarray(w, np.float64).reshape(w.shape[0], -1, 32)
        d16 = (np.abs(x).max(-1) / 8.0).astype(np.float16)
        d = d16.astype(np.float64)[..., None]
        q = np.where(d > 0, np.clip(np.rint(x / np.where(d > 0, d, 1)), -8, 7) + 8, 8)
        q = q.astype(np.uint8)
        return d16.view(np.uint16), (q[..., :16] | (q[..., 16:] << 4)).astype(np.uint8)
    assert not golden_ok(bad)


def test_truncating_rounding_is_caught():
    def bad(w):  # truncation instead of round-half-even
        x = np.asarray(w, np.float64).reshape(w.shape[0], -1, 32)
        d16 = q4_0.f16_scale(np.abs(x).max(-1))
        d = d16.astype(np.float64)[..., None]
        q = np.where(d > 0, np.clip(np.trunc(x / np.where(d > 0, d, 1)), -7, 7) + 8, 8)
        q = q.astype(np.uint8)
        return d16.view(np.uint16), (q[..., :16] | (q[..., 16:] << 4)).astype(np.uint8)
    assert not golden_ok(bad)


def rope_pin_ok(rope):
    hd, p = 8, 3
    e0 = np.zeros(hd)
    e0[0] = 1.0
    r = rope(e0, p, 10000.0)
    return abs(r[0] - math.cos(p)) < 1e-15 and abs(r[hd // 2] - math.sin(p)) < 1e-15


def test_adjacent_rope_pairing_is_caught():
    def bad(v, position, theta):  # GPT-J interleaved pairs (2i, 2i+1)
        v = np.asarray(v, np.float64)
        ang = ops.rope_angles(position, v.shape[-1], theta)
        a, b = v[..., 0::2], v[..., 1::2]
        out = np.empty_like(v)
        out[..., 0::2] = a * np.cos(ang) - b * np.sin(ang)
        out[..., 1::2] = a * np.sin(ang) + b * np.cos(ang)
        return out
    assert rope_pin_ok(ops.rope)
    assert not rope_pin_ok(bad)


def test_rope_sign_error_is_caught():
    def bad(v, position, theta):
        return ops.rope(v, -position, theta)
    assert not rope_pin_ok(bad)


def test_wrong_gqa_mapping_is_caught(monkeypatch):
    nh, nkv, L, hd = 8, 2, 5, 4
    rng = np.random.default_rng(0)
    v = np.stack([np.full((L, hd), float(g)) for g in range(nkv)])
    args = (rng.standard_normal((nh, hd)), rng.standard_normal((nkv, L, hd)), v, 1.0)
    monkeypatch.setattr(ops, "kv_head_of", lambda h, a, b: h % b)
    o = ops.gqa_attention(*args)
    assert not np.allclose(o[:, 0], [0, 0, 0, 0, 1, 1, 1, 1])


def test_rmsnorm_without_mean_is_caught():
    w = np.linspace(0.5, 1.5, 16)
    v = np.full(16, 3.0)
    bad = v / np.sqrt(np.sum(v * v) + 1e-6) * w
    assert not np.allclose(bad, 3.0 / math.sqrt(9.0 + 1e-6) * w, rtol=1e-14)


SMALL = ql_inputs.Config(hidden=64, n_layers=1, n_heads=4, n_kv_heads=2, head_dim=16,
                         intermediate=96, vocab=80)


def incremental_matches_full(model):
    toks = ql_inputs.prompt_tokens(6, SMALL.vocab, seed=3)
    cache = decode.KVCache(SMALL, 1, len(toks))
    inc = np.array([decode.decode_step(model, cache, [t], [i])[0] for i, t in enumerate(toks)])
    return np.allclose(inc, decode.forward_full(model, toks), rtol=1e-10, atol=1e-12)


def test_causal_off_by_one_is_caught(monkeypatch):
    model = decode.Q4Model(SMALL, ql_inputs.weights(SMALL, seed=7))
    assert incremental_matches_full(model)
    real = ops.gqa_attention

    def drops_last_key(q, k, v, scale):   # attends to positions 0..p-1 only (when p > 0)
        if k.shape[1] > 1:
            return real(q, k[:, :-1], v[:, :-1], scale)
        return real(q, k, v, scale)
    monkeypatch.setattr(ops, "gqa_attention", drops_last_key)
    assert not incremental_matches_full(model)


def test_missing_qk_norm_is_caught(monkeypatch):
    # dropping the per-head norm in only one formulation breaks the incremental = full pin
    model = decode.Q4Model(SMALL, ql_inputs.weights(SMALL, seed=7))
    real = ops.rmsnorm
    calls = {"n": 0}

    def skip_head_norm(v, w, eps):
        if np.asarray(w).shape[-1] == SMALL.head_dim and np.asarray(v).ndim == 2 \
                and np.asarray(v).shape[0] in (SMALL.n_heads, SMALL.n_kv_heads):
            calls["n"] += 1
            return np.asarray(v, np.float64) * w
        return real(v, w, eps)
    monkeypatch.setattr(ops, "rmsnorm", skip_head_norm)
    assert not incremental_matches_full(model)
    assert calls["n"] > 0
