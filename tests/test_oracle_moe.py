"""Pins of the oracle's routed-expert (MoE) block (no GPU).

inferencelayer ``cuda_llm.rs``: router logits from f32 router weights, a top-k of the experts
with weights (``norm_topk``), per expert ``silu(gate) * up`` (expert e's gate|up rows
``[e 2mi, e 2mi + mi)`` and ``[e 2mi + mi, (e + 1) 2mi)`` of one q4_0 matrix) and the down
projection (rows ``[e hidden, (e + 1) hidden)``), combined by the weights.
"""
import math

import numpy as np
import pytest

import ql_inputs
from oracle import decode, moe, ops, q4_0 as oq


def test_route_hand_derived():
    # probabilities proportional to 1, 2, 4, 4, 1 (sum 12)
    logits = np.log([1.0, 2.0, 4.0, 4.0, 1.0])
    idx, w = moe.route(logits, 2, norm_topk=True)
    assert idx.tolist() == [2, 3]                  # equal probabilities: the lower index first
    assert np.allclose(w, [0.5, 0.5], rtol=0, atol=1e-15)
    idx, w = moe.route(logits, 3, norm_topk=True)
    assert idx.tolist() == [2, 3, 1] and np.allclose(w, [0.4, 0.4, 0.2], rtol=0, atol=1e-15)
    idx, w = moe.route(logits, 3, norm_topk=False)
    assert np.allclose(w, [4 / 12, 4 / 12, 2 / 12], rtol=0, atol=1e-15)


def test_route_invariances():
    rng = np.random.default_rng(0)
    logits = rng.standard_normal(128)
    idx, w = moe.route(logits, 8)
    idx2, w2 = moe.route(logits + 3.25, 8)          # softmax ignores a common shift
    assert np.array_equal(idx, idx2) and np.allclose(w, w2, rtol=1e-13, atol=0)
    assert abs(w.sum() - 1.0) < 1e-14 and np.all(np.diff(w) <= 0)
    assert np.array_equal(idx, np.argsort(-logits, kind="stable")[:8])   # the k largest logits
    full, wf = moe.route(logits, 128, norm_topk=False)
    assert np.allclose(wf, np.sort(ops.softmax(logits))[::-1], rtol=1e-14, atol=0)


def dense_ffn(hn, wg, wu, wd):
    """The dense SwiGLU block written out: wd (silu(wg hn) * (wu hn))."""
    g = wg @ hn
    u = wu @ hn
    return wd @ (g / (1.0 + np.exp(-g)) * u)


def test_identical_experts_give_the_dense_block():
    rng = np.random.default_rng(1)
    E, hidden, mi = 6, 64, 32
    cfg = ql_inputs.Config(hidden=hidden, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=64, intermediate=0,
                           vocab=8, num_experts=E, topk=3, moe_inter=mi)
    one_gu = (rng.standard_normal((2 * mi, hidden)) * 0.1).astype(np.float32)
    one_d = (rng.standard_normal((hidden, mi)) * 0.1).astype(np.float32)
    w1 = oq.quantize(np.tile(one_gu, (E, 1)))
    w2 = oq.quantize(np.tile(one_d, (E, 1)))
    router = rng.standard_normal((E, hidden))
    hn = rng.standard_normal(hidden)
    out, idx, w = moe.moe_ffn(hn, router, w1, w2, cfg)
    gu = oq.dequantize(*oq.quantize(one_gu))
    dn = oq.dequantize(*oq.quantize(one_d))
    ref = dense_ffn(hn, gu[:mi], gu[mi:], dn)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_single_route_selects_the_experts_own_rows():
    """A router that strongly prefers expert 2 of 4 (k = 1): the block equals the dense block
    made of rows [2 2mi, 2 2mi + mi) (gate), the next mi (up) and down rows [2 hidden, 3 hidden)."""
    rng = np.random.default_rng(2)
    E, hidden, mi = 4, 64, 32
    cfg = ql_inputs.Config(hidden=hidden, n_layers=1, n_heads=1, n_kv_heads=1, head_dim=64, intermediate=0,
                           vocab=8, num_experts=E, topk=1, moe_inter=mi)
    w1f = (rng.standard_normal((E * 2 * mi, hidden)) * 0.1).astype(np.float32)
    w2f = (rng.standard_normal((E * hidden, mi)) * 0.1).astype(np.float32)
    w1, w2 = oq.quantize(w1f), oq.quantize(w2f)
    hn = rng.standard_normal(hidden)
    router = np.zeros((E, hidden))
    router[2] = hn * 10.0                          # logit of expert 2 >> the others (0)
    out, idx, w = moe.moe_ffn(hn, router, w1, w2, cfg)
    assert idx.tolist() == [2] and w.tolist() == [1.0]
    W1, W2 = oq.dequantize(*w1), oq.dequantize(*w2)
    ref = dense_ffn(hn, W1[4 * mi:5 * mi], W1[5 * mi:6 * mi], W2[2 * hidden:3 * hidden])
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_moe_decode_incremental_equals_full_recomputation():
    cfg = ql_inputs.TINY_MOE
    w = ql_inputs.weights(cfg, seed=0)
    m = decode.Q4Model(cfg, w)
    toks = ql_inputs.prompt_tokens(8, cfg.vocab, seed=1)
    full = decode.forward_full(m, toks)
    cache = decode.KVCache(cfg, 1, 16)
    for p, t in enumerate(toks):
        step = decode.decode_step(m, cache, [int(t)], [p])[0]
        assert np.allclose(step, full[p], rtol=0, atol=1e-10)


def test_moe_routing_varies_and_matters():
    """Non-vacuity: different positions pick different experts, and perturbing one selected
    expert's weights changes the block's output."""
    cfg = ql_inputs.TINY_MOE
    w = ql_inputs.weights(cfg, seed=0)
    m = decode.Q4Model(cfg, w)
    L = m.layers[0]
    rng = np.random.default_rng(3)
    picks = set()
    for _ in range(6):
        hn = rng.standard_normal(cfg.hidden)
        _, idx, _ = moe.moe_ffn(hn, L["router"], L["w1"], L["w2"], cfg)
        picks.add(tuple(idx.tolist()))
    assert len(picks) > 1
    hn = rng.standard_normal(cfg.hidden)
    out, idx, _ = moe.moe_ffn(hn, L["router"], L["w1"], L["w2"], cfg)
    s, q = L["w2"]
    s2 = s.copy()
    e = int(idx[0])
    s2[e * cfg.hidden:(e + 1) * cfg.hidden] = (s[e * cfg.hidden:(e + 1) * cfg.hidden].view(np.float16) * 2).view(np.uint16)
    out2, _, _ = moe.moe_ffn(hn, L["router"], L["w1"], (s2, q), cfg)
    assert not np.allclose(out, out2)
