"""Pins of the oracle's decode step (no GPU).

* incremental decode over a KV cache equals full recomputation in matrix form (the pages run
  prefill as sequential decode, inferencelayer ``cuda_llm.rs`` module doc);
* a batch of identical sequences equals batch 1;
* the greedy tie rule and the top-2 margin agreement rule;
* the block allocator rule (ferrum-kernels ``cuda_decode.rs`` ``alloc_block``).
"""
import numpy as np
import pytest

import ql_inputs
from oracle import decode, ops
from oracle.blockpool import BlockPool, PoolExhausted

SMALL = ql_inputs.Config(hidden=64, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=16,
                         intermediate=96, vocab=80)


@pytest.fixture(scope="module")
def small_model():
    return decode.Q4Model(SMALL, ql_inputs.weights(SMALL, seed=7))


def run_incremental(model, tokens, ctx=None):
    cfg = model.cfg
    n0 = 0 if ctx is None else ctx[0].shape[2]
    cache = decode.KVCache(cfg, 1, n0 + len(tokens))
    if ctx is not None:
        cache.preload(0, *ctx)
    out = []
    for i, t in enumerate(tokens):
        out.append(decode.decode_step(model, cache, [t], [n0 + i])[0])
    return np.array(out), cache


def test_incremental_equals_full_recompute(small_model):
    toks = ql_inputs.prompt_tokens(12, SMALL.vocab, seed=3)
    inc, _ = run_incremental(small_model, toks)
    full = decode.forward_full(small_model, toks)
    np.testing.assert_allclose(inc, full, rtol=1e-10, atol=1e-12)


def test_incremental_equals_full_with_prefilled_context(small_model):
    ctx = ql_inputs.kv_context(SMALL.n_layers, SMALL.n_kv_heads, SMALL.head_dim, 21, seed=4)
    toks = ql_inputs.prompt_tokens(5, SMALL.vocab, seed=8)
    inc, _ = run_incremental(small_model, toks, ctx)
    full = decode.forward_full(small_model, toks, *ctx)
    np.testing.assert_allclose(inc, full, rtol=1e-10, atol=1e-12)


def test_context_changes_the_result(small_model):
    # non-vacuity: the pre-filled context is actually attended to
    toks = ql_inputs.prompt_tokens(2, SMALL.vocab, seed=8)
    ctx = ql_inputs.kv_context(SMALL.n_layers, SMALL.n_kv_heads, SMALL.head_dim, 7, seed=4)
    a = decode.forward_full(small_model, toks, *ctx)
    b = decode.forward_full(small_model, toks)
    assert np.max(np.abs(a - b)) > 1e-3


def test_identical_batch_equals_batch_one(small_model):
    toks = ql_inputs.prompt_tokens(4, SMALL.vocab, seed=5)
    single, _ = run_incremental(small_model, toks)
    B = 3
    cache = decode.KVCache(SMALL, B, len(toks))
    for i, t in enumerate(toks):
        lg = decode.decode_step(small_model, cache, [t] * B, [i] * B)
        for b in range(B):
            np.testing.assert_allclose(lg[b], single[i], rtol=1e-12, atol=1e-13)


def test_slots_are_independent(small_model):
    # two different sequences decoded together equal each decoded alone
    ta = ql_inputs.prompt_tokens(3, SMALL.vocab, seed=11)
    tb = ql_inputs.prompt_tokens(3, SMALL.vocab, seed=12)
    la, _ = run_incremental(small_model, ta)
    lb, _ = run_incremental(small_model, tb)
    cache = decode.KVCache(SMALL, 2, 3)
    for i in range(3):
        lg = decode.decode_step(small_model, cache, [ta[i], tb[i]], [i, i])
        np.testing.assert_allclose(lg[0], la[i], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lg[1], lb[i], rtol=1e-12, atol=1e-13)


def test_cache_holds_f16_keys_at_their_positions(small_model):
    toks = ql_inputs.prompt_tokens(3, SMALL.vocab, seed=13)
    _, cache = run_incremental(small_model, toks)
    k = cache.k[0, 0, :, :3]
    assert np.array_equal(k, k.astype(np.float16).astype(np.float64))
    # position 0's key is rope(rms(k) * k_norm, 0) = rms(k) * k_norm: unit-ish rms per head
    assert np.all(np.abs(k) < 10)


def test_greedy_rules():
    assert decode.greedy(np.array([[0.0, 2.0, 2.0]])).tolist() == [1]
    assert decode.greedy_must_agree(np.array([1.0, 0.5, 0.2]))
    assert not decode.greedy_must_agree(np.array([19.9, 19.9 - 0.0018, 3.0]))
    tol = decode.agreement_tolerance(19.9)
    assert abs(tol - (0.02 + 0.199)) < 1e-12
    ok = decode.logits_close(np.array([1.0, 10.0]), np.array([1.025, 10.11]))
    assert ok.tolist() == [True, True]
    assert decode.logits_close(np.array([0.0]), np.array([0.05])).tolist() == [False]


def test_block_pool_rule():
    p = BlockPool(3)
    assert [p.alloc(), p.alloc()] == [0, 1]
    p.release([0, 1])
    assert p.alloc() == 1          # last freed, first reused
    assert p.alloc() == 0
    assert p.alloc() == 2          # then the bump pointer
    with pytest.raises(PoolExhausted):
        p.alloc()
    assert p.in_use() == 3


def test_hidden_and_chunked_head_equal_the_step():
    """decode_step = lm_head x decode_hidden, and the lm_head taken in row chunks gives the
    same logits (each is the same dot product); a model rebuilt from its own codes
    (Q4Model.from_codes) decodes identically."""
    cfg = ql_inputs.TINY
    w = ql_inputs.weights(cfg, seed=0)
    m = decode.Q4Model(cfg, w)
    toks = ql_inputs.prompt_tokens(3, cfg.vocab, seed=9)
    c1, c2 = decode.KVCache(cfg, 3, 8), decode.KVCache(cfg, 3, 8)
    want = decode.decode_step(m, c1, toks, [0, 0, 0])
    m2 = decode.Q4Model.from_codes(cfg, [{k: L[k] for k in L} for L in m.layers], m.final_norm, m.lm_head)
    hf = decode.decode_hidden(m2, c2, m.embed[toks], [0, 0, 0])
    got = decode.logits_by_rows(m2.lm_head, hf, rows_per_chunk=100)
    assert np.array_equal(c1.k, c2.k) and np.array_equal(c1.v, c2.v)
    assert np.allclose(got, want, rtol=0, atol=1e-12)
