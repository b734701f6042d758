"""Chunked prefill (ql_prefill_chunk) against the oracle.

inferencelayer ``cuda_llm.rs`` runs a prompt as sequential decode, and the oracle pins that
sequential decode equals the full causal recomputation (tests/test_oracle_decode.py). A chunk
of T prompt tokens through ``ql_prefill_chunk`` must therefore give, for its last token, the
logits of T oracle decode steps over the same tokens, and leave the same K and V rows in the
cache, so that decode steps after it continue as after sequential decode.

Tolerances: logits at the step tolerance ``2e-2 + 1e-2 |ref|`` (the chunk's GEMVs run in the
batched forms of the step, f16 activations from 3 tokens; above 32 tokens the tcgen05 GEMM with
the same arithmetic: (q - 8) d and the activations in f16, f32 products and sums); cached K / V
rows, which are f16 on both sides after f16 rounding of values the GPU computes in f32 from
f16-rounded activations, within ``2e-3 + 1e-2 |ref|``.
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import decode

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu


def host(t):
    return t.cpu().numpy()


def run_chunks(gm, om, cfg, prompt, chunks, bt_row, cache):
    """Prefill `prompt` in the given chunk sizes; after each chunk check the last token's logits
    and greedy token against the oracle's sequential decode. Returns (position, oracle token)."""
    position = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.zeros(cfg.vocab, dtype=torch.float32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_bt = dev(bt_row)
    p = 0
    for T in chunks:
        toks = prompt[p:p + T]
        for t in range(T):
            want = decode.decode_step(om, cache, [int(toks[t])], [p + t])[0]
        gm.ql_prefill_chunk(dev(toks.astype(np.int32)), position, d_bt, logits=logits, next_token=nxt)
        torch.cuda.synchronize()
        got = host(logits).astype(np.float64)
        ok = decode.logits_close(got, want)
        assert ok.all(), f"chunk at {p} (T={T}): max err {np.abs(got - want).max():.3e}"
        if decode.greedy_must_agree(want):
            assert int(nxt.item()) == int(decode.greedy(want))
        p += T
        assert int(position.item()) == p
    return p, int(decode.greedy(want))


@pytest.mark.parametrize("form", ["mma_sync", "tcgen05"])
def test_tiny_prefill_chunks_then_decode(form):
    ql = lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    prev = ql.ql_set_batched_gemv_form(ql.QL_BATCHED_TCGEN05 if form == "tcgen05" else ql.QL_BATCHED_MMA_SYNC)
    cfg = ql_inputs.TINY
    w = ql_inputs.weights(cfg, seed=0)
    gm = DeviceModel(cfg, w, num_blocks=16, max_batch=16, max_blocks_per_seq=8)
    try:
        om = decode.Q4Model(cfg, w)
        cache = decode.KVCache(cfg, 1, 128)
        prompt = ql_inputs.prompt_tokens(43, cfg.vocab, seed=1)
        bt_row = ql_inputs.fragmented_block_ids(16, seed=5)[:8].copy()
        p, tok = run_chunks(gm, om, cfg, prompt, [16, 16, 8, 2, 1], bt_row, cache)
        # the cache rows the chunks appended equal the oracle's (f16 on both sides)
        for li in range(cfg.n_layers):
            for pos in range(p):
                blk, slot = int(bt_row[pos // 16]), pos % 16
                gk = host(gm.k_pool[li, blk, :, slot]).astype(np.float64)
                gv = host(gm.v_pool[li, blk, :, slot]).astype(np.float64)
                wk, wv = cache.k[0, li, :, pos], cache.v[0, li, :, pos]
                assert np.all(np.abs(gk - wk) <= 2e-3 + 1e-2 * np.abs(wk)), (li, pos)
                assert np.all(np.abs(gv - wv) <= 2e-3 + 1e-2 * np.abs(wv)), (li, pos)
        # decode continues from the prefilled cache
        tokens = dev(np.array([tok], np.int32))
        positions = dev(np.array([p], np.int32))
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, dev(bt_row.reshape(1, -1)), nxt, logits=logits)
        for step in range(6):
            want = decode.decode_step(om, cache, [tok], [p + step])[0]
            tokens.fill_(tok)
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            got = host(logits)[0].astype(np.float64)
            assert decode.logits_close(got, want).all(), f"decode step {step}"
            tok = int(decode.greedy(want))
        gm.ql_check_device_error()
    finally:
        gm.close()
        ql.ql_set_batched_gemv_form(prev)


def test_tiny_prefill_gemm_chunks_then_decode():
    """Chunks above 32 tokens (the tcgen05 GEMM) mixed with smaller ones (the GEMVs): each
    chunk's last-token logits and the appended cache rows against the oracle's sequential
    decode, then decode steps from the prefilled cache.

    Cache rows: layer 0 at the module's bar ``2e-3 + 1e-2 |ref|``. A row of a later layer is
    projected from the previous layer's output, which already carries the rounding that bar
    allows for one row (f16 activations and cache, f32 sums), so its absolute term is counted
    twice: ``4e-3 + 1e-2 |ref|``. (The GEMM sums a row's products in one tensor-core
    accumulator, in another order than the GEMVs' windows: the same rounding, other bits.)"""
    ql = lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.TINY
    w = ql_inputs.weights(cfg, seed=0)
    gm = DeviceModel(cfg, w, num_blocks=16, max_batch=64, max_blocks_per_seq=8)
    try:
        om = decode.Q4Model(cfg, w)
        cache = decode.KVCache(cfg, 1, 128)
        prompt = ql_inputs.prompt_tokens(118, cfg.vocab, seed=2)
        bt_row = ql_inputs.fragmented_block_ids(16, seed=6)[:8].copy()
        p, tok = run_chunks(gm, om, cfg, prompt, [64, 33, 20, 1], bt_row, cache)
        worst = {}
        for li in range(cfg.n_layers):
            for pos in range(p):
                blk, slot = int(bt_row[pos // 16]), pos % 16
                for name, g, wref in (("k", gm.k_pool, cache.k), ("v", gm.v_pool, cache.v)):
                    got = host(g[li, blk, :, slot]).astype(np.float64)
                    want = wref[0, li, :, pos]
                    ex = np.abs(got - want) - ((2e-3 if li == 0 else 4e-3) + 1e-2 * np.abs(want))
                    i = np.unravel_index(np.argmax(ex), ex.shape)
                    if ex[i] > worst.get((name, li), (-1.0,))[0]:
                        worst[(name, li)] = (float(ex[i]), pos, float(got[i]), float(want[i]))
        assert all(v[0] <= 0 for v in worst.values()), "; ".join(
            f"{k[0]}{k[1]} {v[0]:+.2e} @{v[1]} {v[2]:.5f}/{v[3]:.5f}" for k, v in worst.items())
        tokens = dev(np.array([tok], np.int32))
        positions = dev(np.array([p], np.int32))
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, dev(bt_row.reshape(1, -1)), nxt, logits=logits)
        for step in range(4):
            want = decode.decode_step(om, cache, [tok], [p + step])[0]
            tokens.fill_(tok)
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            got = host(logits)[0].astype(np.float64)
            assert decode.logits_close(got, want).all(), f"decode step {step}"
            tok = int(decode.greedy(want))
        gm.ql_check_device_error()
    finally:
        gm.close()


def test_prefill_rejects_bad_chunks():
    ql = lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.TINY
    gm = DeviceModel(cfg, ql_inputs.weights(cfg, seed=0), num_blocks=8, max_batch=4, max_blocks_per_seq=4)
    try:
        pos = torch.zeros(1, dtype=torch.int32, device="cuda")
        bt = dev(np.arange(4, dtype=np.int32))
        for T in (5, 33):   # above max_batch
            with pytest.raises(ql.QLError) as e:
                gm.ql_prefill_chunk(torch.zeros(T, dtype=torch.int32, device="cuda"), pos, bt)
            assert e.value.status == ql.QL_EINVAL
    finally:
        gm.close()
    gb = DeviceModel(cfg, ql_inputs.weights(cfg, seed=0), num_blocks=32, max_batch=300, max_blocks_per_seq=32)
    try:   # above 256 tokens
        with pytest.raises(ql.QLError) as e:
            gb.ql_prefill_chunk(torch.zeros(257, dtype=torch.int32, device="cuda"),
                                torch.zeros(1, dtype=torch.int32, device="cuda"), dev(np.arange(32, dtype=np.int32)))
        assert e.value.status == ql.QL_EINVAL
    finally:
        gb.close()
    gq = DeviceModel(cfg, ql_inputs.weights(cfg, seed=0), num_blocks=8, max_batch=4, max_blocks_per_seq=4,
                     kv_format=ql.QL_KV_Q8_0_Q5_1)
    try:
        with pytest.raises(ql.QLError) as e:
            gq.ql_prefill_chunk(torch.zeros(2, dtype=torch.int32, device="cuda"),
                                torch.zeros(1, dtype=torch.int32, device="cuda"), dev(np.arange(4, dtype=np.int32)))
        assert e.value.status == ql.QL_EINVAL
    finally:
        gq.close()


@pytest.mark.parametrize("T", [32, 128])
def test_full_width_prefill_chunk_after_context(T):
    """The 8B width (two layers, full vocabulary): a 2048-position pre-filled context, then one
    chunk of T tokens (32: the batched GEMVs; 128: the tcgen05 GEMM); the chunk's last-token
    logits against T oracle decode steps."""
    lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    from test_gpu_decode_full import oracle_model
    cfg = ql_inputs.qwen3_8b_layers(2)
    ctx = 2048
    maxb = (ctx + T + 15) // 16
    gm = DeviceModel.from_layer_fn(cfg, ql_inputs.device_tensor_fn(cfg, seed=0), num_blocks=maxb, max_batch=T,
                                   max_blocks_per_seq=maxb)
    try:
        om = oracle_model(gm)
        bt_row = ql_inputs.fragmented_block_ids(maxb, seed=5).copy()
        k, v = ql_inputs.kv_context(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim, ctx, seed=4)
        gm.write_context(bt_row.tolist(), k, v)
        cache = decode.KVCache(cfg, 1, maxb * 16)
        cache.preload(0, k, v)
        prompt = ql_inputs.prompt_tokens(T, cfg.vocab, seed=1)
        embed = gm.embed
        for t in range(T):
            x0 = host(embed[torch.tensor([int(prompt[t])], device="cuda")]).astype(np.float64)
            hf = decode.decode_hidden(om, cache, x0, [ctx + t])
        want = decode.logits_by_rows(om.lm_head, hf)[0]
        position = dev(np.array([ctx], np.int32))
        logits = torch.zeros(cfg.vocab, dtype=torch.float32, device="cuda")
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        gm.ql_prefill_chunk(dev(prompt.astype(np.int32)), position, dev(bt_row), logits=logits, next_token=nxt)
        torch.cuda.synchronize()
        got = host(logits).astype(np.float64)
        ok = decode.logits_close(got, want)
        assert ok.all(), f"{int((~ok).sum())} logits off, max err {np.abs(got - want).max():.3e}"
        if decode.greedy_must_agree(want):
            assert int(nxt.item()) == int(decode.greedy(want[None, :])[0])
        assert int(position.item()) == ctx + T
        gm.ql_check_device_error()
    finally:
        gm.close()
