"""The full Qwen3-8B shape in the benchmark's decode configurations: 36 layers, the full
151,936-row vocabulary, batch 1 (the tile stream GEMVs) and batch 32 (the split-K tensor-core
GEMVs with the RMSNorm folded into their merges), with the f16 and the q8_0 / q5_1 KV cache;
and the full Qwen3-30B-A3B routed-expert shape (48 layers) at batch 1.

The f64 oracle cannot hold 36 layers of these weights, so the element-by-element comparison
with it is made at two layers of the same width (test_gpu_decode_full.py). At the full depth the
step is checked through properties that hold at any size:
* the replayed graph gives the eager step's logits and tokens bit for bit;
* identical sequences within a batch give identical logits bit for bit (2 at batch 2, 32 at
  batch 32). Across batch sizes the o GEMV's grid changes (it leaves one SM per attention merge,
  batch x kv heads of them), so its tiles' partial sums are grouped differently. Batch 2 then
  agrees with batch 1 within the step's logit tolerance (|d| <= 2e-2 + 1e-2 |w|).
* every greedy token is the argmax of the logits the step wrote (the first index among equal
  maxima).
The weights are seeded device draws (as in bench.py); every slot holds the same synthetic
N(0, 1) context in its own blocks of a fragmented pool.
"""
import numpy as np
import pytest
import torch

import ql_inputs

from oracle import decode

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu

CFG = ql_inputs.QWEN3_8B
N_POS = 256


def _model(max_batch, cfg=CFG, quantised_cache=False):
    """A full-depth model whose every slot holds the same N_POS-position context (f16 pool, or
    the q8_0 / q5_1 records written by ql_kvq_write)."""
    import quantized_transformer_decode_ql_gb300 as ql
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    kvf = ql.QL_KV_Q8_0_Q5_1 if quantised_cache else ql.QL_KV_F16
    maxb = (N_POS + 40 + 15) // 16   # room for 40 more positions (a 32-token chunk)
    nb = max_batch * maxb
    gm = DeviceModel.from_layer_fn(cfg, ql_inputs.device_tensor_fn(cfg, seed=0), num_blocks=nb,
                                   max_batch=max_batch, max_blocks_per_seq=maxb, kv_format=kvf)
    bt = ql_inputs.fragmented_block_ids(nb, seed=5).reshape(max_batch, maxb).copy()
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    nblk = (N_POS + 15) // 16
    if quantised_cache:
        k = torch.randn((cfg.n_layers, N_POS, cfg.n_kv_heads, cfg.head_dim), generator=g, device="cuda")
        v = torch.randn((cfg.n_layers, N_POS, cfg.n_kv_heads, cfg.head_dim), generator=g, device="cuda")
        pos = torch.arange(N_POS, device="cuda")
        for b in range(max_batch):
            idx = torch.as_tensor(bt[b, :nblk], dtype=torch.long, device="cuda")
            slots = (idx[pos // 16] * 16 + pos % 16).contiguous()
            for li in range(cfg.n_layers):
                ql.ql_kvq_write(k[li].contiguous(), v[li].contiguous(), slots, cfg.n_kv_heads, cfg.head_dim,
                                gm.kvq_pool[li], gm.num_blocks)
        return gm, bt
    shape = (cfg.n_layers, nblk, cfg.n_kv_heads, 16, cfg.head_dim)
    k = torch.randn(shape, generator=g, device="cuda").half()
    v = torch.randn(shape, generator=g, device="cuda").half()
    for b in range(max_batch):
        idx = torch.as_tensor(bt[b, :nblk], dtype=torch.long, device="cuda")
        gm.k_pool[:, idx] = k
        gm.v_pool[:, idx] = v
    return gm, bt


def _step(gm, bt, B, token, graph=False):
    """One decode step of B slots (the first B rows of bt), all with `token` at position N_POS;
    returns (logits [B, vocab], next tokens [B])."""
    vocab = gm.cfg.vocab
    tokens = torch.full((B,), token, dtype=torch.int32, device="cuda")
    positions = torch.full((B,), N_POS, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    logits = torch.zeros((B, vocab), dtype=torch.float32, device="cuda")
    args = gm.step_args(tokens, positions, dev(bt[:B].copy()), nxt, logits=logits)
    if graph:
        s = torch.cuda.Stream()
        gm.ql_decode_graph_capture(args, s)
        positions.fill_(N_POS)
        tokens.fill_(token)
        with torch.cuda.stream(s):
            gm.ql_decode_graph_replay(B, 1, s)
        s.synchronize()
    else:
        gm.ql_decode_step(args)
    torch.cuda.synchronize()
    gm.ql_check_device_error()
    return logits.cpu().numpy().copy(), nxt.cpu().numpy().copy()


def _argmax_first(row):
    return int(np.flatnonzero(row == row.max())[0])


@pytest.mark.parametrize("case", ["b1", "b32", "b32_quantised_cache", "moe_b1"])
def test_full_depth_graph_equals_eager_and_identical_slots_agree(case):
    """Also the follow-on rows at full size: the q8_0 / q5_1 cache at batch 32, and the
    Qwen3-30B-A3B-shaped routed-expert model (48 layers, 128 experts, top-8) at batch 1."""
    lib()
    B = 32 if case.startswith("b32") else 1
    cfg = ql_inputs.QWEN3_30B_A3B if case == "moe_b1" else CFG
    gm, bt = _model(B, cfg, quantised_cache=case == "b32_quantised_cache")
    try:
        token = int(ql_inputs.prompt_tokens(1, cfg.vocab, seed=1)[0])
        le, te = _step(gm, bt, B, token)
        lg, tg = _step(gm, bt, B, token, graph=True)
        assert np.isfinite(le).all()
        assert np.array_equal(le, lg), "graph replay differs from the eager step"
        assert np.array_equal(te, tg)
        for b in range(B):
            assert np.array_equal(le[b], le[0]), f"slot {b} differs from slot 0 on identical inputs"
            assert int(te[b]) == _argmax_first(le[b]), f"slot {b}: the token is not the logits' argmax"
    finally:
        gm.close()


def test_full_depth_two_identical_slots_equal_batch_one():
    lib()
    gm, bt = _model(2)
    try:
        token = int(ql_inputs.prompt_tokens(1, CFG.vocab, seed=1)[0])
        l1, t1 = _step(gm, bt, 1, token)
        l2, t2 = _step(gm, bt, 2, token)
        assert np.array_equal(l2[1], l2[0]), "two identical slots differ"
        assert decode.logits_close(l2[0].astype(np.float64), l1[0].astype(np.float64)).all()
        assert int(t2[0]) == int(t2[1]) == _argmax_first(l2[0])
        assert int(t1[0]) == _argmax_first(l1[0])
        if decode.greedy_must_agree(l1[0].astype(np.float64)):
            assert int(t2[0]) == int(t1[0])
    finally:
        gm.close()


def test_full_depth_prefill_chunk_equals_sequential_decode():
    """[IL] runs a prompt as sequential decode (its module doc): one 32-token prefill chunk (the
    batch-32 split-K GEMVs, the chunk attention) must give the last token's logits of 32
    teacher-forced decode steps (the batch-1 stream GEMVs, the split attention) at the full
    depth. Both are held to the step tolerance tol(w) = 2e-2 + 1e-2 |w| against the exact result,
    so two GPU paths are compared at twice it (|a - b| <= |a - exact| + |exact - b|): logits and
    the appended K/V rows within 2 tol(w), the greedy tokens equal where the top-2 margin
    exceeds 2 tol(top)."""
    lib()
    gm, bt = _model(32)
    try:
        T = 32
        toks = ql_inputs.prompt_tokens(T, CFG.vocab, seed=2).astype(np.int32)
        row = bt[0].copy()
        # 32 decode steps of slot 0, one token each (teacher-forced)
        tokens = torch.zeros(1, dtype=torch.int32, device="cuda")
        positions = torch.full((1,), N_POS, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.zeros((1, CFG.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, dev(row.reshape(1, -1)), nxt, logits=logits)
        for t in range(T):
            tokens.fill_(int(toks[t]))
            gm.ql_decode_step(args)
        torch.cuda.synchronize()
        gm.ql_check_device_error()
        assert int(positions.item()) == N_POS + T
        want = logits.cpu().numpy()[0].astype(np.float64)
        nblk_new = (N_POS + T + 15) // 16
        idx = torch.as_tensor(row[N_POS // 16:nblk_new], dtype=torch.long, device="cuda")
        k_dec = gm.k_pool[:, idx].float().cpu().numpy()
        v_dec = gm.v_pool[:, idx].float().cpu().numpy()
        # the same 32 tokens as one prefill chunk from the same position
        position = torch.full((1,), N_POS, dtype=torch.int32, device="cuda")
        plog = torch.zeros(CFG.vocab, dtype=torch.float32, device="cuda")
        pnxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        gm.ql_prefill_chunk(dev(toks), position, dev(row), logits=plog, next_token=pnxt)
        torch.cuda.synchronize()
        gm.ql_check_device_error()
        assert int(position.item()) == N_POS + T
        got = plog.cpu().numpy().astype(np.float64)
        two_tol = 2 * (2e-2 + 1e-2 * np.abs(want))
        assert (np.abs(got - want) <= two_tol).all(), f"max err {np.abs(got - want).max():.3e}"
        top = _argmax_first(want)
        margin = want[top] - np.delete(want, top).max()
        if margin > 2 * (2e-2 + 1e-2 * abs(want[top])):
            assert int(pnxt.item()) == top
        k_pre = gm.k_pool[:, idx].float().cpu().numpy()
        v_pre = gm.v_pool[:, idx].float().cpu().numpy()
        lo = N_POS % 16   # the new rows: positions N_POS .. N_POS + T - 1 of these blocks
        sel = np.zeros((len(idx), 16), bool)
        for p in range(N_POS, N_POS + T):
            sel[p // 16 - N_POS // 16, p % 16] = True
        assert lo == 0
        for name, a, b in (("K", k_pre, k_dec), ("V", v_pre, v_dec)):
            d = np.abs(a - b)[:, sel.nonzero()[0], :, sel.nonzero()[1], :]
            w = np.abs(b)[:, sel.nonzero()[0], :, sel.nonzero()[1], :]
            assert (d <= 2 * (2e-2 + 1e-2 * w)).all(), f"{name} rows: max err {d.max():.3e}"
    finally:
        gm.close()
