"""Routed-expert (MoE) decode on the GPU against the oracle.

inferencelayer ``cuda_llm.rs``: the MoE branch of ``CudaQwen3::step`` (router logits from f32
router weights, top-k with renormalised weights, gate|up and down of the selected experts, the
weighted combine into the residual); the oracle is ``oracle.moe`` inside ``oracle.decode``.

The GPU picks the experts from f32 logits and the oracle from f64 ones: they agree unless two
logits at the k-th place are within rounding of each other, which these seeded weights do not
produce (the test asserts the oracle's gap at every step and layer). With the same experts the
block's arithmetic is the stream GEMV's (16-bit fixed-point activations, exact block sums) plus
an f32 router and softmax, so the logits are held to the step tolerance
``|got - want| <= 2e-2 + 1e-2 |want|``, and the greedy token to the oracle's where its top-2
margin exceeds it.
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import decode, moe, ops, q4_0 as oq

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu


def host(t):
    return t.cpu().numpy()


def router_gaps(om, cache_before, x0, positions):
    """The smallest gap, over layers, between the k-th and (k+1)-th router logit of the oracle
    for this step (recomputed on a copy of the cache)."""
    cfg = om.cfg
    import copy
    cache = copy.deepcopy(cache_before)
    gaps = []
    orig = moe.moe_ffn

    def spy(hn, router, w1, w2, c):
        lg = np.sort(np.asarray(router) @ np.asarray(hn))[::-1]
        gaps.append(lg[c.topk - 1] - lg[c.topk])
        return orig(hn, router, w1, w2, c)
    moe.moe_ffn = spy
    try:
        decode.decode_hidden(om, cache, x0, positions)
    finally:
        moe.moe_ffn = orig
    return min(gaps)


def test_tiny_moe_teacher_forced_16_steps():
    lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.TINY_MOE
    w = ql_inputs.weights(cfg, seed=0)
    gm = DeviceModel(cfg, w, num_blocks=16, max_batch=1, max_blocks_per_seq=4)
    try:
        om = decode.Q4Model(cfg, w)
        cache = decode.KVCache(cfg, 1, 64)
        bt = dev(ql_inputs.fragmented_block_ids(16, seed=5)[:4].reshape(1, 4).copy())
        tokens = torch.zeros(1, dtype=torch.int32, device="cuda")
        positions = torch.zeros(1, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, bt, nxt, logits=logits)
        tok = int(ql_inputs.prompt_tokens(1, cfg.vocab, seed=1)[0])
        for step in range(16):
            gap = router_gaps(om, cache, om.embed[[tok]], [step])
            assert gap > 1e-4, f"step {step}: the oracle's router has a near-tie ({gap:.2e})"
            want = decode.decode_step(om, cache, [tok], [step])[0]
            tokens.fill_(tok)
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            got = host(logits)[0].astype(np.float64)
            ok = decode.logits_close(got, want)
            assert ok.all(), f"step {step}: max err {np.abs(got - want).max():.3e}"
            if decode.greedy_must_agree(want):
                assert int(nxt.item()) == int(decode.greedy(want)), f"step {step}"
            tok = int(decode.greedy(want))
        assert int(host(positions)[0]) == 16
        gm.ql_check_device_error()
    finally:
        gm.close()


def test_moe_step_rejects_batches_and_the_persistent_kernel():
    ql = lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.TINY_MOE
    gm = DeviceModel(cfg, ql_inputs.weights(cfg, seed=0), num_blocks=16, max_batch=2, max_blocks_per_seq=4)
    try:
        with pytest.raises(ql.QLError) as e:
            gm.ql_model_set_option(ql.QL_OPT_STEP_KERNEL, ql.QL_STEP_PERSISTENT)
        assert e.value.status == ql.QL_EINVAL
        bt = dev(np.arange(8, dtype=np.int32).reshape(2, 4))
        t = torch.zeros(2, dtype=torch.int32, device="cuda")
        p = torch.zeros(2, dtype=torch.int32, device="cuda")
        n = torch.zeros(2, dtype=torch.int32, device="cuda")
        with pytest.raises(ql.QLError) as e:
            gm.ql_decode_step(gm.step_args(t, p, bt, n))
        assert e.value.status == ql.QL_EINVAL
    finally:
        gm.close()


def test_a3b_width_step_matches_oracle():
    """The Qwen3-30B-A3B width (two layers, 128 experts of 768, top-8, the full vocabulary) at
    batch 1 over a 2048-position pre-filled context, two teacher-forced steps. Weights are
    drawn and quantised on the GPU; the codes of three experts' rows of each expert matrix, and
    the attention matrices, are first checked byte for byte against the oracle's quantisation
    of the same draws, then the oracle decodes from those codes."""
    lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.qwen3_30b_a3b_layers(2)
    fn = ql_inputs.device_tensor_fn(cfg, seed=0)
    ctx, steps = 2048, 2
    maxb = (ctx + steps + 15) // 16
    gm = DeviceModel.from_layer_fn(cfg, fn, num_blocks=maxb, max_batch=1, max_blocks_per_seq=maxb)
    try:
        mi, hid = cfg.moe_inter, cfg.hidden
        for li in range(cfg.n_layers):
            for name, span in (("wqkv", None), ("wo", None), ("w1", 2 * mi), ("w2", hid)):
                T = gm.layers[li][name]
                wf = fn(li, name)
                chunks = [(0, T.rows)] if span is None else [(e * span, (e + 1) * span) for e in (0, 77, 127)]
                for r0, r1 in chunks:
                    s_ref, q_ref = oq.quantize(host(wf[r0:r1]))
                    assert np.array_equal(host(T.scales[r0:r1]).view(np.uint16), s_ref), (li, name, r0)
                    assert np.array_equal(host(T.quants[r0:r1]), q_ref), (li, name, r0)
                del wf
        layers = []
        for L in gm.layers:
            d = {n: host(L[n]) for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm", "router")}
            d.update({n: (host(L[n].scales).view(np.uint16), host(L[n].quants)) for n in ("wqkv", "wo", "w1", "w2")})
            layers.append(d)
        om = decode.Q4Model.from_codes(cfg, layers, host(gm.final_norm),
                                       (host(gm.lm_head.scales).view(np.uint16), host(gm.lm_head.quants)))
        bt = ql_inputs.fragmented_block_ids(maxb, seed=5).reshape(1, maxb).copy()
        cache = decode.KVCache(cfg, 1, maxb * 16)
        k, v = ql_inputs.kv_context(cfg.n_layers, cfg.n_kv_heads, cfg.head_dim, ctx, seed=4)
        gm.write_context(bt[0].tolist(), k, v)
        cache.preload(0, k, v)
        toks = ql_inputs.prompt_tokens(1, cfg.vocab, seed=1).astype(np.int64)
        tokens = dev(toks.astype(np.int32))
        positions = dev(np.array([ctx], np.int32))
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda")
        d_bt = dev(bt)
        args = gm.step_args(tokens, positions, d_bt, nxt, logits=logits)
        pos = np.array([ctx])
        for step in range(steps):
            x0 = host(gm.embed[torch.from_numpy(toks).cuda()]).astype(np.float64)
            gap = router_gaps(om, cache, x0, pos)
            assert gap > 1e-4, f"step {step}: the oracle's router has a near-tie ({gap:.2e})"
            hf = decode.decode_hidden(om, cache, x0, pos)
            want = decode.logits_by_rows(om.lm_head, hf)[0]
            tokens.copy_(torch.from_numpy(toks.astype(np.int32)))
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            got = host(logits)[0].astype(np.float64)
            ok = decode.logits_close(got, want)
            assert ok.all(), f"step {step}: {int((~ok).sum())} logits off, max err {np.abs(got - want).max():.3e}"
            if decode.greedy_must_agree(want):
                assert int(host(nxt)[0]) == int(decode.greedy(want[None, :])[0])
            toks = decode.greedy(want[None, :]).astype(np.int64)
            pos = pos + 1
        gm.ql_check_device_error()
    finally:
        gm.close()


def _run_steps(cfg, w, n_steps):
    """GPU logits and greedy tokens of n_steps teacher-forced decode steps (the oracle's greedy
    tokens fed back), with the oracle's logits, for the weights w."""
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    gm = DeviceModel(cfg, w, num_blocks=16, max_batch=1, max_blocks_per_seq=4)
    try:
        om = decode.Q4Model(cfg, w)
        cache = decode.KVCache(cfg, 1, 64)
        bt = dev(ql_inputs.fragmented_block_ids(16, seed=5)[:4].reshape(1, 4).copy())
        tokens = torch.zeros(1, dtype=torch.int32, device="cuda")
        positions = torch.zeros(1, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, bt, nxt, logits=logits)
        tok = int(ql_inputs.prompt_tokens(1, cfg.vocab, seed=1)[0])
        out = []
        for step in range(n_steps):
            gaps = []
            orig = moe.moe_ffn

            def spy(hn, router, w1, w2, c):
                lg = np.sort(np.asarray(router) @ np.asarray(hn))[::-1]
                gaps.append(lg[c.topk - 1] - lg[c.topk])
                return orig(hn, router, w1, w2, c)
            moe.moe_ffn = spy
            try:
                want = decode.decode_step(om, cache, [tok], [step])[0]
            finally:
                moe.moe_ffn = orig
            tokens.fill_(tok)
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            out.append((host(logits)[0].astype(np.float64), int(nxt.item()), want, gaps))
            tok = int(decode.greedy(want))
        gm.ql_check_device_error()
        return out
    finally:
        gm.close()


def _reversed_experts(cfg, w):
    """The same model with its experts in reverse order: exact router ties then break toward the
    other end of the original order."""
    import copy
    r = copy.deepcopy(w)
    E, inter, hid = cfg.num_experts, cfg.moe_inter, cfg.hidden
    for L in r["layers"]:
        L["router"] = L["router"][::-1].copy()
        L["w1"] = L["w1"].reshape(E, 2 * inter, hid)[::-1].reshape(E * 2 * inter, hid).copy()
        L["w2"] = L["w2"].reshape(E, hid, inter)[::-1].reshape(E * hid, inter).copy()
    return r


@pytest.mark.parametrize("form", ["zero_router", "three_equal_rows"])
def test_router_ties_take_the_lowest_index(form):
    """Exact ties between router logits ([IL] CudaQwen3::step's top-k; the reading in oracle.moe:
    the lower expert index first among equal values). An all-zero router makes every logit 0;
    equal router rows for experts 0, 1 and 2 make those three logits equal (bit for bit on the
    GPU too: each is the same dot product in the same order). The GPU must pick what the oracle
    picks: its logits within the step tolerance at every step. A near-tie that is not exact is
    still excluded (gap > 1e-4 unless exactly 0). Non-vacuity: the oracle of the same model with
    its experts reversed (ties then resolved toward the other end) differs from the oracle by
    more than the tolerance at some step."""
    import copy
    lib()
    cfg = ql_inputs.TINY_MOE
    w = copy.deepcopy(ql_inputs.weights(cfg, seed=0))
    for L in w["layers"]:
        if form == "zero_router":
            L["router"] = np.zeros_like(L["router"])
        else:
            r = L["router"].copy()
            r[1] = r[0]
            r[2] = r[0]
            L["router"] = r
    steps = 8
    res = _run_steps(cfg, w, steps)
    for step, (got, nxt, want, gaps) in enumerate(res):
        assert all(g == 0.0 or g > 1e-4 for g in gaps), f"step {step}: a near-tie that is not exact: {gaps}"
        ok = decode.logits_close(got, want)
        assert ok.all(), f"step {step}: max err {np.abs(got - want).max():.3e}"
        if decode.greedy_must_agree(want):
            assert nxt == int(decode.greedy(want)), f"step {step}"
    # non-vacuity: resolving the ties the other way changes the result beyond the tolerance
    om_r = decode.Q4Model(cfg, _reversed_experts(cfg, w))
    cache_r = decode.KVCache(cfg, 1, 64)
    tok = int(ql_inputs.prompt_tokens(1, cfg.vocab, seed=1)[0])
    differs = False
    for step in range(steps):
        want_r = decode.decode_step(om_r, cache_r, [tok], [step])[0]
        differs |= not decode.logits_close(want_r, res[step][2]).all()
        tok = int(decode.greedy(res[step][2]))
    assert differs, "reversing the experts left every step within the tolerance: the test would not see a wrong tie-break"
