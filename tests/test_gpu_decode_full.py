"""The decode step at the full Qwen3-8B width against the oracle.

The 8B shape with two layers (hidden 4096, 32/8 heads of 128, SwiGLU 12288, the full 151,936
vocabulary and lm_head), in the configurations the benchmark times: batch 1 over a
2048-position pre-filled context (the stream GEMVs at batch 1, 8-warp attention) and batch 32
over mixed context lengths (the split-K batched GEMVs, in both tensor-core forms, and their
merge kernels). Weights are
drawn on the GPU (``ql_inputs.device_tensor_fn``) and packed there by ``ql_q4_0_pack_device``.
``test_device_codes_are_the_oracles`` first checks those codes, every byte of every matrix kind,
against the oracle's own quantisation (``oracle.q4_0.quantize``) of the same f32 draws copied to
the host; the step tests then hand the oracle those q4_0 codes and the same f16 contexts, and it
decodes in f64 with the lm_head taken in row chunks.

Every logit of every sequence is compared with the step tolerance
(``|got - want| <= 2e-2 + 1e-2 |want|``), and the greedy token must equal the oracle's
wherever the oracle's top-2 margin exceeds that tolerance. Two steps, the second fed the
oracle's tokens (teacher forcing).
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import decode

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu

CFG = ql_inputs.qwen3_8b_layers(2)


def host(t):
    return t.cpu().numpy()


def oracle_model(gm):
    """The oracle's model over the GPU model's own q4_0 codes and norm weights."""
    def q4(T):
        return host(T.scales).view(np.uint16), host(T.quants)
    layers = []
    for L in gm.layers:
        d = {n: host(L[n]) for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm")}
        d.update({n: q4(L[n]) for n in ("wqkv", "wo", "wgu", "wd")})
        layers.append(d)
    return decode.Q4Model.from_codes(CFG, layers, host(gm.final_norm), q4(gm.lm_head))


def test_device_codes_are_the_oracles():
    """Every byte the device quantiser wrote for the two layers and the full lm_head equals the
    oracle's quantisation of the same f32 draw: q4_0 packing must be bit-exact."""
    from oracle import q4_0 as oq
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    lib()
    fn = ql_inputs.device_tensor_fn(CFG, seed=0)
    gm = DeviceModel.from_layer_fn(CFG, fn, num_blocks=4, max_batch=1, max_blocks_per_seq=4)
    try:
        mats = [(li, n, gm.layers[li][n]) for li in range(CFG.n_layers) for n in ("wqkv", "wo", "wgu", "wd")]
        mats.append((None, "lm_head", gm.lm_head))
        for li, name, T in mats:
            w = fn(li, name)
            s_dev, q_dev = host(T.scales).view(np.uint16), host(T.quants)
            step = 8192
            for r0 in range(0, T.rows, step):
                s_ref, q_ref = oq.quantize(host(w[r0:r0 + step]))
                assert np.array_equal(s_dev[r0:r0 + step], s_ref), (li, name, r0)
                assert np.array_equal(q_dev[r0:r0 + step], q_ref), (li, name, r0)
            del w
    finally:
        gm.close()


@pytest.mark.parametrize("B,form", [(1, "mma_sync"), (32, "mma_sync"), (32, "tcgen05")])
def test_full_width_step_matches_oracle(B, form):
    ql = lib()
    prev = ql.ql_set_batched_gemv_form(ql.QL_BATCHED_TCGEN05 if form == "tcgen05" else ql.QL_BATCHED_MMA_SYNC)
    try:
        _full_width_step(B)
    finally:
        ql.ql_set_batched_gemv_form(prev)


def _full_width_step(B):
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    if B == 1:
        lens = np.array([2048], np.int64)
    else:
        lens = ql_inputs.batched_lengths(B, 16, 300, seed=7).astype(np.int64)
    steps = 2
    maxb = int((lens.max() + steps + 15) // 16)
    num_blocks = B * maxb
    gm = DeviceModel.from_layer_fn(CFG, ql_inputs.device_tensor_fn(CFG, seed=0), num_blocks=num_blocks,
                                   max_batch=B, max_blocks_per_seq=maxb)
    try:
        om = oracle_model(gm)
        embed = gm.embed   # f32 [vocab, hidden] on the device; rows gathered per step
        ids = ql_inputs.fragmented_block_ids(num_blocks, seed=5)
        bt = ids.reshape(B, maxb).copy()
        cache = decode.KVCache(CFG, B, maxb * 16)
        for b in range(B):
            k, v = ql_inputs.kv_context(CFG.n_layers, CFG.n_kv_heads, CFG.head_dim, int(lens[b]), seed=4, slot=b)
            gm.write_context(bt[b].tolist(), k, v)
            cache.preload(b, k, v)
        toks = ql_inputs.prompt_tokens(B, CFG.vocab, seed=1).astype(np.int64)
        tokens = dev(toks.astype(np.int32))
        positions = dev(lens.astype(np.int32))
        nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
        logits = torch.zeros((B, CFG.vocab), dtype=torch.float32, device="cuda")
        d_bt = dev(bt)   # referenced for the whole test: the step reads it through a raw pointer
        args = gm.step_args(tokens, positions, d_bt, nxt, logits=logits)
        pos = lens.copy()
        for step in range(steps):
            x0 = host(embed[torch.from_numpy(toks).cuda()]).astype(np.float64)
            hf = decode.decode_hidden(om, cache, x0, pos)
            want = decode.logits_by_rows(om.lm_head, hf)
            tokens.copy_(torch.from_numpy(toks.astype(np.int32)))
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            got = host(logits).astype(np.float64)
            g_tok = host(nxt)
            for b in range(B):
                ok = decode.logits_close(got[b], want[b])
                assert ok.all(), (f"step {step} seq {b}: {int((~ok).sum())} logits off, "
                                  f"max err {np.abs(got[b] - want[b]).max():.3e}")
                if decode.greedy_must_agree(want[b]):
                    assert int(g_tok[b]) == int(decode.greedy(want[b:b + 1])[0]), f"step {step} seq {b}"
            toks = decode.greedy(want).astype(np.int64)   # teacher forcing
            pos = pos + 1
            assert host(positions).tolist() == pos.tolist()
        gm.ql_check_device_error()
    finally:
        gm.close()
