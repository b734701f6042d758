"""The quantised KV pool on the GPU: keys q8_0, values q5_1 (memra-engine qwen4exp_gpu.rs, the
Q8Q5 quantised-cache store and its host twins host_quant_q8_row / host_quant_q5_row).

* ql_kvq_write: every byte it writes equals the oracle's codec (``oracle.kvq``) of the same f32
  rows, once the record layout documented in include/ql.h is undone by a NumPy restatement;
  slots it does not address keep their bytes.
* ql_paged_attn_decode_kvq: over records made on the host by the oracle's codec, against
  ``oracle.kvq.paged_attention_q8k_q5v`` on the same bytes. The decoded keys and values enter
  the MMAs rounded to f16 (relative 2^-12), the rest is the f16 attention's arithmetic, so the
  bar is the attention tests' ``|o - o_ref| <= 2e-3 + 1e-2 |o_ref|``.
* The decode step with the quantised cache (``kv_format = QL_KV_Q8_0_Q5_1``): its fused append
  quantises each new K and V row on the GPU; against the oracle's decode with
  ``KVCache(kv="q8_0/q5_1")`` (the tiny model, and the 8B width with a pre-filled context of
  host-quantised records). The GPU decides each code from its own K and V rows, which differ
  from the oracle's by the rounding of its GEMVs (about 1e-3 relative at batch 3-32, with f16
  activations); where the two straddle a rounding boundary the code differs by one, a whole step
  of the format. The oracle alone, given rows perturbed at that level, moves its logits by 1 to 3
  times the step tolerance (tests/test_oracle_kv_cache.py), so the bar here is three times the
  step tolerance, ``6e-2 + 3e-2 |ref|``, and the greedy token must match where the oracle's
  top-2 margin exceeds that.
"""
import math

import numpy as np
import pytest
import torch

import ql_inputs
from oracle import decode, kvq

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu

TOL_ABS, TOL_REL = 6e-2, 3e-2


def close_q(got, want):
    return np.abs(got - want) <= TOL_ABS + TOL_REL * np.abs(want)


def must_agree_q(want):
    top = np.sort(want)[-2:]
    return top[1] - top[0] > TOL_ABS + TOL_REL * abs(top[1])


def record_from_rows(kb, vb, hd):
    """Page-format bytes of 16 key rows (q8_0) and 16 value rows (q5_1) -> one record."""
    nb = hd // 32
    K = np.asarray(kb, np.uint8).reshape(16, nb, 34)
    V = np.asarray(vb, np.uint8).reshape(16, nb, 24)
    rec = np.zeros(29 * hd, np.uint8)
    rec[0:16 * hd] = K[:, :, 2:].reshape(-1)
    rec[16 * hd:24 * hd] = V[:, :, 8:].reshape(-1)
    rec[24 * hd:25 * hd] = K[:, :, :2].reshape(-1)
    rec[25 * hd:27 * hd] = V[:, :, 4:8].reshape(-1)
    rec[27 * hd:28 * hd] = V[:, :, 0:2].reshape(-1)
    rec[28 * hd:29 * hd] = V[:, :, 2:4].reshape(-1)
    return rec


def rows_from_record(rec, hd):
    """The inverse: one record -> page-format key rows [16, q8 bytes], value rows [16, q5 bytes]."""
    nb = hd // 32
    K = np.zeros((16, nb, 34), np.uint8)
    V = np.zeros((16, nb, 24), np.uint8)
    K[:, :, 2:] = rec[0:16 * hd].reshape(16, nb, 32)
    V[:, :, 8:] = rec[16 * hd:24 * hd].reshape(16, nb, 16)
    K[:, :, :2] = rec[24 * hd:25 * hd].reshape(16, nb, 2)
    V[:, :, 4:8] = rec[25 * hd:27 * hd].reshape(16, nb, 4)
    V[:, :, 0:2] = rec[27 * hd:28 * hd].reshape(16, nb, 2)
    V[:, :, 2:4] = rec[28 * hd:29 * hd].reshape(16, nb, 2)
    return K.reshape(16, -1), V.reshape(16, -1)


def test_record_bytes():
    ql = lib()
    assert ql.ql_kvq_record_bytes(128) == 3712 and ql.ql_kvq_record_bytes(64) == 1856
    assert ql.ql_kvq_record_bytes(96) == 0


@pytest.mark.parametrize("hd", [64, 128])
def test_write_bytes_equal_the_oracle_codec(hd):
    ql = lib()
    n_kv, num_blocks = 3, 9
    rng = np.random.default_rng(hd)
    n = 40
    k = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    v = rng.standard_normal((n, n_kv, hd)).astype(np.float32)
    k[3] = 0.0                                             # all-zero rows: scale 0, codes 0
    v[3] = 0.0
    k[5, :, :32] = np.linspace(-2.5, 2.5, 32)               # exact half-steps after scaling
    v[6] = -1.0 + 0.125 * rng.integers(0, 32, size=(n_kv, hd))
    k[7] *= 1e-4                                            # a subnormal f16 scale
    slots = rng.permutation(num_blocks * 16)[:n].astype(np.int64)
    rec = 29 * hd
    pool = torch.full((num_blocks, n_kv, rec), 0xA5, dtype=torch.uint8, device="cuda")
    ql.ql_kvq_write(dev(k), dev(v), dev(slots), n_kv, hd, pool, num_blocks)
    torch.cuda.synchronize()
    ql.ql_check_device_error()
    got = pool.cpu().numpy()
    kref = kvq.quantize_q8_0(k.reshape(-1, hd)).reshape(n, n_kv, -1)
    vref = kvq.quantize_q5_1(v.reshape(-1, hd)).reshape(n, n_kv, -1)
    written = set()
    for i, sl in enumerate(slots):
        b, s = int(sl) // 16, int(sl) % 16
        written.add((b, s))
        for g in range(n_kv):
            K, V = rows_from_record(got[b, g], hd)
            assert np.array_equal(K[s], kref[i, g]), (i, g)
            assert np.array_equal(V[s], vref[i, g]), (i, g)
    # slots nobody wrote keep the sentinel in every field
    sentinel = np.full(29 * hd, 0xA5, np.uint8)
    K0, V0 = rows_from_record(sentinel, hd)
    for b in range(num_blocks):
        for s in range(16):
            if (b, s) in written:
                continue
            for g in range(n_kv):
                K, V = rows_from_record(got[b, g], hd)
                assert np.array_equal(K[s], K0[s]) and np.array_equal(V[s], V0[s])


def test_write_out_of_range_slot_is_recorded_not_written():
    ql = lib()
    hd, n_kv, num_blocks = 64, 2, 2
    k = torch.ones((2, n_kv, hd), dtype=torch.float32, device="cuda")
    slots = dev(np.array([5, 2 * 16 + 3], np.int64))        # the second is past the pool
    pool = torch.zeros((num_blocks, n_kv, 29 * hd), dtype=torch.uint8, device="cuda")
    ql.ql_kvq_write(k, k, slots, n_kv, hd, pool, num_blocks)
    with pytest.raises(ql.QLError) as e:
        ql.ql_check_device_error()
    assert e.value.status == ql.QL_EDEVICE
    assert int(pool[1].sum().item()) == 0                   # block 1 untouched


def host_records(case_k, case_v, hd):
    """f32 pools [num_blocks, n_kv, 16, hd] -> (records [num_blocks, n_kv, 29 hd], page bytes of
    the K and V rows [num_blocks, n_kv, 16, row bytes]) with the oracle's codec."""
    nbk, nkv = case_k.shape[:2]
    kb = kvq.quantize_q8_0(case_k.reshape(-1, hd)).reshape(nbk, nkv, 16, -1)
    vb = kvq.quantize_q5_1(case_v.reshape(-1, hd)).reshape(nbk, nkv, 16, -1)
    recs = np.zeros((nbk, nkv, 29 * hd), np.uint8)
    for b in range(nbk):
        for g in range(nkv):
            recs[b, g] = record_from_rows(kb[b, g], vb[b, g], hd)
    return recs, kb, vb


@pytest.mark.parametrize("n_heads,n_kv,hd", [(32, 8, 128), (4, 2, 64), (16, 2, 64), (8, 8, 128)])
def test_attention_over_quantised_pool(n_heads, n_kv, hd):
    ql = lib()
    lens = [1, 15, 16, 17, 33, 700, 2049]
    case = ql_inputs.attention_case(len(lens), n_heads, n_kv, hd, lens, seed=31)
    kf = case["k_pool"].astype(np.float32)
    vf = case["v_pool"].astype(np.float32)
    recs, kb, vb = host_records(kf, vf, hd)
    B, mb = len(lens), case["max_blocks"]
    out = torch.full((B, n_heads * hd), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.zeros(ql.ql_paged_attn_workspace_bytes(B, n_heads, n_kv, hd, 16, mb), dtype=torch.uint8, device="cuda")
    ql.ql_paged_attn_decode_kvq(dev(case["q"]), dev(recs), dev(case["block_tables"]), dev(case["lens"]), B, n_heads,
                                n_kv, hd, 16, mb, case["num_blocks"], 1.0 / math.sqrt(hd), out, ws)
    torch.cuda.synchronize()
    ql.ql_check_device_error()
    got = out.float().cpu().numpy().reshape(B, n_heads, hd).astype(np.float64)
    want = kvq.paged_attention_q8k_q5v(case["q"], kb, vb, hd, case["block_tables"], case["lens"], 1.0 / math.sqrt(hd))
    assert not np.isnan(got).any()
    err = np.abs(got - want)
    assert (err <= 2e-3 + 1e-2 * np.abs(want)).all(), f"max err {err.max():.3e}"


def test_persistent_step_rejects_the_quantised_cache():
    ql = lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.TINY
    gm = DeviceModel(cfg, ql_inputs.weights(cfg, seed=0), num_blocks=8, max_batch=1, max_blocks_per_seq=4,
                     kv_format=ql.QL_KV_Q8_0_Q5_1)
    try:
        with pytest.raises(ql.QLError) as e:
            gm.ql_model_set_option(ql.QL_OPT_STEP_KERNEL, ql.QL_STEP_PERSISTENT)
        assert e.value.status == ql.QL_EINVAL
    finally:
        gm.close()


@pytest.mark.parametrize("batch", [1, 3])
def test_tiny_decode_with_quantised_cache(batch):
    ql = lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.TINY
    w = ql_inputs.weights(cfg, seed=0)
    gm = DeviceModel(cfg, w, num_blocks=32, max_batch=4, max_blocks_per_seq=4, kv_format=ql.QL_KV_Q8_0_Q5_1)
    try:
        om = decode.Q4Model(cfg, w)
        cache = decode.KVCache(cfg, batch, 64, kv=decode.KV_Q8_Q5)
        bt = dev(ql_inputs.fragmented_block_ids(32, seed=5)[: batch * 4].reshape(batch, 4).copy())
        tokens = torch.zeros(batch, dtype=torch.int32, device="cuda")
        positions = torch.zeros(batch, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(batch, dtype=torch.int32, device="cuda")
        logits = torch.zeros((batch, cfg.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, bt, nxt, logits=logits)
        toks = ql_inputs.prompt_tokens(batch, cfg.vocab, seed=1).astype(np.int64)
        for step in range(20):
            want = decode.decode_step(om, cache, toks, [step] * batch)
            tokens.copy_(torch.from_numpy(toks.astype(np.int32)))
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            got = logits.cpu().numpy().astype(np.float64)
            for b in range(batch):
                ok = close_q(got[b], want[b])
                assert ok.all(), f"step {step} seq {b}: max err {np.abs(got[b] - want[b]).max():.3e}"
                if must_agree_q(want[b]):
                    assert int(nxt[b].item()) == int(decode.greedy(want[b:b + 1])[0])
            toks = decode.greedy(want).astype(np.int64)
        gm.ql_check_device_error()
    finally:
        gm.close()


@pytest.mark.parametrize("B", [1, 32])
def test_full_width_step_with_quantised_cache(B):
    """The 8B width (two layers, full vocabulary): a pre-filled context quantised on the host by
    the oracle's codec (records uploaded as bytes), then two teacher-forced steps whose appends
    the GPU quantises itself."""
    ql = lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    from test_gpu_decode_full import oracle_model, host
    cfg = ql_inputs.qwen3_8b_layers(2)
    lens = np.array([2048], np.int64) if B == 1 else ql_inputs.batched_lengths(B, 16, 300, seed=7).astype(np.int64)
    steps = 2
    maxb = int((lens.max() + steps + 15) // 16)
    num_blocks = B * maxb
    gm = DeviceModel.from_layer_fn(cfg, ql_inputs.device_tensor_fn(cfg, seed=0), num_blocks=num_blocks,
                                   max_batch=B, max_blocks_per_seq=maxb, kv_format=ql.QL_KV_Q8_0_Q5_1)
    try:
        om = oracle_model(gm)
        ids = ql_inputs.fragmented_block_ids(num_blocks, seed=5)
        bt = ids.reshape(B, maxb).copy()
        cache = decode.KVCache(cfg, B, maxb * 16, kv=decode.KV_Q8_Q5)
        hd, nkv = cfg.head_dim, cfg.n_kv_heads
        for b in range(B):
            L = int(lens[b])
            k, v = ql_inputs.kv_context(cfg.n_layers, nkv, hd, L, seed=4, slot=b)
            cache.preload(b, k, v)
            nblk = (L + 15) // 16
            pad = nblk * 16
            for li in range(cfg.n_layers):
                kf = np.zeros((nkv, pad, hd), np.float32)
                vf = np.zeros((nkv, pad, hd), np.float32)
                kf[:, :L] = k[li].astype(np.float32)
                vf[:, :L] = v[li].astype(np.float32)
                kf = kf.reshape(nkv, nblk, 16, hd).transpose(1, 0, 2, 3)
                vf = vf.reshape(nkv, nblk, 16, hd).transpose(1, 0, 2, 3)
                recs, _, _ = host_records(kf, vf, hd)
                idx = torch.as_tensor(bt[b, :nblk].astype(np.int64), device="cuda")
                gm.kvq_pool[li, idx] = dev(recs)
        toks = ql_inputs.prompt_tokens(B, cfg.vocab, seed=1).astype(np.int64)
        tokens = dev(toks.astype(np.int32))
        positions = dev(lens.astype(np.int32))
        nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
        logits = torch.zeros((B, cfg.vocab), dtype=torch.float32, device="cuda")
        d_bt = dev(bt)
        args = gm.step_args(tokens, positions, d_bt, nxt, logits=logits)
        pos = lens.copy()
        for step in range(steps):
            x0 = host(gm.embed[torch.from_numpy(toks).cuda()]).astype(np.float64)
            hf = decode.decode_hidden(om, cache, x0, pos)
            want = decode.logits_by_rows(om.lm_head, hf)
            tokens.copy_(torch.from_numpy(toks.astype(np.int32)))
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            got = host(logits).astype(np.float64)
            for b in range(B):
                ok = close_q(got[b], want[b])
                assert ok.all(), (f"step {step} seq {b}: {int((~ok).sum())} logits off, "
                                  f"max err {np.abs(got[b] - want[b]).max():.3e}")
                if must_agree_q(want[b]):
                    assert int(host(nxt)[b]) == int(decode.greedy(want[b:b + 1])[0]), f"step {step} seq {b}"
            toks = decode.greedy(want).astype(np.int64)
            pos = pos + 1
        gm.ql_check_device_error()
    finally:
        gm.close()
