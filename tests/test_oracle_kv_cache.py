"""Pins of the oracle's quantised KV cache (no GPU).

memra-engine ``qwen4exp_gpu.rs``, the Q8Q5 quantised-cache store: a K row is kept as its q8_0
row and a V row as its q5_1 row (``oracle.kvq``); the decode then attends over the decoded
values. ``KVCache(kv="q8_0/q5_1")`` stores every row that way; the f16 cache stays the default.
"""
import numpy as np

import ql_inputs
from oracle import decode, kvq


def exact_rows():
    """K rows in q8_0's grid (codes times a power-of-two scale whose block max is 127 steps)
    and V rows in q5_1's grid (minimum -1, step 1/8, codes 0..31 with both ends used)."""
    rng = np.random.default_rng(3)
    k = rng.integers(-127, 128, size=(2, 4, 128)).astype(np.float64)
    k[..., ::32] = 127.0                                   # every block reaches +127
    k *= 2.0 ** -5
    c = rng.integers(0, 32, size=(2, 4, 128)).astype(np.float64)
    c[..., ::32] = 0.0
    c[..., 1::32] = 31.0
    v = -1.0 + c * 0.125
    return k, v


def test_stored_is_identity_on_the_formats_grid():
    cfg = ql_inputs.QWEN3_8B
    cache = decode.KVCache(cfg, 1, 4, kv=decode.KV_Q8_Q5)
    k, v = exact_rows()
    kd, vd = cache.stored(k, v)
    assert np.array_equal(kd, k) and np.array_equal(vd, v)


def test_stored_rows_within_the_formats_error():
    cfg = ql_inputs.QWEN3_8B
    cache = decode.KVCache(cfg, 1, 4, kv=decode.KV_Q8_Q5)
    rng = np.random.default_rng(4)
    k = rng.standard_normal((8, 128))
    v = rng.standard_normal((8, 128))
    kd, vd = cache.stored(k, v)
    kb = k.reshape(8, 4, 32)
    vb = v.reshape(8, 4, 32)
    dk = np.abs(kb).max(axis=2, keepdims=True) / 127
    dv = (vb.max(axis=2, keepdims=True) - vb.min(axis=2, keepdims=True)) / 31
    # half a step, plus the f16 rounding of the scale (and of the minimum) applied to the codes
    assert np.all(np.abs(kd.reshape(8, 4, 32) - kb) <= dk * (0.5 + 127 * 2.0 ** -11) + 1e-6)
    assert np.all(np.abs(vd.reshape(8, 4, 32) - vb) <= dv * (0.5 + 31 * 2.0 ** -11) + np.abs(vb).max() * 2.0 ** -10)
    # the f16 cache keeps f16 values
    f = decode.KVCache(cfg, 1, 4)
    kf, vf = f.stored(k, v)
    assert np.array_equal(kf, k.astype(np.float16).astype(np.float64))


def test_decode_over_the_quantised_cache():
    """The quantised cache changes the decode (its rows are really quantised) and stays near the
    f16 cache's decode: logits within 15% of their largest magnitude over 6 steps of the tiny
    model (q5_1 values keep about 5 bits per 32-element block, so a few per cent is expected)."""
    cfg = ql_inputs.TINY
    w = ql_inputs.weights(cfg, seed=0)
    m = decode.Q4Model(cfg, w)
    cq = decode.KVCache(cfg, 1, 16, kv=decode.KV_Q8_Q5)
    cf = decode.KVCache(cfg, 1, 16)
    toks = ql_inputs.prompt_tokens(6, cfg.vocab, seed=1)
    differ = False
    for p, t in enumerate(toks):
        lq = decode.decode_step(m, cq, [int(t)], [p])
        lf = decode.decode_step(m, cf, [int(t)], [p])
        assert np.abs(lq - lf).max() < 0.15 * np.abs(lf).max()
        differ = differ or not np.array_equal(lq, lf)
    assert differ
    # every stored K row is a decoded q8_0 row of some f32 row: re-quantising gives it back
    rows = cq.k[0, :, :, :6].reshape(-1, cfg.head_dim).astype(np.float32)
    again = kvq.dequantize_q8_0(kvq.quantize_q8_0(rows), cfg.head_dim)
    assert np.array_equal(again.astype(np.float64), rows.astype(np.float64))


def test_quantised_cache_amplifies_input_rounding():
    """Why the GPU's quantised-cache decode is held to three times the step tolerance: the
    codes are decided from the K and V rows, so a relative change of 1e-3 in those rows (the
    rounding level of a GEMV with f16 activations) flips codes at rounding boundaries, and each
    flip moves a value by a whole step. Measured here on the oracle alone (tiny model, batch 3,
    20 teacher-forced steps): the f16 cache's logits move by well under the step tolerance
    (2e-2 + 1e-2 |ref|), the quantised cache's by more than it, and by less than three times it."""
    cfg = ql_inputs.TINY
    w = ql_inputs.weights(cfg, seed=0)
    m = decode.Q4Model(cfg, w)

    class Perturbed(decode.KVCache):
        def __init__(self, *a, **k):
            super().__init__(*a, **k)
            self.rng = np.random.default_rng(0)

        def stored(self, k, v):
            k = k * (1 + 1e-3 * self.rng.standard_normal(np.shape(k)))
            v = v * (1 + 1e-3 * self.rng.standard_normal(np.shape(v)))
            return super().stored(k, v)

    worst = {}
    for kv in (decode.KV_F16, decode.KV_Q8_Q5):
        c0 = decode.KVCache(cfg, 3, 32, kv=kv)
        c1 = Perturbed(cfg, 3, 32, kv=kv)
        toks = ql_inputs.prompt_tokens(3, cfg.vocab, seed=1).astype(np.int64)
        r = 0.0
        for step in range(20):
            a = decode.decode_step(m, c0, toks, [step] * 3)
            b = decode.decode_step(m, c1, toks, [step] * 3)
            r = max(r, float((np.abs(a - b) / (2e-2 + 1e-2 * np.abs(a))).max()))
            toks = decode.greedy(a).astype(np.int64)
        worst[kv] = r
    assert worst[decode.KV_F16] < 0.25
    assert 1.0 < worst[decode.KV_Q8_Q5] < 3.0
