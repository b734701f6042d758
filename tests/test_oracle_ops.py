"""Pins of the oracle's per-op definitions (no GPU): closed forms, invariants, brute force."""
import math

import numpy as np
import pytest

from oracle import ops, q4_0


def brute_gemv(w, x):
    rows, cols = len(w), len(w[0])
    out = []
    for b in range(len(x)):
        row = []
        for r in range(rows):
            acc = 0.0
            for k in range(cols):
                acc += float(w[r][k]) * float(x[b][k])
            row.append(acc)
        out.append(row)
    return np.array(out)


@pytest.mark.parametrize("rows,cols,batch", [(1, 32, 1), (3, 64, 2), (5, 96, 3)])
def test_gemv_matches_bruteforce_of_dequantised(rows, cols, batch):
    rng = np.random.default_rng(rows * 100 + cols)
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    x = rng.standard_normal((batch, cols)).astype(np.float16)
    s, q = q4_0.quantize(w)
    wd = q4_0.dequantize(s, q)
    # dequantise by hand, element by element, from the codes
    def weight(r, k):
        byte = int(q[r, k // 32, k % 16])
        code = (byte >> (4 * ((k % 32) // 16))) & 0xF
        d = float(s[r, k // 32:k // 32 + 1].view(np.float16)[0])
        return (code - 8) * d
    hand = [[weight(r, k) for k in range(cols)] for r in range(rows)]
    assert np.array_equal(wd, np.array(hand))
    np.testing.assert_allclose(ops.gemv(wd, x), brute_gemv(hand, x.astype(np.float64)),
                               rtol=1e-13, atol=1e-15)


def test_gemv_orientation():
    # y[b, r] = sum_k w[r, k] x[b, k]: a transposed operand would give a different shape/value
    w = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    x = np.array([[1.0, 0.0, -1.0]])
    assert ops.gemv(w, x).tolist() == [[-2.0, -2.0]]


def test_rmsnorm_constant_vector():
    # rms(c * 1) * w = c / sqrt(c^2 + eps) * w
    w = np.linspace(0.5, 1.5, 16)
    for c in (3.0, -0.25, 1e-3):
        v = np.full(16, c)
        np.testing.assert_allclose(ops.rmsnorm(v, w, 1e-6), c / math.sqrt(c * c + 1e-6) * w,
                                   rtol=1e-14)


def test_rmsnorm_bruteforce_and_invariants():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(64)
    w = 1 + 0.1 * rng.standard_normal(64)
    ms = sum(float(a) * float(a) for a in v) / 64
    want = [float(v[i]) / math.sqrt(ms + 1e-6) * float(w[i]) for i in range(64)]
    np.testing.assert_allclose(ops.rmsnorm(v, w, 1e-6), want, rtol=1e-13)
    # with eps = 0 the output has unit rms when w = 1, and is scale invariant
    u = ops.rmsnorm(v, np.ones(64), 0.0)
    assert abs(np.sqrt(np.mean(u * u)) - 1.0) < 1e-14
    np.testing.assert_allclose(ops.rmsnorm(5.0 * v, w, 0.0), ops.rmsnorm(v, w, 0.0), rtol=1e-14)
    # a batch of rows is normalised row by row
    vv = np.stack([v, 2 * v + 1])
    np.testing.assert_allclose(ops.rmsnorm(vv, w, 1e-6)[1], ops.rmsnorm(2 * v + 1, w, 1e-6))


def test_rope_identity_at_zero_and_norms():
    rng = np.random.default_rng(4)
    v = rng.standard_normal((3, 64))
    np.testing.assert_array_equal(ops.rope(v, 0, 1e6), v)
    for p in (1, 17, 2047, 32767):
        r = ops.rope(v, p, 1e6)
        n0 = v[:, :32] ** 2 + v[:, 32:] ** 2
        n1 = r[:, :32] ** 2 + r[:, 32:] ** 2
        np.testing.assert_allclose(n1, n0, rtol=1e-12)


def test_rope_pairs_split_half():
    # a one-hot at dim 0 rotates into dim hd/2 (NeoX pairing), never into dim 1
    hd, p, theta = 8, 3, 10000.0
    e0 = np.zeros(hd)
    e0[0] = 1.0
    r = ops.rope(e0, p, theta)
    assert abs(r[0] - math.cos(p)) < 1e-15 and abs(r[hd // 2] - math.sin(p)) < 1e-15
    assert np.all(np.delete(r, [0, hd // 2]) == 0.0)
    # dim i has frequency theta^(-2i/hd); one-hot at dim 1 at position p
    e1 = np.zeros(hd)
    e1[1] = 1.0
    r = ops.rope(e1, p, theta)
    ang = p * theta ** (-2.0 / hd)
    assert abs(r[1] - math.cos(ang)) < 1e-15 and abs(r[1 + hd // 2] - math.sin(ang)) < 1e-15
    # second half one-hot: (a, b) = (0, 1) -> (-sin, cos)
    e4 = np.zeros(hd)
    e4[hd // 2] = 1.0
    r = ops.rope(e4, p, theta)
    assert abs(r[0] + math.sin(p)) < 1e-15 and abs(r[hd // 2] - math.cos(p)) < 1e-15


def test_rope_composes():
    rng = np.random.default_rng(8)
    v = rng.standard_normal(128)
    np.testing.assert_allclose(ops.rope(ops.rope(v, 100, 1e6), 23, 1e6), ops.rope(v, 123, 1e6),
                               rtol=1e-12, atol=1e-12)


def test_silu_closed_forms():
    assert ops.silu(0.0) == 0.0
    z = np.linspace(-6, 6, 25)
    np.testing.assert_allclose(ops.silu(z) - ops.silu(-z), z, atol=1e-14)
    assert abs(ops.silu(40.0) - 40.0) < 1e-12 and abs(ops.silu(-40.0)) < 1e-15
    np.testing.assert_allclose(ops.silu(1.0), 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    np.testing.assert_allclose(ops.swiglu(np.array([1.0, -2.0]), np.array([3.0, 0.5])),
                               [3.0 / (1 + math.exp(-1.0)), -1.0 / (1 + math.exp(2.0))],
                               rtol=1e-15)


def brute_attention(q, k, v, scale):
    nh, hd = len(q), len(q[0])
    nkv, L = len(k), len(k[0])
    g = nh // nkv
    out = []
    for h in range(nh):
        kv = h // g
        s = [sum(q[h][d] * k[kv][t][d] for d in range(hd)) * scale for t in range(L)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        out.append([sum(e[t] / z * v[kv][t][d] for t in range(L)) for d in range(hd)])
    return np.array(out)


@pytest.mark.parametrize("L", [1, 15, 16, 17, 33])
def test_attention_bruteforce(L):
    rng = np.random.default_rng(L)
    q = rng.standard_normal((4, 8))
    k = rng.standard_normal((2, L, 8))
    v = rng.standard_normal((2, L, 8))
    got = ops.gqa_attention(q, k, v, 1 / math.sqrt(8))
    want = brute_attention(q.tolist(), k.tolist(), v.tolist(), 1 / math.sqrt(8))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def test_softmax_rows_sum_to_one_and_special_cases():
    rng = np.random.default_rng(1)
    s = rng.standard_normal((5, 37)) * 30
    np.testing.assert_allclose(ops.softmax(s).sum(axis=-1), 1.0, rtol=1e-14)
    # one key: the output is that key's value
    q = rng.standard_normal((4, 8))
    k = rng.standard_normal((2, 1, 8))
    v = rng.standard_normal((2, 1, 8))
    o = ops.gqa_attention(q, k, v, 0.3)
    np.testing.assert_array_equal(o[:2], np.repeat(v[0], 2, axis=0))
    np.testing.assert_array_equal(o[2:], np.repeat(v[1], 2, axis=0))
    # equal scores (zero query): the plain mean of the values
    o = ops.gqa_attention(np.zeros((4, 8)), rng.standard_normal((2, 9, 8)),
                          vv := rng.standard_normal((2, 9, 8)), 1.0)
    np.testing.assert_allclose(o[0], vv[0].mean(axis=0), rtol=1e-13)


def test_gqa_head_mapping():
    # kv head g holds the constant value g: query head h must read kv head h // (nh/nkv)
    nh, nkv, L, hd = 8, 2, 5, 4
    rng = np.random.default_rng(0)
    v = np.stack([np.full((L, hd), float(g)) for g in range(nkv)])
    o = ops.gqa_attention(rng.standard_normal((nh, hd)), rng.standard_normal((nkv, L, hd)), v, 1.0)
    np.testing.assert_allclose(o[:, 0], [0, 0, 0, 0, 1, 1, 1, 1], atol=1e-14)


def test_paged_equals_contiguous():
    rng = np.random.default_rng(9)
    L, nkv, hd, bs = 37, 2, 8, 16
    nblk = (L + bs - 1) // bs
    k = rng.standard_normal((nkv, L, hd)).astype(np.float16)
    v = rng.standard_normal((nkv, L, hd)).astype(np.float16)
    perm = rng.permutation(6)[:nblk]
    kp = np.zeros((6, nkv, bs, hd), np.float16)
    vp = np.zeros((6, nkv, bs, hd), np.float16)
    for p in range(L):
        kp[perm[p // bs], :, p % bs] = k[:, p]
        vp[perm[p // bs], :, p % bs] = v[:, p]
    np.testing.assert_array_equal(ops.gather_paged(kp, perm, L), k.astype(np.float64))
    q = rng.standard_normal((1, 4, hd))
    got = ops.paged_attention(q, kp, vp, perm[None, :], [L], 0.5)
    want = ops.gqa_attention(q[0], k, v, 0.5)
    np.testing.assert_array_equal(got[0], want)


def test_argmax_lowest_index_on_ties():
    assert int(ops.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0]))) == 1
    assert ops.argmax_lowest(np.array([[0.0, 0.0], [1.0, 5.0]])).tolist() == [0, 1]
