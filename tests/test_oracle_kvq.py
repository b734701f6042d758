"""Pins of the oracle's quantised KV-row codecs (no GPU).

The codecs follow memra-engine ``qwen4exp_gpu.rs`` (the q8_0 / q5_1 cache rows and their host
twins). Each pin is fixed by something other than the oracle's own code: bytes derived by
hand from the format, closed forms where the f32 arithmetic is exact, the rounding rule on
exact ties, the guard for a subnormal scale, the error bound of the format, and exact
invariances (sign, powers of two).
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import kvq, ops


def le16(b, i):
    return int(b[i]) | (int(b[i + 1]) << 8)


def test_row_sizes_and_ragged_tail():
    assert kvq.q8_row_bytes(128) == 4 * 34 and kvq.q5_row_bytes(128) == 4 * 24
    assert kvq.q8_row_bytes(33) == 68 and kvq.q5_row_bytes(33) == 48
    x = np.zeros((1, 33), np.float32)
    x[0, 32] = 1.0   # the tail block: one value, 31 zeros of padding
    q8 = kvq.quantize_q8_0(x)[0]
    assert q8.shape == (68,)
    assert list(q8[34 + 2:]) == [127] + [0] * 31          # amax 1 -> d = 1/127, code 127
    q5 = kvq.quantize_q5_1(x)[0]
    assert q5.shape == (48,)
    assert le16(q5, 24 + 2) == 0x0000                      # the padding makes the minimum 0


def test_zero_row_gives_zero_scale_and_codes():
    z = np.zeros((2, 64), np.float32)
    assert not kvq.quantize_q8_0(z).any()
    assert not kvq.quantize_q5_1(z).any()
    assert not kvq.dequantize_q8_0(kvq.quantize_q8_0(z), 64).any()
    assert not kvq.dequantize_q5_1(kvq.quantize_q5_1(z), 64).any()


def test_q8_block_derived_by_hand():
    # x_l = l - 16: amax = 16, d = f32(16/127), and 1/d rounds to 127/16 = 7.9375 exactly, so
    # x * id = k * 127 / 16 is exact in f32 and the code is that rational rounded half-even.
    x = (np.arange(32, dtype=np.float32) - 16)[None, :]
    b = kvq.quantize_q8_0(x)[0]
    # f16 nearest to 16/127 = 0.12598...: 2^-3 * (1 + 8/1024) -> bits 0x3008
    assert le16(b, 0) == 0x3008
    want = [round(Fraction(k * 127, 16)) for k in range(-16, 16)]   # Python round: half-even
    assert list(b[2:].view(np.int8)) == want
    assert want[16 + 8] == 64 and want[16 - 8] == -64                # the ties 63.5 / -63.5
    # decoded: 0.1259765625 * code, exact
    dq = kvq.dequantize_q8_0(b[None, :], 32)[0]
    assert np.array_equal(dq, np.float32(0.1259765625) * np.array(want, np.float32))


def test_q8_ties_round_half_even():
    # amax 127 -> d = 1, id = 1: the codes are the values rounded half-even
    x = np.zeros(32, np.float32)
    x[:9] = [127, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5, 126.5]
    codes = kvq.quantize_q8_0(x[None, :])[0][2:].view(np.int8)
    assert list(codes[:9]) == [127, 2, 4, -2, -4, 0, 2, 0, 126]
    assert le16(kvq.quantize_q8_0(x[None, :])[0], 0) == 0x3C00       # f16(1.0)


def test_q5_block_derived_by_hand():
    # x_l = l: min 0, max 31, d = 1, code l; bit 4 set for l >= 16; byte l = l | (l << 4)
    x = np.arange(32, dtype=np.float32)[None, :]
    b = kvq.quantize_q5_1(x)[0]
    assert le16(b, 0) == 0x3C00 and le16(b, 2) == 0x0000
    qh = int(b[4]) | (int(b[5]) << 8) | (int(b[6]) << 16) | (int(b[7]) << 24)
    assert qh == 0xFFFF0000
    assert list(b[8:]) == [17 * l for l in range(16)]
    assert np.array_equal(kvq.dequantize_q5_1(b[None, :], 32)[0], x[0])
    # shifted by 0.25: the same codes, m = f16(0.25) = 0x3400, decoded exactly
    y = x + np.float32(0.25)
    c = kvq.quantize_q5_1(y)[0]
    assert le16(c, 2) == 0x3400 and np.array_equal(c[4:], b[4:])
    assert np.array_equal(kvq.dequantize_q5_1(c[None, :], 32)[0], y[0])


def test_q5_ties_and_clamp():
    # min 0, max 31 (d = 1): (x - 0) * 1 rounds half-even
    x = np.zeros(32, np.float32)
    x[:6] = [31, 2.5, 3.5, 30.5, 0.5, 1.5]
    codes = kvq.q5_1_codes(kvq.quantize_q5_1(x[None, :]), 32)[0]
    assert list(codes[:6]) == [31, 2, 4, 30, 0, 2]


def test_subnormal_scale_guard():
    # amax = 1e-40 (an f32 subnormal): d = amax / 127 is subnormal, 1/d overflows -> id = 0
    x = np.zeros((1, 32), np.float32)
    x[0, 3] = np.float32(1e-40)
    b = kvq.quantize_q8_0(x)[0]
    assert not b[2:].any()
    c = kvq.quantize_q5_1(x)[0]
    assert not kvq.q5_1_codes(c[None, :], 32).any()


@pytest.mark.parametrize("sigma", [1e-3, 1.0, 37.0, 3000.0])
def test_error_bound_of_the_format(sigma):
    rng = np.random.default_rng(int(sigma * 7) + 1)
    x = (rng.standard_normal((64, 128)) * sigma).astype(np.float32)
    xb = x.reshape(64, 4, 32).astype(np.float64)
    # q8_0: |x - d16 q| <= d/2 + 127 |d16 - d| + f32 rounding of d and of x * id
    d = np.abs(xb).max(axis=2) / 127.0
    d16 = d.astype(np.float32).astype(np.float16).astype(np.float64)
    e8 = np.abs(xb - kvq.dequantize_q8_0(kvq.quantize_q8_0(x), 128).reshape(64, 4, 32))
    bound8 = 0.5 * d + 127 * np.abs(d16 - d) + 1e-6 * d * 127
    assert (e8 <= bound8[:, :, None]).all()
    assert e8.max() > 0.2 * d.max()          # not vacuous: the codes do round
    # q5_1: |x - (d16 q + m16)| <= d/2 + 31 |d16 - d| + |m16 - mn| + f32 roundings
    mn, mx = xb.min(axis=2), xb.max(axis=2)
    d5 = (mx - mn) / 31.0
    d516 = d5.astype(np.float32).astype(np.float16).astype(np.float64)
    m16 = mn.astype(np.float32).astype(np.float16).astype(np.float64)
    e5 = np.abs(xb - kvq.dequantize_q5_1(kvq.quantize_q5_1(x), 128).reshape(64, 4, 32))
    bound5 = 0.5 * d5 + 31 * np.abs(d516 - d5) + np.abs(m16 - mn) + 1e-6 * (np.abs(mx) + np.abs(mn) + 31 * d5)
    assert (e5 <= bound5[:, :, None]).all()


def test_sign_and_power_of_two_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((8, 96)).astype(np.float32)
    a = kvq.quantize_q8_0(x)
    n = kvq.quantize_q8_0(-x)
    # same scale bytes, codes negated
    a3, n3 = a.reshape(8, 3, 34), n.reshape(8, 3, 34)
    assert np.array_equal(a3[:, :, :2], n3[:, :, :2])
    assert np.array_equal(a3[:, :, 2:].view(np.int8), -n3[:, :, 2:].view(np.int8))
    # x * 4: every f32 step scales exactly, so the codes are unchanged and d is 4x
    s = kvq.quantize_q8_0(x * np.float32(4.0)).reshape(8, 3, 34)
    assert np.array_equal(s[:, :, 2:], a3[:, :, 2:])
    d_a = a3[:, :, :2].copy().view(np.float16).astype(np.float64)
    d_s = s[:, :, :2].copy().view(np.float16).astype(np.float64)
    assert np.array_equal(d_s, 4 * d_a)
    t = kvq.quantize_q5_1(x * np.float32(0.5)).reshape(8, 3, 24)
    u = kvq.quantize_q5_1(x).reshape(8, 3, 24)
    assert np.array_equal(t[:, :, 4:], u[:, :, 4:])


def test_quantised_attention_equals_exact_attention_on_representable_pools():
    # keys in {-127..127} * 2^-6 and values l + 0.25 per block are represented exactly by
    # q8_0 / q5_1 (amax 127 * 2^-6 in every key block, a 0..31 ramp in every value block), so
    # the attention over the decoded pools equals the plain attention over the originals
    rng = np.random.default_rng(5)
    nb, nkv, hd = 4, 2, 64
    kint = rng.integers(-127, 128, size=(nb, nkv, 16, hd)).astype(np.float32)
    kint.reshape(-1, hd // 32, 32)[:, :, 0] = 127          # every block's amax is 127
    k = kint * np.float32(2.0 ** -6)
    ramp = np.arange(32, dtype=np.float32)
    v = np.empty((nb, nkv, 16, hd), np.float32)
    for blk in range(hd // 32):
        v[..., blk * 32:(blk + 1) * 32] = rng.permutation(ramp) + np.float32(0.25)
    kc = kvq.quantize_q8_0(k.reshape(-1, hd)).reshape(nb, nkv, 16, -1)
    vc = kvq.quantize_q5_1(v.reshape(-1, hd)).reshape(nb, nkv, 16, -1)
    assert np.array_equal(kvq.dequantize_q8_0(kc.reshape(-1, kc.shape[-1]), hd), k.reshape(-1, hd))
    assert np.array_equal(kvq.dequantize_q5_1(vc.reshape(-1, vc.shape[-1]), hd), v.reshape(-1, hd))
    q = rng.standard_normal((2, 4, hd)).astype(np.float32)
    bt = np.array([[0, 2], [1, 3]], np.int32)
    lens = np.array([20, 31], np.int32)
    got = kvq.paged_attention_q8k_q5v(q, kc, vc, hd, bt, lens, 1.0 / math.sqrt(hd))
    want = ops.paged_attention(q, k, v, bt, lens, 1.0 / math.sqrt(hd))
    assert np.array_equal(got, want)


def test_non_finite_rows_are_rejected():
    x = np.zeros((1, 32), np.float32)
    x[0, 1] = np.inf
    with pytest.raises(ValueError):
        kvq.quantize_q8_0(x)
    with pytest.raises(ValueError):
        kvq.quantize_q5_1(x)
