"""Pins of the oracle's q4_0 codec (no GPU).

The codec follows the q4_0 format of inferencelayer ``cuda_llm.rs`` (``Q4Dev``): 32-weight
blocks, one f16 scale, 16 bytes of 4-bit codes, weight = (q - 8) * d.
"""
import os

import numpy as np
import pytest

from oracle import q4_0

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q4_0_blocks.txt")


def load_golden():
    lines = [l.strip() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    cases = []
    for i in range(0, len(lines), 4):
        name = lines[i]
        x = np.array([float(t) for t in lines[i + 1].split()], dtype=np.float32)
        scale = int(lines[i + 2], 16)
        qb = np.array([int(t, 16) for t in lines[i + 3].split()], dtype=np.uint8)
        cases.append((name, x, scale, qb))
    return cases


@pytest.mark.parametrize("case", load_golden(), ids=lambda c: c[0])
def test_golden_blocks(case):
    name, x, scale, qb = case
    assert x.shape == (32,) and qb.shape == (16,)
    s, q = q4_0.quantize(x[None, :])
    assert int(s[0, 0]) == scale, name
    assert np.array_equal(q[0, 0], qb), (name, q[0, 0], qb)


def test_golden_dequant_values():
    # nibble_order case: d = 1 exactly, so the dequantised block equals the input.
    for name, x, scale, qb in load_golden():
        if name in ("nibble_order", "plus_amax_first", "minus_amax_element17", "zeros"):
            w = q4_0.dequantize(np.array([[scale]], np.uint16), qb[None, None, :])
            assert np.array_equal(w[0], x.astype(np.float64)), name


def test_roundtrip_error_bound():
    # |x - (q-8) d| <= d/2 for every weight of a block with a normal f16 scale.
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((64, 4096)) * 0.02).astype(np.float32)
    s, q = q4_0.quantize(w)
    d = s.view(np.float16).astype(np.float64)
    assert np.all(d >= np.finfo(np.float16).tiny), "every scale must be a normal f16"
    err = np.abs(w.astype(np.float64) - q4_0.dequantize(s, q)).reshape(64, -1, 32)
    assert np.all(err <= d[..., None] / 2 + 0.0)
    # the extreme element of each block is reproduced to within d/2 and codes stay in 1..15
    c = q4_0.codes(q)
    assert c.min() >= 1 and c.max() <= 15
    assert np.all(np.any((c == 1) | (c == 15), axis=-1))


def _nearest_f16_bruteforce(v: float) -> int:
    """Bits of the f16 nearest to v (ties to the even bit pattern), by exhaustive search."""
    allbits = np.arange(0, 0x7C00, dtype=np.uint16)           # all finite non-negative f16
    vals = allbits.view(np.float16).astype(np.float64)
    dist = np.abs(vals - v)
    best = np.flatnonzero(dist == dist.min())
    if len(best) == 1:
        return int(allbits[best[0]])
    even = [b for b in best if int(allbits[b]) % 2 == 0]
    return int(allbits[even[0]])


def test_scale_is_nearest_f16_bruteforce():
    rng = np.random.default_rng(5)
    amax = np.concatenate([np.abs(rng.standard_normal(200)) * 0.05,
                           np.array([1.0, 7.0, 0.1, 3e-5, 1e-7, 100.0])])
    got = q4_0.f16_scale(amax).view(np.uint16)
    for a, g in zip(amax, got):
        assert int(g) == _nearest_f16_bruteforce(a / 7.0), a


def test_scale_ties_to_even():
    # amax/7 exactly halfway between two f16 neighbours: 1 + 2^-11 (between 1 and 1+2^-10)
    # rounds to 1.0 (even); 1 + 3*2^-11 rounds up to 1 + 2^-9 (even mantissa 2).
    for mid, want in ((1.0 + 2.0 ** -11, 0x3C00), (1.0 + 3 * 2.0 ** -11, 0x3C02)):
        got = int(q4_0.f16_scale(np.array([mid * 7.0])).view(np.uint16)[0])
        assert got == want, hex(got)


def test_zero_block_and_single_nonzero():
    x = np.zeros((2, 64), np.float32)
    x[1, 40] = -0.3
    s, q = q4_0.quantize(x)
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0
    assert np.all(q[0] == 0x88) and np.all(q[1, 0] == 0x88)
    c = q4_0.codes(q[1, 1])
    assert c[8] == 1 and np.all(np.delete(c, 8) == 8)


def test_errors():
    with pytest.raises(ValueError):
        q4_0.quantize(np.zeros((2, 33), np.float32))
    bad = np.zeros((1, 32), np.float32)
    bad[0, 3] = np.nan
    with pytest.raises(ValueError):
        q4_0.quantize(bad)
    big = np.zeros((1, 32), np.float32)
    big[0, 0] = 7.0 * 70000.0
    with pytest.raises(ValueError):
        q4_0.quantize(big)


def test_rows_are_independent():
    # q4_0 quantises row-wise, so concatenating matrices along rows commutes with quantising
    # (the fused q|k|v and gate|up matrices of inferencelayer LayerDev rely on this).
    rng = np.random.default_rng(3)
    a = (rng.standard_normal((5, 96)) * 0.02).astype(np.float32)
    b = (rng.standard_normal((7, 96)) * 0.02).astype(np.float32)
    sa, qa = q4_0.quantize(a)
    sb, qb = q4_0.quantize(b)
    s, q = q4_0.quantize(np.concatenate([a, b]))
    assert np.array_equal(s, np.concatenate([sa, sb]))
    assert np.array_equal(q, np.concatenate([qa, qb]))
