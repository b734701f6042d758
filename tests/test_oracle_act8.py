"""Pins of the oracle's int8 absmax activation quantisation (no GPU).

The form: inferencelayer ``cuda_llm.rs`` computes ``xs = [max|x|, 1/max|x|]`` before every GEMV
(``CudaQwen3::absmax``); the library's reading is one scale per vector, codes
``round_half_even(x * 127 / max|x|)``, the GEMV multiplying ``q * max|x| / 127``. The values below
are worked out by hand from that rule; the invariants follow from it.
"""
import numpy as np
import pytest

from oracle import act8


def test_hand_derived_codes():
    # m = 2, scale 127/2 = 63.5: products 127, -63.5, 31.75, -127, 0, 1.5875
    x = np.array([2.0, -1.0, 0.5, -2.0, 0.0, 0.025])
    q, m = act8.absmax_codes(x)
    assert float(m[0]) == 2.0
    # -63.5 ties to the even -64; 31.75 -> 32; 0.025 * 63.5 = 1.5875 -> 2
    assert q.tolist() == [127, -64, 32, -127, 0, 2]
    xh = act8.absmax_dequant(x)
    assert np.allclose(xh, np.array([127, -64, 32, -127, 0, 2]) * (2.0 / 127), rtol=0, atol=0)


def test_ties_go_to_even():
    # m = 127: scale exactly 1, so x itself is the product
    x = np.array([127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5])
    q, _ = act8.absmax_codes(x)
    assert q.tolist() == [127, 0, 2, 2, 0, -2, -2, 4]


def test_zero_vector_and_batch_rows_independent():
    q, m = act8.absmax_codes(np.zeros((2, 8)))
    assert not q.any() and not m.any()
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 64))
    q, m = act8.absmax_codes(x)
    for r in range(3):
        qr, mr = act8.absmax_codes(x[r])
        assert np.array_equal(q[r], qr) and m[r, 0] == mr[0]


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_bounds_extremes_and_symmetry(seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(4096) * 10.0 ** rng.uniform(-3, 3)
    q, m = act8.absmax_codes(x)
    assert np.abs(q.astype(int)).max() == 127                     # the largest |x| maps to 127
    assert q[np.argmax(np.abs(x.astype(np.float32)))] in (127, -127)
    xh = act8.absmax_dequant(x)
    x32 = x.astype(np.float32).astype(np.float64)
    # one rounding to the nearest code: at most half a step (plus f32 rounding of the scale)
    assert np.all(np.abs(x32 - xh) <= float(m[0]) / 254 * (1 + 1e-5))
    qn, _ = act8.absmax_codes(-x)
    assert np.array_equal(qn, -q)                                  # odd symmetry
    q2, m2 = act8.absmax_codes(x * 8.0)                            # a power of two: same codes
    assert np.array_equal(q2, q) and float(m2[0]) == 8.0 * float(m[0])
