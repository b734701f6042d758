"""Deliberate-defect gates for the quantised KV-row codecs: a plausible mistake planted in the
oracle (on the CPU) must make one of its pins fail."""
import numpy as np

from oracle import kvq

import test_oracle_kvq as pins


def fails(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def q8_with(round_fn=np.rint, qmax=127.0):
    """A q8_0 quantiser with one rule changed (the rounding, or the divisor of the scale)."""
    def quantize(rows):
        b = kvq._blocks(rows)
        n, nblk, _ = b.shape
        d = (np.max(np.abs(b), axis=2) / np.float32(qmax)).astype(np.float32)
        inv = kvq._inverse(d)
        code = np.clip(round_fn((b * inv[:, :, None]).astype(np.float32)), -127, 127).astype(np.int8)
        out = np.zeros((n, nblk, 34), np.uint8)
        db = kvq._f16_bits(d)
        out[:, :, 0], out[:, :, 1] = db & 0xFF, db >> 8
        out[:, :, 2:] = code.view(np.uint8)
        return out.reshape(n, -1)
    return quantize


def test_the_pins_accept_the_oracle():
    for pin in (pins.test_q8_block_derived_by_hand, pins.test_q8_ties_round_half_even,
                pins.test_q5_block_derived_by_hand, pins.test_q5_ties_and_clamp):
        pin()


def test_half_up_rounding_is_caught(monkeypatch):
    monkeypatch.setattr(kvq, "quantize_q8_0", q8_with(round_fn=lambda a: np.floor(a + 0.5)))
    assert fails(pins.test_q8_ties_round_half_even)
    assert fails(pins.test_q8_block_derived_by_hand)


def test_scale_divisor_128_is_caught(monkeypatch):
    monkeypatch.setattr(kvq, "quantize_q8_0", q8_with(qmax=128.0))
    assert fails(pins.test_q8_block_derived_by_hand)


def test_q5_adjacent_nibble_pairs_are_caught(monkeypatch):
    real = kvq.quantize_q5_1

    def bad(rows):   # element 2j in the low nibble of byte j, 2j + 1 in the high one
        out = real(rows)
        n = out.shape[0]
        blk = out.reshape(n, -1, 24)
        codes = kvq.q5_1_codes(out, blk.shape[1] * 32).reshape(n, -1, 32)
        lo = (codes & 0x0F).astype(np.uint8)
        blk[:, :, 8:] = lo[:, :, 0::2] | (lo[:, :, 1::2] << 4)
        return blk.reshape(n, -1)
    monkeypatch.setattr(kvq, "quantize_q5_1", bad)
    assert fails(pins.test_q5_block_derived_by_hand)


def test_q5_high_bits_in_reverse_order_are_caught(monkeypatch):
    real = kvq.quantize_q5_1

    def bad(rows):   # bit 31 - l of the high-bit word for element l
        out = real(rows)
        blk = out.reshape(out.shape[0], -1, 24)
        qh = np.zeros(blk.shape[:2], np.uint32)
        for k in range(4):
            qh |= blk[:, :, 4 + k].astype(np.uint32) << np.uint32(8 * k)
        rev = np.zeros_like(qh)
        for l in range(32):
            rev |= ((qh >> np.uint32(l)) & 1) << np.uint32(31 - l)
        for k in range(4):
            blk[:, :, 4 + k] = ((rev >> np.uint32(8 * k)) & 0xFF).astype(np.uint8)
        return blk.reshape(out.shape[0], -1)
    monkeypatch.setattr(kvq, "quantize_q5_1", bad)
    assert fails(pins.test_q5_block_derived_by_hand)


def test_q5_without_the_minimum_is_caught(monkeypatch):
    real_deq = kvq.dequantize_q5_1

    def bad_deq(data, dim):   # d * code, the minimum forgotten
        raw = np.asarray(data, np.uint8)
        blk = raw.reshape(raw.shape[0], -1, 24)
        d = (blk[:, :, 0].astype(np.uint16) | (blk[:, :, 1].astype(np.uint16) << 8)).view(np.float16)
        codes = kvq.q5_1_codes(raw, dim).reshape(raw.shape[0], -1, 32).astype(np.float32)
        return (d.astype(np.float32)[:, :, None] * codes).reshape(raw.shape[0], -1)[:, :dim]
    assert real_deq is not bad_deq
    monkeypatch.setattr(kvq, "dequantize_q5_1", bad_deq)
    assert fails(pins.test_q5_block_derived_by_hand)


def test_scale_divisor_126_is_caught(monkeypatch):
    monkeypatch.setattr(kvq, "quantize_q8_0", q8_with(qmax=126.0))   # the largest code clips
    assert fails(pins.test_q8_block_derived_by_hand)
    assert fails(lambda: pins.test_error_bound_of_the_format(1.0))
