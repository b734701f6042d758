"""The library's host codec for quantised KV rows (``ql_kv_*``, q8_0 keys / q5_1 values)
against the oracle (no GPU): identical bytes, identical decoded f32 values, the same errors.

Rows cover the cases the format distinguishes: N(0, s^2) values over eight orders of magnitude,
ragged tails (dim not a multiple of 32), constant and all-zero blocks, exact ties of the
rounding, negative zeros, and a block whose scale is subnormal.
"""
import numpy as np
import pytest

import quantized_transformer_decode_ql_gb300 as ql
from oracle import kvq


def rows_for(dim, seed):
    rng = np.random.default_rng(seed)
    blocks = []
    for s in (1e-4, 1e-2, 1.0, 3.5, 250.0, 1e4):   # |x| stays inside f16 (the minimum is stored)
        blocks.append(rng.standard_normal((6, dim)) * s)
    x = np.concatenate(blocks).astype(np.float32)
    x[0, :] = 0.0                                   # all zero
    x[1, :] = np.float32(-0.0)                      # negative zeros
    x[2, :] = np.float32(1.25)                      # constant
    x[3, : min(dim, 32)] = np.arange(min(dim, 32), dtype=np.float32) + np.float32(0.5)  # ties
    x[4, 0] = np.float32(1e-40)                     # a subnormal amax in its block
    x[4, 1:32] = 0.0
    return x


@pytest.mark.parametrize("dim", [32, 128, 1024, 33, 100])
def test_host_codec_matches_the_oracle(dim):
    x = rows_for(dim, dim)
    for q, dq, oq, odq, rb in (
            (ql.ql_kv_quantize_q8_0, ql.ql_kv_dequantize_q8_0, kvq.quantize_q8_0, kvq.dequantize_q8_0,
             kvq.q8_row_bytes),
            (ql.ql_kv_quantize_q5_1, ql.ql_kv_dequantize_q5_1, kvq.quantize_q5_1, kvq.dequantize_q5_1,
             kvq.q5_row_bytes)):
        got = q(x)
        want = oq(x)
        assert got.shape == (x.shape[0], rb(dim))
        assert np.array_equal(got, want), np.argwhere(got != want)[:5]
        a, b = dq(got, dim), odq(want, dim)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_row_bytes():
    assert ql.ql_kv_q8_0_row_bytes(128) == 136 and ql.ql_kv_q5_1_row_bytes(128) == 96
    assert ql.ql_kv_q8_0_row_bytes(33) == 68 and ql.ql_kv_q5_1_row_bytes(33) == 48
    assert ql.ql_kv_q8_0_row_bytes(0) == 0 and ql.ql_kv_q5_1_row_bytes(-4) == 0


def test_host_codec_errors():
    lib = ql.lib()
    x = np.ones((2, 64), np.float32)
    out = np.zeros((2, 136), np.uint8)
    assert lib.ql_kv_quantize_q8_0(None, 2, 64, out.ctypes.data) == ql.QL_EINVAL
    assert lib.ql_kv_quantize_q8_0(x.ctypes.data, 0, 64, out.ctypes.data) == ql.QL_EINVAL
    x[1, 5] = np.nan
    assert lib.ql_kv_quantize_q5_1(x.ctypes.data, 2, 64, out.ctypes.data) == ql.QL_EINVAL
    big = np.full((1, 32), 1e7, np.float32)        # d = 1e7 / 127 overflows f16
    assert lib.ql_kv_quantize_q8_0(big.ctypes.data, 1, 32, out.ctypes.data) == ql.QL_EINVAL
    neg = np.full((1, 32), -7e4, np.float32)        # the minimum overflows f16
    assert lib.ql_kv_quantize_q5_1(neg.ctypes.data, 1, 32, out.ctypes.data) == ql.QL_EINVAL
