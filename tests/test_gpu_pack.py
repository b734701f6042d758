"""The q4_0 quantiser on the GPU (ql_q4_0_pack_device) against the oracle's, byte for byte.

Every model the library builds is quantised on the device, so this is the pin that the codes the
GPU multiplies are the codes the oracle defines (inferencelayer ``cuda_llm.rs``, ``Q4Dev``: one
f16 scale and 16 bytes of 4-bit codes per 32 weights, weight = (q - 8) d; the quantiser rule is
the library's reading: d = nearest f16 of max|x| / 7, q = clamp(round_half_even(x / d), -7, 7)
+ 8). The expected bytes come from ``oracle.q4_0.quantize`` and, for the hand-derived blocks,
from ``tests/golden/q4_0_blocks.txt``; nothing here is taken from the GPU.
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import q4_0 as oq

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu


def device_pack(w: np.ndarray):
    """Quantise the f32 host matrix ``w`` on the GPU; returns (scale bits u16, codes u8)."""
    ql = lib()
    rows, cols = w.shape
    d_w = dev(np.ascontiguousarray(w, np.float32))
    s = torch.empty((rows, cols // 32), dtype=torch.int16, device="cuda")
    q = torch.empty((rows, cols // 32, 16), dtype=torch.uint8, device="cuda")
    ql.ql_q4_0_pack_device(d_w, s, q)
    torch.cuda.synchronize()
    ql.ql_check_device_error()
    return s.cpu().numpy().view(np.uint16), q.cpu().numpy()


def test_golden_blocks_bit_exact():
    from test_oracle_q4_0 import load_golden
    cases = load_golden()
    x = np.stack([c[1] for c in cases]).astype(np.float32)       # one block per row
    s, q = device_pack(x)
    for i, (name, _, scale, qb) in enumerate(cases):
        assert int(s[i, 0]) == scale, name
        assert np.array_equal(q[i, 0], qb), name


def test_edge_blocks_bit_exact():
    rows = []
    rows.append(np.zeros(32))                                  # all zero: d = 0, q = 8
    r = np.zeros(32); r[3] = 5.0; rows.append(r)                # +amax alone
    r = np.zeros(32); r[20] = -5.0; rows.append(r)              # -amax alone (high nibble)
    r = np.full(32, -3.25); rows.append(r)                      # constant block, every q = 1
    # exact half-steps of d = 1 (amax 7): ties go to the even integer
    rows.append(np.array([0.5, 1.5, 2.5, 3.5, 4.5, 5.5, 6.5, -0.5, -1.5, -2.5, -3.5, -4.5, -5.5,
                          -6.5, 7.0] + [0.0] * 17))
    # a block whose f16 scale is subnormal (max|x| / 7 < 2^-14)
    rows.append(np.linspace(-3e-4, 2e-4, 32))
    # tiny values that round to zero codes against a large amax
    r = np.full(32, 1e-3); r[0] = 70.0; rows.append(r)
    # values just either side of a half-step after the scale's f16 rounding
    r = np.arange(32, dtype=np.float64) * 0.41 - 6.5; rows.append(r)
    x = np.stack(rows).astype(np.float32)
    s, q = device_pack(x)
    s_ref, q_ref = oq.quantize(x)
    d = s_ref.view(np.float16)
    assert d[5, 0] != 0 and abs(float(d[5, 0])) < 2.0 ** -14, "the subnormal-scale case must have one"
    assert np.array_equal(s, s_ref)
    assert np.array_equal(q, q_ref)


def test_wide_dynamic_range_bit_exact():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((256, 128)) * np.logspace(-6, 3, 256)[:, None]).astype(np.float32)
    s, q = device_pack(w)
    s_ref, q_ref = oq.quantize(w)
    assert np.array_equal(s, s_ref) and np.array_equal(q, q_ref)


def test_full_gate_up_matrix_bit_exact():
    """A whole 24576 x 4096 N(0, 0.02) matrix (the gate|up shape), every byte compared."""
    rows, cols = 24576, 4096
    w = ql_inputs.gemv_weight(rows, cols, seed=2)
    s, q = device_pack(w)
    step = 2048
    for r0 in range(0, rows, step):
        s_ref, q_ref = oq.quantize(w[r0:r0 + step])
        assert np.array_equal(s[r0:r0 + step], s_ref), f"scales differ in rows {r0}..{r0 + step}"
        assert np.array_equal(q[r0:r0 + step], q_ref), f"codes differ in rows {r0}..{r0 + step}"


def test_non_finite_weight_recorded_not_faulted():
    ql = lib()
    x = np.zeros((2, 64), np.float32)
    x[1, 40] = np.nan
    d_w = dev(x)
    s = torch.empty((2, 2), dtype=torch.int16, device="cuda")
    q = torch.empty((2, 2, 16), dtype=torch.uint8, device="cuda")
    ql.ql_q4_0_pack_device(d_w, s, q)
    with pytest.raises(ql.QLError) as e:
        ql.ql_check_device_error()
    assert e.value.status == ql.QL_EDEVICE
    # the bad block is written as d = 0, q = 8; the others are the oracle's
    sh, qh = s.cpu().numpy().view(np.uint16), q.cpu().numpy()
    assert sh[1, 1] == 0 and np.all(qh[1, 1] == 0x88)
    s_ref, q_ref = oq.quantize(x[:1])
    assert np.array_equal(sh[:1], s_ref) and np.array_equal(qh[:1], q_ref)
