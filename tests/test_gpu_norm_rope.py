"""Fused q/k RMSNorm + RoPE + paged KV append on the GPU against the oracle.

q and K are f32 computations rounded to f16 (bar: 2e-3 + 2e-3 |ref|, a few f16 ulps plus the
f32 cos/sin tables); V is copied, and block-table indexing is checked bit-exactly: exactly the
slot (block_tables[b][p/16], p%16) of each kv head changes, every other slot keeps its
sentinel.
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import ops

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hd,nh,nkv", [(64, 4, 2), (128, 32, 8), (128, 8, 8)])
def test_norm_rope_append(hd, nh, nkv):
    ql = lib()
    rng = np.random.default_rng(hd + nh)
    B, maxb, num_blocks, theta, eps = 5, 6, 40, 1e6, 1e-6
    positions = np.array([0, 15, 16, 33, 95], np.int32)
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = perm[: B * maxb].reshape(B, maxb)
    qkv = (rng.standard_normal((B, (nh + 2 * nkv) * hd)) * 1.5).astype(np.float32)
    # V values exactly representable in f16 so the copy is bit-exact
    qkv[:, (nh + nkv) * hd:] = qkv[:, (nh + nkv) * hd:].astype(np.float16).astype(np.float32)
    qn = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
    kn = (1 + 0.1 * rng.standard_normal(hd)).astype(np.float32)
    max_pos = maxb * 16
    cos_t = np.empty((max_pos, hd // 2), np.float32)
    sin_t = np.empty((max_pos, hd // 2), np.float32)
    ql.ql_rope_tables(cos_t, sin_t, theta)
    sentinel = np.float16(-7.5)
    kp = torch.full((num_blocks, nkv, 16, hd), float(sentinel), dtype=torch.float16, device="cuda")
    vp = kp.clone()
    qo = torch.empty((B, nh, hd), dtype=torch.float16, device="cuda")
    ql.ql_fused_norm_rope(dev(qkv), dev(qn), dev(kn), dev(cos_t), dev(sin_t), dev(positions), None,
                          eps, B, nh, nkv, hd, qo, kp, vp, dev(bt), maxb, 16, num_blocks, max_pos)
    torch.cuda.synchronize()
    q_got = qo.float().cpu().numpy()
    K = kp.cpu().numpy()
    V = vp.cpu().numpy()
    touched = np.zeros(K.shape[:3], bool)
    for b in range(B):
        p = int(positions[b])
        y = qkv[b].astype(np.float64)
        q = y[: nh * hd].reshape(nh, hd)
        k = y[nh * hd:(nh + nkv) * hd].reshape(nkv, hd)
        v = y[(nh + nkv) * hd:].reshape(nkv, hd)
        q_ref = ops.rope(ops.rmsnorm(q, qn, eps), p, theta)
        k_ref = ops.rope(ops.rmsnorm(k, kn, eps), p, theta)
        np.testing.assert_allclose(q_got[b], q_ref, rtol=2e-3, atol=2e-3)
        blk, slot = int(bt[b, p // 16]), p % 16
        np.testing.assert_allclose(K[blk, :, slot].astype(np.float64), k_ref, rtol=2e-3, atol=2e-3)
        assert np.array_equal(V[blk, :, slot], v.astype(np.float16))
        touched[blk, :, slot] = True
    assert np.all(K[~touched] == sentinel) and np.all(V[~touched] == sentinel)


def test_norm_rope_inactive_slot_and_position_zero():
    ql = lib()
    hd, nh, nkv, B = 64, 4, 2, 2
    rng = np.random.default_rng(3)
    qkv = rng.standard_normal((B, (nh + 2 * nkv) * hd)).astype(np.float32)
    ones = np.ones(hd, np.float32)
    cos_t = np.empty((32, hd // 2), np.float32)
    sin_t = np.empty((32, hd // 2), np.float32)
    ql.ql_rope_tables(cos_t, sin_t, 1e6)
    kp = torch.zeros((4, nkv, 16, hd), dtype=torch.float16, device="cuda")
    vp = kp.clone()
    qo = torch.zeros((B, nh, hd), dtype=torch.float16, device="cuda")
    bt = np.array([[0, 1], [2, 3]], np.int32)
    ql.ql_fused_norm_rope(dev(qkv), dev(ones), dev(ones), dev(cos_t), dev(sin_t),
                          dev(np.array([0, 5], np.int32)), dev(np.array([1, 0], np.int32)), 1e-6,
                          B, nh, nkv, hd, qo, kp, vp, dev(bt), 2, 16, 4, 32)
    torch.cuda.synchronize()
    # slot 1 inactive: nothing written; slot 0 at position 0: rope is the identity
    assert float(kp[2:].abs().sum()) == 0.0 and float(qo[1].abs().sum()) == 0.0
    q0 = qkv[0, : nh * hd].reshape(nh, hd).astype(np.float64)
    np.testing.assert_allclose(qo[0].float().cpu().numpy(), ops.rmsnorm(q0, ones, 1e-6),
                               rtol=2e-3, atol=2e-3)
