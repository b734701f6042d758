"""Causal attention of a prefill chunk (ql_paged_attn_chunk) against the oracle.

inferencelayer ``cuda_llm.rs`` runs a prompt as sequential decode: token t of a chunk that
starts at position p0 attends keys 0 .. p0 + t. The oracle's reference is its paged attention
with one row per token (length p0 + t + 1, the sequence's block table). Shapes cover query
groups of 1, 2, 4 and 8 heads per kv head (G = 8 with 32 tokens puts 256 query rows per kv head
into two row groups), head_dim 64 and 128, single-token chunks, a chunk at position 0, chunks
that start and end inside a block, and a fragmented block table. Tolerance as the decode
attention's (tests/test_gpu_attention.py): ``|o - o_ref| <= 2e-3 + 1e-2 |o_ref|``.
"""
import math

import numpy as np
import pytest
import torch

import ql_inputs
from oracle import ops

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu


def run_chunk(T, p0, n_heads, n_kv, hd, seed, maxb=None):
    ql = lib()
    rng = np.random.default_rng(seed)
    L = p0 + T
    nb = (L + 15) // 16
    maxb = maxb or nb + 2
    num_blocks = maxb + 5
    k_pool = rng.standard_normal((num_blocks, n_kv, 16, hd)).astype(np.float16)
    v_pool = rng.standard_normal((num_blocks, n_kv, 16, hd)).astype(np.float16)
    perm = ql_inputs.fragmented_block_ids(num_blocks, seed=seed + 1)
    table = np.full(maxb, -1, np.int32)
    table[:nb] = perm[:nb]
    q = rng.standard_normal((T, n_heads, hd)).astype(np.float16)
    scale = 1.0 / math.sqrt(hd)
    want = ops.paged_attention(q.astype(np.float64), k_pool.astype(np.float64), v_pool.astype(np.float64),
                               np.tile(table[:nb], (T, 1)), np.arange(p0 + 1, p0 + T + 1), scale)
    out = torch.full((T, n_heads * hd), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.empty(ql.ql_paged_attn_chunk_workspace_bytes(T, n_heads, n_kv, hd), dtype=torch.uint8, device="cuda")
    ql.ql_paged_attn_chunk(dev(q), dev(k_pool), dev(v_pool), dev(table), dev(np.array([p0], np.int32)), T, n_heads,
                           n_kv, hd, 16, maxb, num_blocks, scale, out, ws)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().reshape(T, n_heads, hd).astype(np.float64)
    return got, want


@pytest.mark.parametrize("n_heads,n_kv,hd", [(32, 8, 128), (16, 16, 64), (16, 8, 128), (64, 8, 128), (8, 2, 64)])
@pytest.mark.parametrize("T,p0", [(32, 2048), (1, 0), (7, 0), (13, 21), (32, 5), (17, 300)])
def test_chunk_attention_matches_oracle(n_heads, n_kv, hd, T, p0):
    got, want = run_chunk(T, p0, n_heads, n_kv, hd, seed=T * 7 + p0)
    assert not np.isnan(got).any()
    err = np.abs(got - want)
    assert np.all(err <= 2e-3 + 1e-2 * np.abs(want)), f"max err {err.max():.3e}"


def test_chunk_attention_is_causal():
    """Non-vacuity: changing the K/V rows after a token's position leaves that token's output
    bit for bit, while an earlier row changes it."""
    ql = lib()
    T, p0, nh, nkv, hd = 8, 40, 8, 2, 64
    rng = np.random.default_rng(5)
    nb = (p0 + T + 15) // 16
    num_blocks = nb + 2
    kp = rng.standard_normal((num_blocks, nkv, 16, hd)).astype(np.float16)
    vp = rng.standard_normal((num_blocks, nkv, 16, hd)).astype(np.float16)
    table = np.arange(nb, dtype=np.int32)
    q = rng.standard_normal((T, nh, hd)).astype(np.float16)
    ws = torch.empty(ql.ql_paged_attn_chunk_workspace_bytes(T, nh, nkv, hd), dtype=torch.uint8, device="cuda")

    def run(k, v):
        out = torch.empty((T, nh * hd), dtype=torch.float16, device="cuda")
        ql.ql_paged_attn_chunk(dev(q), dev(k), dev(v), dev(table), dev(np.array([p0], np.int32)), T, nh, nkv, hd, 16,
                               nb, num_blocks, 1.0 / math.sqrt(hd), out, ws)
        torch.cuda.synchronize()
        return out.cpu().numpy().reshape(T, nh, hd)
    base = run(kp, vp)
    k2, v2 = kp.copy(), vp.copy()
    last = p0 + T - 1   # the last token's own row: only the last token sees it
    k2[last // 16, :, last % 16] += np.float16(1.0)
    v2[last // 16, :, last % 16] += np.float16(1.0)
    after = run(k2, v2)
    assert np.array_equal(base[:-1], after[:-1])
    assert not np.array_equal(base[-1], after[-1])


def test_chunk_attention_rejects_bad_arguments():
    ql = lib()
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    q = torch.zeros((4, 8, 64), dtype=torch.float16, device="cuda")
    kp = torch.zeros((4, 2, 16, 64), dtype=torch.float16, device="cuda")
    out = torch.empty((4, 512), dtype=torch.float16, device="cuda")
    bt = dev(np.arange(4, dtype=np.int32))
    pos = dev(np.array([0], np.int32))
    for args in ((4, 8, 2, 96, 16), (4, 8, 3, 64, 16), (0, 8, 2, 64, 16), (4, 8, 2, 64, 32)):
        T, nh, nkv, hd, bs = args
        with pytest.raises(ql.QLError) as e:
            ql.ql_paged_attn_chunk(q, kp, kp, bt, pos, T, nh, nkv, hd, bs, 4, 4, 0.125, out, ws)
        assert e.value.status == ql.QL_EINVAL
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(ql.QLError) as e:
        ql.ql_paged_attn_chunk(q, kp, kp, bt, pos, 4, 8, 2, 64, 16, 4, 4, 0.125, out, small)
    assert e.value.status == ql.QL_EINVAL
