"""Paged split-K GQA decode attention on the GPU against the oracle.

Tolerance, from the kernel's arithmetic: q, K, V are f16 on both sides; scores, softmax and
the weighted sum are f32 (exp2 with a pre-scaled log2 e); the output is rounded to f16
(relative 2^-11). Outputs are convex combinations of N(0,1) values, so the bar is
``|o - o_ref| <= 2e-3 + 1e-2 |o_ref|``.
"""
import math

import numpy as np
import pytest
import torch

import ql_inputs
from oracle import ops

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu


def gpu_attention(case, n_heads, n_kv, hd, max_blocks=None, block_tables=None, k_pool=None,
                  v_pool=None, lens=None):
    ql = lib()
    q = dev(case["q"])
    kp = dev(case["k_pool"] if k_pool is None else k_pool)
    vp = dev(case["v_pool"] if v_pool is None else v_pool)
    bt_np = case["block_tables"] if block_tables is None else block_tables
    B = case["q"].shape[0]
    mb = bt_np.shape[1] if max_blocks is None else max_blocks
    bt = np.full((B, mb), -1, np.int32)
    bt[:, : bt_np.shape[1]] = bt_np
    lens = case["lens"] if lens is None else lens
    out = torch.full((B, n_heads * hd), float("nan"), dtype=torch.float16, device="cuda")
    wsb = ql.ql_paged_attn_workspace_bytes(B, n_heads, n_kv, hd, 16, mb)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    num_blocks = kp.shape[0]
    ql.ql_paged_attn_decode(q, kp, vp, dev(bt), dev(np.asarray(lens, np.int32)), B, n_heads, n_kv,
                            hd, 16, mb, num_blocks, 1.0 / math.sqrt(hd), out, ws)
    torch.cuda.synchronize()
    # the workspace is left zero-filled (tickets re-armed) for the next call
    assert int(ws[:4 * B * n_kv].view(torch.int32).abs().sum()) == 0
    return out.float().cpu().numpy().reshape(B, n_heads, hd).astype(np.float64)


def oracle_attention(case, hd):
    return ops.paged_attention(case["q"], case["k_pool"], case["v_pool"], case["block_tables"],
                               case["lens"], 1.0 / math.sqrt(hd))


def check(got, want, what):
    assert not np.any(np.isnan(got)), what
    err = np.abs(got - want)
    bad = err > 2e-3 + 1e-2 * np.abs(want)
    assert not bad.any(), f"{what}: {bad.sum()} bad, max err {err.max():.3e}"


@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("n_heads,n_kv", [(4, 4), (4, 2), (32, 8), (16, 2)])
def test_attention_lengths(hd, n_heads, n_kv):
    lens = [1, 15, 16, 17, 33, 100, 257, 1000]
    case = ql_inputs.attention_case(len(lens), n_heads, n_kv, hd, lens, seed=4)
    got = gpu_attention(case, n_heads, n_kv, hd)
    check(got, oracle_attention(case, hd), f"hd{hd} {n_heads}/{n_kv}")


@pytest.fixture(params=["cluster", "ticket"])
def merge(request):
    """Runs a test under each split-merge form (batch 1-2 shapes with 2..16 splits take the
    cluster form when it is selected and the device holds the launch's clusters)."""
    ql = lib()
    prev = ql.ql_set_attn_merge_form(ql.QL_ATTN_MERGE_CLUSTER if request.param == "cluster"
                                     else ql.QL_ATTN_MERGE_TICKET)
    yield request.param
    ql.ql_set_attn_merge_form(prev)


@pytest.mark.parametrize("L", [1, 2, 16, 17, 63, 64, 65, 511, 2049, 4096, 4100])
def test_attention_single_sequence(L, merge):
    case = ql_inputs.attention_case(1, 32, 8, 128, [L], seed=L)
    check(gpu_attention(case, 32, 8, 128), oracle_attention(case, 128), f"L={L}")


def test_split_count_independence():
    # a larger block-table capacity changes the split layout; results agree within tolerance
    lens = [700, 2048, 33]
    case = ql_inputs.attention_case(3, 32, 8, 128, lens, seed=11)
    a = gpu_attention(case, 32, 8, 128)
    b = gpu_attention(case, 32, 8, 128, max_blocks=case["max_blocks"] * 16)
    check(a, b, "split independence")
    check(a, oracle_attention(case, 128), "vs oracle")


def test_paged_equals_contiguous_bit_exact():
    lens = [300, 47, 1024]
    case = ql_inputs.attention_case(3, 32, 8, 128, lens, seed=12)
    got_perm = gpu_attention(case, 32, 8, 128)
    # the same logical KV laid out contiguously: sequence b's blocks are b*mb .. b*mb+n-1
    B, mb = 3, case["max_blocks"]
    kp = np.zeros((B * mb,) + case["k_pool"].shape[1:], np.float16)
    vp = np.zeros_like(kp)
    bt = np.full((B, mb), -1, np.int32)
    for b in range(B):
        n = (lens[b] + 15) // 16
        for i in range(n):
            kp[b * mb + i] = case["k_pool"][case["block_tables"][b, i]]
            vp[b * mb + i] = case["v_pool"][case["block_tables"][b, i]]
            bt[b, i] = b * mb + i
    got_id = gpu_attention(case, 32, 8, 128, block_tables=bt, k_pool=kp, v_pool=vp)
    assert np.array_equal(got_perm, got_id)


def test_idle_slot_untouched_and_rows_sum(merge):
    # context length 0 marks an idle slot: its output stays as it was (NaN sentinel here)
    case = ql_inputs.attention_case(2, 8, 2, 64, [40, 1], seed=13)
    got = gpu_attention(case, 8, 2, 64, lens=[40, 0])
    assert np.all(np.isnan(got[1]))
    check(got[:1], oracle_attention(case, 64)[:1], "live slot")
    # V = constant c for every key -> output c exactly up to f16 (softmax rows sum to 1)
    case2 = ql_inputs.attention_case(1, 8, 2, 64, [77], seed=14)
    case2["v_pool"][:] = np.float16(0.375)
    got2 = gpu_attention(case2, 8, 2, 64)
    assert np.allclose(got2, 0.375, atol=1e-3)


@pytest.mark.parametrize("B,lens", [(1, [511]), (1, [2049]), (1, [2304]), (1, [4096]), (1, [4100]),
                                    (2, [1000, 333]), (2, [2049, 17])])
def test_merge_forms_bit_identical(B, lens):
    """The cluster merge (partials in shared memory, read through distributed shared memory)
    and the ticket merge (partials in the workspace, merged by the last split) take the same
    merge over the splits in order: bit-identical outputs, both within the oracle's tolerance.
    The batch-1 shape of the decode benchmark (2049..2304 positions: 9-10 splits) must take
    the cluster form; shapes with more than 16 splits take the ticket form."""
    ql = lib()
    case = ql_inputs.attention_case(B, 32, 8, 128, lens, seed=sum(lens) + B)
    mb = case["max_blocks"]
    prev = ql.ql_set_attn_merge_form(ql.QL_ATTN_MERGE_CLUSTER)
    try:
        form = ql.ql_paged_attn_merge_form(B, 32, 8, 128, mb)
        a = gpu_attention(case, 32, 8, 128)
        ql.ql_set_attn_merge_form(ql.QL_ATTN_MERGE_TICKET)
        assert ql.ql_paged_attn_merge_form(B, 32, 8, 128, mb) == ql.QL_ATTN_MERGE_TICKET
        b = gpu_attention(case, 32, 8, 128)
    finally:
        ql.ql_set_attn_merge_form(prev)
    nsplit = -(-mb // 16)
    if nsplit > 16:
        assert form == ql.QL_ATTN_MERGE_TICKET
    if B == 1 and 9 <= nsplit <= 10:
        assert form == ql.QL_ATTN_MERGE_CLUSTER
    assert np.array_equal(a, b), f"forms differ: max {np.abs(a - b).max():.3e} (form {form})"
    check(a, oracle_attention(case, 128), f"B={B} lens={lens}")


@pytest.mark.slow
@pytest.mark.parametrize("batch", [1, 8, 64])
def test_attention_full_size_sampled(batch):
    """The attention-alone workload at full size (32/8 heads, hd 128, lengths uniform in
    [512, 32768], fragmented tables); the oracle checks sampled (sequence, head) pairs."""
    lens = ql_inputs.batched_lengths(batch, 512, 32768, seed=6)
    case = ql_inputs.attention_case(batch, 32, 8, 128, lens, seed=4)
    got = gpu_attention(case, 32, 8, 128)
    rng = np.random.default_rng(batch)
    for b in rng.choice(batch, min(batch, 4), replace=False):
        sub = {k: case[k] for k in ("k_pool", "v_pool")}
        L = int(lens[b])
        k = ops.gather_paged(sub["k_pool"], case["block_tables"][b], L)
        v = ops.gather_paged(sub["v_pool"], case["block_tables"][b], L)
        want = ops.gqa_attention(case["q"][b], k, v, 1.0 / math.sqrt(128))
        check(got[b], want, f"b={b} L={L}")
