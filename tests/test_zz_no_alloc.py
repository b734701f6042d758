"""The no-allocation attention entry point (collected last on purpose).

ql_paged_attn_decode_noalloc is for callers that cannot allocate device memory - for example a
plugin living inside an application whose memory pool owns the whole GPU, or a tight loop that
cannot afford cudaMalloc/cudaFree and the device synchronisation they can cause. It takes no
workspace: its split-K scratch is a fixed 8 MiB array built into the library.

It runs the same kernel with the same split layout as ql_paged_attn_decode, so its outputs must
be bit-identical to that entry point's, on two calls in a row (the second with other shapes, so
that whatever the first call left in the shared array cannot leak into the second), under both
merge forms. The first call is also compared with the oracle at the attention tests' tolerance
(``|o - o_ref| <= 2e-3 + 1e-2 |o_ref|``). A misaligned pool is refused on the host.
"""
import math

import numpy as np
import pytest
import torch

import ql_inputs
from oracle import ops

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu


def both_paths(case, n_heads, n_kv, hd):
    ql = lib()
    B = case["q"].shape[0]
    mb = case["max_blocks"]
    args = (dev(case["q"]), dev(case["k_pool"]), dev(case["v_pool"]), dev(case["block_tables"]),
            dev(case["lens"]))
    common = (B, n_heads, n_kv, hd, 16, mb, case["num_blocks"], 1.0 / math.sqrt(hd))
    ref = torch.full((B, n_heads * hd), float("nan"), dtype=torch.float16, device="cuda")
    ws = torch.zeros(ql.ql_paged_attn_workspace_bytes(B, n_heads, n_kv, hd, 16, mb),
                     dtype=torch.uint8, device="cuda")
    ql.ql_paged_attn_decode(*args, *common, ref, ws)
    got = torch.full_like(ref, float("nan"))
    ql.ql_paged_attn_decode_noalloc(*args, *common, got)
    torch.cuda.synchronize()
    return got.float().cpu().numpy(), ref.float().cpu().numpy()


def against_oracle(got, case, n_heads, hd, what):
    B = case["q"].shape[0]
    want = ops.paged_attention(case["q"], case["k_pool"], case["v_pool"], case["block_tables"],
                               case["lens"], 1.0 / math.sqrt(hd)).reshape(B, n_heads * hd)
    assert not np.any(np.isnan(got)), what
    err = np.abs(got - want)
    assert np.all(err <= 2e-3 + 1e-2 * np.abs(want)), f"{what}: max err {err.max():.3e}"


@pytest.mark.parametrize("form", ["ticket", "cluster"])
def test_noalloc_matches_workspace_path_on_two_calls_in_a_row(form):
    ql = lib()
    prev = ql.ql_set_attn_merge_form(ql.QL_ATTN_MERGE_CLUSTER if form == "cluster" else ql.QL_ATTN_MERGE_TICKET)
    try:
        # call 1: batch 1 with several splits of its (sequence, kv head): the merge form under
        # test runs (the cluster form where the device can hold the clusters)
        lens1 = [3000]
        case1 = ql_inputs.attention_case(1, 32, 8, 128, lens1, seed=21)
        got1, ref1 = both_paths(case1, 32, 8, 128)
        assert np.array_equal(got1, ref1), "first call: noalloc and workspace paths differ"
        against_oracle(got1, case1, 32, 128, "first call")
        # call 2: other batch, heads, head_dim and lengths, reusing the same built-in scratch
        lens2 = [1, 17, 333, 2049, 64]
        case2 = ql_inputs.attention_case(5, 16, 2, 64, lens2, seed=22)
        got2, ref2 = both_paths(case2, 16, 2, 64)
        assert np.array_equal(got2, ref2), "second call: noalloc and workspace paths differ"
        # call 3: batch 3 with long contexts (the ticket merge at any setting)
        lens3 = [3000, 700, 4100]
        case3 = ql_inputs.attention_case(3, 32, 8, 128, lens3, seed=23)
        got3, ref3 = both_paths(case3, 32, 8, 128)
        assert np.array_equal(got3, ref3), "third call: noalloc and workspace paths differ"
    finally:
        ql.ql_set_attn_merge_form(prev)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    ql = lib()
    # 2000 sequences x 32 heads of split partials need far more than the built-in 8 MiB
    t = torch.zeros(16, dtype=torch.float16, device="cuda")
    i = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(ql.QLError) as e:
        ql.ql_paged_attn_decode_noalloc(t, t, t, i, i, 2000, 32, 8, 128, 16, 4, 4, 0.1, t)
    assert e.value.status == ql.QL_EINVAL and "8388608" in str(e.value)


def test_noalloc_rejects_misaligned_buffers_on_the_host():
    """A pool 2 bytes off a 16-byte boundary (or q off a 4-byte one) is QL_EINVAL; the kernel
    is never launched, so nothing on the device reads through the misaligned pointer."""
    ql = lib()
    case = ql_inputs.attention_case(1, 4, 2, 64, [40], seed=24)
    q = dev(case["q"])
    kp = dev(case["k_pool"])
    vp = dev(case["v_pool"])
    bt, cl = dev(case["block_tables"]), dev(case["lens"])
    out = torch.zeros((1, 4 * 64), dtype=torch.float16, device="cuda")
    nb, mb = case["num_blocks"], case["max_blocks"]
    kp_off = kp.reshape(-1)[1:]     # data pointer 2 bytes past a 16-byte boundary
    with pytest.raises(ql.QLError) as e:
        ql.ql_paged_attn_decode_noalloc(q, kp_off, vp, bt, cl, 1, 4, 2, 64, 16, mb, nb, 0.125, out)
    assert e.value.status == ql.QL_EINVAL and "aligned" in str(e.value)
    q_off = q.reshape(-1)[1:]       # 2 bytes past a 4-byte boundary
    with pytest.raises(ql.QLError) as e:
        ql.ql_paged_attn_decode_noalloc(q_off, kp, vp, bt, cl, 1, 4, 2, 64, 16, mb, nb, 0.125, out)
    assert e.value.status == ql.QL_EINVAL
    torch.cuda.synchronize()
    assert int(out.abs().sum().item()) == 0   # nothing was written
