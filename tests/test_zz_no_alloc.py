"""The no-allocation attention entry point (collected last on purpose).

ql_paged_attn_decode_noalloc is for callers that cannot allocate device memory - for example a
plugin living inside an application whose memory pool owns the whole GPU, or a tight loop that
cannot afford cudaMalloc/cudaFree and the device synchronisation they can cause. It takes no
workspace: its split-K scratch is a fixed 8 MiB array built into the library.

Here it must give the same outputs as ql_paged_attn_decode (same tolerance as the attention
tests: |o - o_ref| <= 2e-3 + 1e-2 |o_ref|) on two calls in a row, the second one with other
shapes, so that whatever the first call left in the shared array cannot leak into the second.
"""
import math

import numpy as np
import pytest
import torch

import ql_inputs

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


def check(got, want, what):
    assert not np.any(np.isnan(got)), what
    err = np.abs(got - want)
    assert np.all(err <= 2e-3 + 1e-2 * np.abs(want)), f"{what}: max err {err.max():.3e}"


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row():
    # call 1: long contexts, several splits per (sequence, kv head) -> the ticket merge runs
    lens1 = [3000, 700, 4100]
    case1 = ql_inputs.attention_case(3, 32, 8, 128, lens1, seed=21)
    got1, ref1 = both_paths(case1, 32, 8, 128)
    check(got1, ref1, "first call")
    # call 2: other heads, head_dim and lengths, reusing the same built-in scratch
    lens2 = [1, 17, 333, 2049, 64]
    case2 = ql_inputs.attention_case(5, 16, 2, 64, lens2, seed=22)
    got2, ref2 = both_paths(case2, 16, 2, 64)
    check(got2, ref2, "second call")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    ql = lib()
    # 2000 sequences x 32 heads of split partials need far more than the built-in 8 MiB
    t = torch.zeros(16, dtype=torch.float16, device="cuda")
    i = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(ql.QLError) as e:
        ql.ql_paged_attn_decode_noalloc(t, t, t, i, i, 2000, 32, 8, 128, 16, 4, 4, 0.1, t)
    assert e.value.status == ql.QL_EINVAL and "8388608" in str(e.value)
