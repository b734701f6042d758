"""The C ABI on the CPU: the library builds, loads and exports every symbol of include/ql.h;
host-side parts (q4_0 codec, RoPE tables, block allocator, argument validation) agree with the
oracle. No GPU call is made here."""
import ctypes
import os
import re

import numpy as np
import pytest

import ql_inputs
from oracle import q4_0 as oq, ops
from oracle.blockpool import BlockPool as OraclePool, PoolExhausted

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ql():
    from quantized_transformer_decode_ql_gb300 import build
    build.build()
    import quantized_transformer_decode_ql_gb300 as q
    return q


def header_functions():
    src = open(os.path.join(ROOT, "include", "ql.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(ql_\w+)\s*\(", src))


def test_header_symbols_exported(ql):
    declared = header_functions()
    assert len(declared) >= 20
    L = ql.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert declared == set(ql.SIGNATURES), declared ^ set(ql.SIGNATURES)
    assert L.ql_version() == 1
    assert L.ql_status_str(-4) == b"QL_EPOOL"


def test_host_codec_bit_exact_with_oracle(ql):
    for (rows, cols, seed) in [(3, 32, 0), (17, 96, 1), (64, 4096, 2), (5, 12288, 3)]:
        w = ql_inputs.gemv_weight(rows, cols, seed=seed)
        s = np.empty((rows, cols // 32), np.uint16)
        q = np.empty((rows, cols // 32, 16), np.uint8)
        ql.ql_q4_0_pack(w, s, q)
        s_ref, q_ref = oq.quantize(w)
        assert np.array_equal(s, s_ref) and np.array_equal(q, q_ref)
        back = np.empty_like(w)
        ql.ql_q4_0_unpack(s, q, back)
        assert np.array_equal(back.astype(np.float64), oq.dequantize(s_ref, q_ref))


def test_host_codec_golden_and_edges(ql):
    from test_oracle_q4_0 import load_golden
    for name, x, scale, qb in load_golden():
        s = np.empty((1, 1), np.uint16)
        q = np.empty((1, 1, 16), np.uint8)
        ql.ql_q4_0_pack(x[None, :].copy(), s, q)
        assert int(s[0, 0]) == scale and np.array_equal(q[0, 0], qb), name
    # wide dynamic range: scales near the f16 subnormal boundary and large ones
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((64, 64)) * np.logspace(-6, 3, 64)[:, None]).astype(np.float32)
    s = np.empty((64, 2), np.uint16)
    q = np.empty((64, 2, 16), np.uint8)
    ql.ql_q4_0_pack(w, s, q)
    s_ref, q_ref = oq.quantize(w)
    assert np.array_equal(s, s_ref) and np.array_equal(q, q_ref)


def test_host_codec_errors(ql):
    s = np.empty((1, 1), np.uint16)
    q = np.empty((1, 1, 16), np.uint8)
    bad = np.zeros((1, 32), np.float32)
    bad[0, 5] = np.inf
    with pytest.raises(ql.QLError) as e:
        ql.ql_q4_0_pack(bad, s, q)
    assert e.value.status == ql.QL_EINVAL
    big = np.zeros((1, 32), np.float32)
    big[0, 0] = 1e6
    with pytest.raises(ql.QLError):
        ql.ql_q4_0_pack(big, s, q)
    assert ql.lib().ql_q4_0_pack(None, 1, 32, None, None) == ql.QL_EINVAL
    assert ql.lib().ql_q4_0_pack(bad.ctypes.data, 1, 33, s.ctypes.data, q.ctypes.data) == ql.QL_EINVAL


def test_rope_tables_match_oracle_angles(ql):
    hd, n, theta = 128, 300, 1e6
    c = np.empty((n, hd // 2), np.float32)
    s = np.empty((n, hd // 2), np.float32)
    ql.ql_rope_tables(c, s, theta)
    for p in (0, 1, 17, 299):
        ang = ops.rope_angles(p, hd, theta)
        np.testing.assert_allclose(c[p], np.cos(ang), rtol=0, atol=1e-7)
        np.testing.assert_allclose(s[p], np.sin(ang), rtol=0, atol=1e-7)


def test_block_pool_matches_oracle_rule(ql):
    rng = np.random.default_rng(0)
    mine, ref = ql.BlockPool(40), OraclePool(40)
    live = []
    for step in range(400):
        if live and rng.random() < 0.45:
            k = int(rng.integers(1, min(5, len(live)) + 1))
            ids = [live.pop(int(rng.integers(len(live)))) for _ in range(k)]
            mine.free(ids)
            ref.release(ids)
        else:
            try:
                want = ref.alloc()
            except PoolExhausted:
                with pytest.raises(ql.QLError) as e:
                    mine.alloc()
                assert e.value.status == ql.QL_EPOOL
                continue
            got = mine.alloc()
            assert got == want
            live.append(got)
        assert mine.in_use() == ref.in_use()
    with pytest.raises(ql.QLError) as e:
        mine.free([999])
    assert e.value.status == ql.QL_ERANGE


def test_argument_validation_without_gpu(ql):
    L = ql.lib()
    assert L.ql_gemv_q4_0(None, None, 4, 32, None, 1, None, 0, 0, None, None) == ql.QL_EINVAL
    assert L.ql_gemv_q4_0(1, 1, 4, 33, 1, 1, 1, 0, 0, None, None) == ql.QL_EINVAL
    assert L.ql_gemv_q4_0(1, 1, 4, 32, 1, 0, 1, 0, 0, None, None) == ql.QL_EINVAL
    assert L.ql_gemv_q4_0(1, 1, 4, 32, 1, 1, 1, 0, 9, None, None) == ql.QL_EINVAL
    assert L.ql_paged_attn_decode(None, None, None, None, None, 1, 4, 2, 64, 16, 4, 4, 0.1,
                                  None, None, 0, None) == ql.QL_EINVAL
    assert L.ql_fused_norm_rope(*([None] * 7), 1e-6, 1, 4, 2, 64, *([None] * 4), 4, 16, 4, 64,
                                None) == ql.QL_EINVAL
    assert L.ql_model_create(None, None) == ql.QL_EINVAL
    assert L.ql_decode_graph_replay(None, 1, 1, None) == ql.QL_EINVAL
    assert L.ql_decode_graph_step_host(None, 1, None, None, None) == ql.QL_EINVAL
    assert L.ql_model_set_option(None, ql.QL_OPT_STEP_KERNEL, ql.QL_STEP_AUTO) == ql.QL_EINVAL
    assert L.ql_model_persistent_max_batch(None) == 0
    assert L.ql_q4_0_stream_pack(None, None, 16, 128, 0, None, None) == ql.QL_EINVAL
    assert L.ql_gemv_q4_0_stream(None, 16, 128, None, 1, None, 0, None, 0, None) == ql.QL_EINVAL
    assert L.ql_block_pool_create(0, ctypes.byref(ctypes.c_void_p())) == ql.QL_EINVAL
    assert ql.ql_paged_attn_workspace_bytes(0, 4, 2, 64, 16, 4) == 0


def test_stream_layout_sizes(ql):
    """Tile stream bytes: 16-row tiles (SiLU*up: 8 gate + 8 up rows) x cols/128 units of 1152 B;
    0 for shapes the layout does not take."""
    assert ql.ql_q4_0_stream_bytes(24576, 4096, 1) == 24576 * 4096 * 18 // 32
    assert ql.ql_q4_0_stream_bytes(4096, 12288, 0) == 4096 * 12288 * 18 // 32
    assert ql.ql_q4_0_stream_bytes(17, 128, 0) == 2 * 1152
    assert ql.ql_q4_0_stream_bytes(18, 128, 1) == 2 * 1152
    assert ql.ql_q4_0_stream_bytes(16, 96, 0) == 0
    assert ql.ql_q4_0_stream_bytes(15, 128, 1) == 0
    assert ql.ql_q4_0_stream_bytes(0, 128, 0) == 0


def test_stream_workspace_bad_shapes(ql):
    """The batched GEMV's workspace size is 0 for shapes it does not take (no device needed)."""
    assert ql.ql_gemv_q4_0_stream_workspace_bytes(16, 96, 0) == 0
    assert ql.ql_gemv_q4_0_stream_workspace_bytes(16, 1152, 0) == 0
    assert ql.ql_gemv_q4_0_stream_workspace_bytes(15, 1024, 1) == 0


def test_batched_gemv_form_switch(ql):
    """The batch 3-32 GEMV form is a process-wide choice: unknown forms are rejected, the
    previous form is returned (no device needed)."""
    assert ql.lib().ql_set_batched_gemv_form(7) == ql.QL_EINVAL
    prev = ql.ql_set_batched_gemv_form(ql.QL_BATCHED_TCGEN05)
    assert prev in (ql.QL_BATCHED_MMA_SYNC, ql.QL_BATCHED_TCGEN05)
    assert ql.ql_set_batched_gemv_form(prev) == ql.QL_BATCHED_TCGEN05


def test_attn_merge_form_switch(ql):
    """The attention merge form is a process-wide choice: unknown forms are rejected, the
    previous form is returned (no device needed)."""
    assert ql.lib().ql_set_attn_merge_form(5) == ql.QL_EINVAL
    prev = ql.ql_set_attn_merge_form(ql.QL_ATTN_MERGE_TICKET)
    assert prev in (ql.QL_ATTN_MERGE_TICKET, ql.QL_ATTN_MERGE_CLUSTER)
    assert ql.ql_set_attn_merge_form(prev) == ql.QL_ATTN_MERGE_TICKET
    assert ql.lib().ql_paged_attn_merge_form(1, 32, 8, 96, 16) == ql.QL_EINVAL
