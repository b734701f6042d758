"""libql Python binding: q4_0 dense-transformer decode on one GB300.

Thin wrappers with the names of the C entry points (``include/ql.h``). Device buffers are
``torch`` CUDA tensors (PyTorch provides memory and streams only); every computation runs in
the CUDA library ``_build/libql.so``. Each wrapper raises :class:`QLError` on a non-zero
status.
"""
from __future__ import annotations

import ctypes

from ._lib import (QLError, QL_OK, QL_EINVAL, QL_ENOMEM, QL_ECUDA, QL_EPOOL, QL_ERANGE,
                   QL_EDEVICE, QL_ESTATE, QL_DTYPE_F32, QL_DTYPE_F16, QL_EPI_NONE,
                   QL_EPI_ADD_RESIDUAL, QL_EPI_SILU_MUL, QL_STEP_AUTO, QL_STEP_LAUNCHES,
                   QL_STEP_PERSISTENT, QL_OPT_STEP_KERNEL, QL_OPT_BARRIER_TIMEOUT_NS,
                   QL_OPT_TEST_BARRIER_EXTRA, QL_OPT_STEP_TRACE, QL_OPT_MERGE_TRACE, QL_BATCHED_MMA_SYNC, QL_BATCHED_TCGEN05,
                   QL_GEMV_ACT_INT16, QL_GEMV_ACT_INT8, QL_KV_F16, QL_KV_Q8_0_Q5_1,
                   QL_ATTN_MERGE_TICKET, QL_ATTN_MERGE_CLUSTER,
                   Q4Matrix, LayerDesc, ModelDesc,
                   StepArgs, SIGNATURES, LIB_PATH, lib, check, ptr, stream_ptr)

__all__ = [
    "QLError", "lib", "ql_q4_0_pack", "ql_q4_0_unpack", "ql_q4_0_pack_device", "ql_gemv_q4_0",
    "ql_q4_0_stream_bytes", "ql_q4_0_stream_pack", "ql_gemv_q4_0_stream",
    "ql_gemv_q4_0_stream_workspace_bytes", "ql_gemm_q4_0_stream", "ql_set_batched_gemv_form", "ql_set_gemv_activation_form",
    "ql_paged_attn_workspace_bytes", "ql_paged_attn_decode", "ql_paged_attn_decode_noalloc",
    "ql_paged_attn_chunk_workspace_bytes", "ql_paged_attn_chunk",
    "ql_kvq_record_bytes", "ql_kvq_write", "ql_paged_attn_decode_kvq",
    "ql_set_attn_merge_form", "ql_paged_attn_merge_form",
    "ql_kv_q8_0_row_bytes", "ql_kv_q5_1_row_bytes", "ql_kv_quantize_q8_0", "ql_kv_dequantize_q8_0",
    "ql_kv_quantize_q5_1", "ql_kv_dequantize_q5_1", "ql_kv_quantize_device", "ql_kv_dequantize_device",
    "ql_fused_norm_rope",
    "ql_rope_tables", "ql_check_device_error", "BlockPool", "SIGNATURES",
]


def ql_q4_0_pack(w, scales, quants):
    """Host codec: ``w`` f32 [rows, cols] numpy -> ``scales`` u16 [rows, cols/32], ``quants`` u8."""
    rows, cols = w.shape
    check(lib().ql_q4_0_pack(w.ctypes.data, rows, cols, scales.ctypes.data, quants.ctypes.data))


def ql_q4_0_unpack(scales, quants, w):
    rows, cols = w.shape
    check(lib().ql_q4_0_unpack(scales.ctypes.data, quants.ctypes.data, rows, cols, w.ctypes.data))


def ql_q4_0_pack_device(w, scales, quants, stream=None):
    rows, cols = w.shape
    check(lib().ql_q4_0_pack_device(ptr(w), rows, cols, ptr(scales), ptr(quants), stream_ptr(stream)))


def ql_gemv_q4_0(scales, quants, rows, cols, x, batch, y, y_dtype=QL_DTYPE_F32,
                 epilogue=QL_EPI_NONE, residual=None, stream=None):
    check(lib().ql_gemv_q4_0(ptr(scales), ptr(quants), rows, cols, ptr(x), batch, ptr(y), y_dtype,
                             epilogue, ptr(residual), stream_ptr(stream)))


def ql_q4_0_stream_bytes(rows, cols, silu=0):
    return int(lib().ql_q4_0_stream_bytes(rows, cols, silu))


def ql_q4_0_stream_pack(scales, quants, rows, cols, silu, out, stream=None):
    check(lib().ql_q4_0_stream_pack(ptr(scales), ptr(quants), rows, cols, silu, ptr(out), stream_ptr(stream)))


def ql_gemv_q4_0_stream_workspace_bytes(rows, cols, silu=0):
    return int(lib().ql_gemv_q4_0_stream_workspace_bytes(rows, cols, silu))


def ql_set_batched_gemv_form(form):
    """Tensor-core form of the batch 3-32 GEMV for this process; returns the previous form."""
    rc = int(lib().ql_set_batched_gemv_form(form))
    if rc < 0:
        check(rc)
    return rc


def ql_set_gemv_activation_form(form):
    """Activation form of the batch 1-2 GEMV for this process; returns the previous form."""
    rc = int(lib().ql_set_gemv_activation_form(form))
    if rc < 0:
        check(rc)
    return rc


def ql_set_attn_merge_form(form):
    """How attention merges its context splits, for this process; returns the previous form."""
    rc = int(lib().ql_set_attn_merge_form(form))
    if rc < 0:
        check(rc)
    return rc


def ql_paged_attn_merge_form(batch, n_heads, n_kv_heads, head_dim, max_blocks_per_seq):
    """The merge form an attention launch of this shape takes on the current device."""
    rc = int(lib().ql_paged_attn_merge_form(batch, n_heads, n_kv_heads, head_dim, max_blocks_per_seq))
    if rc < 0:
        check(rc)
    return rc


def ql_kv_q8_0_row_bytes(dim):
    return int(lib().ql_kv_q8_0_row_bytes(dim))


def ql_kv_q5_1_row_bytes(dim):
    return int(lib().ql_kv_q5_1_row_bytes(dim))


def _kv_quantize(fn, row_bytes, x):
    import numpy as np
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, dim = x.shape
    out = np.zeros((rows, row_bytes(dim)), dtype=np.uint8)
    check(fn(x.ctypes.data, rows, dim, out.ctypes.data))
    return out


def _kv_dequantize(fn, data, dim):
    import numpy as np
    data = np.ascontiguousarray(data, dtype=np.uint8)
    x = np.zeros((data.shape[0], dim), dtype=np.float32)
    check(fn(data.ctypes.data, data.shape[0], dim, x.ctypes.data))
    return x


def ql_kv_quantize_q8_0(x):
    """Host codec: f32 rows [n, dim] numpy -> q8_0 bytes [n, ql_kv_q8_0_row_bytes(dim)]."""
    return _kv_quantize(lib().ql_kv_quantize_q8_0, ql_kv_q8_0_row_bytes, x)


def ql_kv_dequantize_q8_0(data, dim):
    return _kv_dequantize(lib().ql_kv_dequantize_q8_0, data, dim)


def ql_kv_quantize_q5_1(x):
    """Host codec: f32 rows [n, dim] numpy -> q5_1 bytes [n, ql_kv_q5_1_row_bytes(dim)]."""
    return _kv_quantize(lib().ql_kv_quantize_q5_1, ql_kv_q5_1_row_bytes, x)


def ql_kv_dequantize_q5_1(data, dim):
    return _kv_dequantize(lib().ql_kv_dequantize_q5_1, data, dim)


def ql_kv_quantize_device(x, out, fmt="q8_0", stream=None):
    """Device codec: ``x`` f32 [rows, dim] CUDA tensor -> ``out`` uint8 [rows, row bytes]."""
    fn = lib().ql_kv_quantize_q8_0_device if fmt == "q8_0" else lib().ql_kv_quantize_q5_1_device
    check(fn(ptr(x), x.shape[0], x.shape[1], ptr(out), stream_ptr(stream)))


def ql_kv_dequantize_device(data, x, fmt="q8_0", stream=None):
    """Device codec: ``data`` uint8 [rows, row bytes] -> ``x`` f32 [rows, dim] CUDA tensor."""
    fn = lib().ql_kv_dequantize_q8_0_device if fmt == "q8_0" else lib().ql_kv_dequantize_q5_1_device
    check(fn(ptr(data), x.shape[0], x.shape[1], ptr(x), stream_ptr(stream)))


def ql_gemv_q4_0_stream(w_stream, rows, cols, x, batch, y, epilogue=QL_EPI_NONE, workspace=None, stream=None):
    """``workspace``: a zero-filled device byte tensor of ql_gemv_q4_0_stream_workspace_bytes
    (batch 3-32; None at batch 1-2)."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(lib().ql_gemv_q4_0_stream(ptr(w_stream), rows, cols, ptr(x), batch, ptr(y), epilogue,
                                    ptr(workspace), nbytes, stream_ptr(stream)))


def ql_gemm_q4_0_stream(w_stream, rows, cols, x, n_tokens, y, epilogue=QL_EPI_NONE, stream=None):
    """The prompt-chunk GEMM over the tile stream copy: ``x`` f16 [n_tokens, cols]."""
    check(lib().ql_gemm_q4_0_stream(ptr(w_stream), rows, cols, ptr(x), n_tokens, ptr(y), epilogue,
                                    stream_ptr(stream)))


def ql_paged_attn_chunk_workspace_bytes(n_tokens, n_heads, n_kv_heads, head_dim):
    return int(lib().ql_paged_attn_chunk_workspace_bytes(n_tokens, n_heads, n_kv_heads, head_dim))


def ql_paged_attn_chunk(q, k_pool, v_pool, block_table, position, n_tokens, n_heads, n_kv_heads, head_dim,
                        block_size, max_blocks_per_seq, num_blocks, scale, out, workspace, stream=None):
    """Causal attention of a prefill chunk: ``q`` f16 [n_tokens][n_heads][head_dim] at positions
    ``position[0] + t`` (int32 [1] device) over the sequence's ``block_table``."""
    check(lib().ql_paged_attn_chunk(ptr(q), ptr(k_pool), ptr(v_pool), ptr(block_table), ptr(position), n_tokens,
                                    n_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                                    scale, ptr(out), ptr(workspace), workspace.numel() * workspace.element_size(),
                                    stream_ptr(stream)))


def ql_paged_attn_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, block_size, max_blocks_per_seq):
    return int(lib().ql_paged_attn_workspace_bytes(batch, n_heads, n_kv_heads, head_dim, block_size,
                                                   max_blocks_per_seq))


def ql_paged_attn_decode(q, k_pool, v_pool, block_tables, context_lens, batch, n_heads, n_kv_heads,
                         head_dim, block_size, max_blocks_per_seq, num_blocks, scale, out,
                         workspace, stream=None):
    check(lib().ql_paged_attn_decode(ptr(q), ptr(k_pool), ptr(v_pool), ptr(block_tables),
                                     ptr(context_lens), batch, n_heads, n_kv_heads, head_dim,
                                     block_size, max_blocks_per_seq, num_blocks, scale, ptr(out),
                                     ptr(workspace), workspace.numel() * workspace.element_size(),
                                     stream_ptr(stream)))


def ql_kvq_record_bytes(head_dim):
    return int(lib().ql_kvq_record_bytes(head_dim))


def ql_kvq_write(k, v, slots, n_kv_heads, head_dim, pool, num_blocks, stream=None):
    """Quantise f32 rows ``k``, ``v`` [n, n_kv, hd] into one layer's pool at physical ``slots``
    (int64 [n], block * 16 + offset)."""
    check(lib().ql_kvq_write(ptr(k), ptr(v), ptr(slots), slots.numel(), n_kv_heads, head_dim, ptr(pool),
                             num_blocks, stream_ptr(stream)))


def ql_paged_attn_decode_kvq(q, pool, block_tables, context_lens, batch, n_heads, n_kv_heads, head_dim,
                             block_size, max_blocks_per_seq, num_blocks, scale, out, workspace, stream=None):
    check(lib().ql_paged_attn_decode_kvq(ptr(q), ptr(pool), ptr(block_tables), ptr(context_lens), batch, n_heads,
                                         n_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                                         ptr(out), ptr(workspace), workspace.numel() * workspace.element_size(),
                                         stream_ptr(stream)))


def ql_paged_attn_decode_noalloc(q, k_pool, v_pool, block_tables, context_lens, batch, n_heads,
                                 n_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks,
                                 scale, out, stream=None):
    """Attention whose split-K scratch is the library's fixed 8 MiB device array (no workspace
    argument, no device allocation); see include/ql.h for its limits."""
    check(lib().ql_paged_attn_decode_noalloc(ptr(q), ptr(k_pool), ptr(v_pool), ptr(block_tables),
                                             ptr(context_lens), batch, n_heads, n_kv_heads,
                                             head_dim, block_size, max_blocks_per_seq, num_blocks,
                                             scale, ptr(out), stream_ptr(stream)))


def ql_fused_norm_rope(qkv, q_norm, k_norm, cos_t, sin_t, positions, active, eps, batch, n_heads,
                       n_kv_heads, head_dim, q_out, k_pool, v_pool, block_tables,
                       max_blocks_per_seq, block_size, num_blocks, max_position, stream=None):
    check(lib().ql_fused_norm_rope(ptr(qkv), ptr(q_norm), ptr(k_norm), ptr(cos_t), ptr(sin_t),
                                   ptr(positions), ptr(active), eps, batch, n_heads, n_kv_heads,
                                   head_dim, ptr(q_out), ptr(k_pool), ptr(v_pool), ptr(block_tables),
                                   max_blocks_per_seq, block_size, num_blocks, max_position,
                                   stream_ptr(stream)))


def ql_rope_tables(cos_t, sin_t, theta):
    """Host: fill numpy f32 ``cos_t``, ``sin_t`` [max_position, head_dim/2]."""
    n, half = cos_t.shape
    check(lib().ql_rope_tables(cos_t.ctypes.data, sin_t.ctypes.data, n, 2 * half, theta))


def ql_check_device_error(model=None):
    h = model.handle if model is not None else None
    check(lib().ql_check_device_error(h))


class BlockPool:
    """Host KV block allocator (free list first, then bump; QL_EPOOL when exhausted)."""

    def __init__(self, num_blocks: int):
        h = ctypes.c_void_p()
        check(lib().ql_block_pool_create(num_blocks, ctypes.byref(h)))
        self.handle = h.value

    def alloc(self) -> int:
        out = ctypes.c_int32()
        check(lib().ql_block_pool_alloc(self.handle, ctypes.byref(out)))
        return int(out.value)

    def free(self, ids):
        arr = (ctypes.c_int32 * len(ids))(*[int(i) for i in ids])
        check(lib().ql_block_pool_free(self.handle, arr, len(ids)))

    def in_use(self) -> int:
        return int(lib().ql_block_pool_in_use(self.handle))

    def close(self):
        if self.handle:
            lib().ql_block_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
