"""ctypes binding of libql (argument marshalling only; every step runs in the CUDA library).

The functions here carry the names of the C entry points in ``include/ql.h`` and take device
buffers as ``torch`` tensors (or raw integer addresses). A missing library raises at import of
:func:`lib`; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p, c_char_p

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libql.so")

QL_OK, QL_EINVAL, QL_ENOMEM, QL_ECUDA, QL_EPOOL, QL_ERANGE, QL_EDEVICE, QL_ESTATE = 0, -1, -2, -3, -4, -5, -6, -7
QL_DTYPE_F32, QL_DTYPE_F16 = 0, 1
QL_EPI_NONE, QL_EPI_ADD_RESIDUAL, QL_EPI_SILU_MUL = 0, 1, 2
QL_STEP_AUTO, QL_STEP_LAUNCHES, QL_STEP_PERSISTENT = 0, 1, 2
QL_OPT_STEP_KERNEL, QL_OPT_BARRIER_TIMEOUT_NS, QL_OPT_TEST_BARRIER_EXTRA, QL_OPT_STEP_TRACE = 1, 2, 3, 4
QL_OPT_MERGE_TRACE = 5
QL_BATCHED_MMA_SYNC, QL_BATCHED_TCGEN05 = 0, 1
QL_GEMV_ACT_INT16, QL_GEMV_ACT_INT8 = 0, 1
QL_KV_F16, QL_KV_Q8_0_Q5_1 = 0, 1
QL_ATTN_MERGE_TICKET, QL_ATTN_MERGE_CLUSTER = 0, 1


class QLError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_status_name(status)}: {msg}")
        self.status = status


class Q4Matrix(ctypes.Structure):
    _fields_ = [("scales", c_void_p), ("quants", c_void_p), ("rows", c_int64), ("cols", c_int64)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("attn_norm", c_void_p), ("ffn_norm", c_void_p), ("q_norm", c_void_p),
                ("k_norm", c_void_p), ("qkv", Q4Matrix), ("o", Q4Matrix), ("gate_up", Q4Matrix),
                ("down", Q4Matrix), ("router", c_void_p), ("experts_gate_up", Q4Matrix),
                ("experts_down", Q4Matrix)]


class ModelDesc(ctypes.Structure):
    _fields_ = [("hidden", c_int64), ("n_layers", c_int64), ("n_heads", c_int64),
                ("n_kv_heads", c_int64), ("head_dim", c_int64), ("intermediate", c_int64),
                ("vocab", c_int64), ("eps", c_float), ("rope_theta", c_double),
                ("embed", c_void_p), ("final_norm", c_void_p), ("lm_head", Q4Matrix),
                ("layers", POINTER(LayerDesc)), ("k_pool", c_void_p), ("v_pool", c_void_p),
                ("num_blocks", c_int64), ("block_size", c_int), ("max_batch", c_int64),
                ("max_blocks_per_seq", c_int64), ("kv_format", c_int), ("kvq_pool", c_void_p),
                ("num_experts", c_int64), ("topk", c_int64), ("moe_inter", c_int64), ("norm_topk", c_int)]


class StepArgs(ctypes.Structure):
    _fields_ = [("batch", c_int64), ("tokens", c_void_p), ("positions", c_void_p),
                ("block_tables", c_void_p), ("active", c_void_p), ("logits", c_void_p),
                ("next_tokens", c_void_p), ("out_tokens", c_void_p), ("out_stride", c_int64)]


# name -> (restype, argtypes); the complete exported surface of include/ql.h
SIGNATURES = {
    "ql_status_str": (c_char_p, [c_int]),
    "ql_last_error": (c_char_p, []),
    "ql_version": (c_int, []),
    "ql_q4_0_pack": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "ql_q4_0_unpack": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_void_p]),
    "ql_q4_0_pack_device": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_void_p, c_void_p]),
    "ql_gemv_q4_0": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_void_p, c_int64, c_void_p,
                             c_int, c_int, c_void_p, c_void_p]),
    "ql_q4_0_stream_bytes": (c_int64, [c_int64, c_int64, c_int]),
    "ql_q4_0_stream_pack": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int, c_void_p, c_void_p]),
    "ql_gemv_q4_0_stream": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_int64, c_void_p, c_int, c_void_p,
                                    c_int64, c_void_p]),
    "ql_gemv_q4_0_stream_workspace_bytes": (c_int64, [c_int64, c_int64, c_int]),
    "ql_gemm_q4_0_stream": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_int64, c_void_p, c_int, c_void_p]),
    "ql_set_batched_gemv_form": (c_int, [c_int]),
    "ql_set_gemv_activation_form": (c_int, [c_int]),
    "ql_kvq_record_bytes": (c_int64, [c_int]),
    "ql_prefill_chunk": (c_int, [c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "ql_kvq_write": (c_int, [c_void_p, c_void_p, c_void_p, c_int64, c_int, c_int, c_void_p, c_int64, c_void_p]),
    "ql_paged_attn_decode_kvq": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int, c_int, c_int, c_int,
                                         c_int64, c_int64, c_float, c_void_p, c_void_p, c_size_t, c_void_p]),
    "ql_paged_attn_workspace_bytes": (c_size_t, [c_int64, c_int, c_int, c_int, c_int, c_int64]),
    "ql_paged_attn_chunk_workspace_bytes": (c_size_t, [c_int64, c_int, c_int, c_int]),
    "ql_paged_attn_chunk": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_int, c_int,
                                    c_int, c_int, c_int64, c_int64, c_float, c_void_p, c_void_p, c_size_t,
                                    c_void_p]),
    "ql_paged_attn_decode": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64,
                                     c_int, c_int, c_int, c_int, c_int64, c_int64, c_float,
                                     c_void_p, c_void_p, c_size_t, c_void_p]),
    "ql_paged_attn_decode_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                             c_int64, c_int, c_int, c_int, c_int, c_int64, c_int64,
                                             c_float, c_void_p, c_void_p]),
    "ql_set_attn_merge_form": (c_int, [c_int]),
    "ql_kv_q8_0_row_bytes": (c_int64, [c_int64]),
    "ql_kv_q5_1_row_bytes": (c_int64, [c_int64]),
    "ql_kv_quantize_q8_0": (c_int, [c_void_p, c_int64, c_int64, c_void_p]),
    "ql_kv_dequantize_q8_0": (c_int, [c_void_p, c_int64, c_int64, c_void_p]),
    "ql_kv_quantize_q5_1": (c_int, [c_void_p, c_int64, c_int64, c_void_p]),
    "ql_kv_dequantize_q5_1": (c_int, [c_void_p, c_int64, c_int64, c_void_p]),
    "ql_kv_quantize_q8_0_device": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "ql_kv_dequantize_q8_0_device": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "ql_kv_quantize_q5_1_device": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "ql_kv_dequantize_q5_1_device": (c_int, [c_void_p, c_int64, c_int64, c_void_p, c_void_p]),
    "ql_paged_attn_merge_form": (c_int, [c_int64, c_int, c_int, c_int, c_int64]),
    "ql_fused_norm_rope": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_float, c_int64, c_int, c_int, c_int, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_int64, c_int, c_int64, c_int64,
                                   c_void_p]),
    "ql_rope_tables": (c_int, [c_void_p, c_void_p, c_int64, c_int, c_double]),
    "ql_model_create": (c_int, [POINTER(ModelDesc), POINTER(c_void_p)]),
    "ql_model_destroy": (c_int, [c_void_p]),
    "ql_model_set_option": (c_int, [c_void_p, c_int, c_int64]),
    "ql_model_persistent_max_batch": (c_int64, [c_void_p]),
    "ql_decode_step": (c_int, [c_void_p, POINTER(StepArgs), c_void_p]),
    "ql_decode_graph_capture": (c_int, [c_void_p, POINTER(StepArgs), c_void_p]),
    "ql_decode_graph_replay": (c_int, [c_void_p, c_int64, c_int, c_void_p]),
    "ql_decode_graph_step_host": (c_int, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p]),
    "ql_check_device_error": (c_int, [c_void_p]),
    "ql_block_pool_create": (c_int, [c_int64, POINTER(c_void_p)]),
    "ql_block_pool_destroy": (c_int, [c_void_p]),
    "ql_block_pool_alloc": (c_int, [c_void_p, POINTER(c_int32)]),
    "ql_block_pool_free": (c_int, [c_void_p, c_void_p, c_int64]),
    "ql_block_pool_in_use": (c_int64, [c_void_p]),
}

_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded libql (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libql is not built ({LIB_PATH} missing): run "
                              "`python -m quantized_transformer_decode_ql_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _status_name(s: int) -> str:
    try:
        return lib().ql_status_str(s).decode()
    except Exception:
        return f"status {s}"


def check(status: int) -> int:
    if status != QL_OK:
        raise QLError(status, lib().ql_last_error().decode())
    return status


def ptr(x) -> int | None:
    """Device/host address of a tensor, an int address, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def stream_ptr(stream=None) -> int | None:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream
