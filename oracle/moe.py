"""The routed-expert (MoE) feed-forward block of a Qwen3-MoE-style layer, in f64 (test
infrastructure; see the package docstring).

inferencelayer ``cuda_llm.rs``: ``Cfg`` (``num_experts``, ``topk``, ``moe_inter``,
``norm_topk``; "Qwen3 MoE has NO shared expert"), the expert weights as loaded (gate|up
interleaved per expert: expert e owns rows ``[e 2mi, e 2mi + mi)`` = gate and the next ``mi`` =
up of one q4_0 matrix; the down rows of expert e are ``[e hidden, (e + 1) hidden)`` of another),
and the "MLP / MoE" branch of ``CudaQwen3::step``: router logits = ``router @ hn`` (f32 router
weights, not quantised), a top-k selection with weights, per selected expert
``silu(gate) * up`` and the down projection, then the weighted combination added to the residual.

The page does not print its ``topk`` kernel. Reading taken (the Qwen3-MoE router): the
probabilities are the softmax of the logits over all experts, the k largest are selected (the
lowest expert index first among equal probabilities), and with ``norm_topk`` their weights are
divided by their sum; without it they are the softmax probabilities themselves.
"""
from __future__ import annotations

import numpy as np

from . import ops
from .q4_0 import dequantize


def route(logits, k: int, norm_topk: bool = True):
    """``logits [E]`` -> (selected experts ``[k]`` by falling probability, weights ``[k]``)."""
    logits = np.asarray(logits, dtype=np.float64)
    p = ops.softmax(logits)
    order = np.argsort(-p, kind="stable")        # stable: equal probabilities keep index order
    idx = order[:k]
    w = p[idx]
    if norm_topk:
        w = w / w.sum()
    return idx, w


def expert_rows(q4, first: int, count: int) -> np.ndarray:
    """Rows ``[first, first + count)`` of a q4_0 matrix, dequantised (f64)."""
    scales, quants = q4
    return dequantize(scales[first:first + count], quants[first:first + count])


def moe_ffn(hn, router, w1, w2, cfg) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """The MoE block for one normalised input ``hn [hidden]``: returns (the block's output to add
    to the residual ``[hidden]``, the selected experts, their weights)."""
    hn = np.asarray(hn, dtype=np.float64)
    mi, hidden = cfg.moe_inter, cfg.hidden
    logits = np.asarray(router, dtype=np.float64) @ hn
    idx, wts = route(logits, cfg.topk, cfg.norm_topk)
    out = np.zeros(hidden)
    for e, we in zip(idx, wts):
        gu = ops.gemv(expert_rows(w1, int(e) * 2 * mi, 2 * mi), hn[None, :])[0]
        act = ops.swiglu(gu[:mi], gu[mi:])
        out += we * ops.gemv(expert_rows(w2, int(e) * hidden, hidden), act[None, :])[0]
    return out, idx, wts
