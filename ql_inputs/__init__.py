"""Seeded synthetic inputs shared by the oracle and the CUDA path.

This module only draws random numbers and describes shapes. It holds none of the
decode method's arithmetic (no quantisation, no normalisation, no attention): both
the oracle and the CUDA library consume the arrays produced here and do their own
work on them.

Workloads follow the dense Qwen3-style decode the pages describe (inferencelayer
``cuda_llm.rs``, ``Cfg`` and ``CudaQwen3::load``): random-init weights drawn as
N(0, 0.02) f32, norm weights as 1 + N(0, 0.1) f32, an f32 embedding table, an
untied lm_head, and an f16 KV cache whose pre-filled context (where a workload
starts from one) is N(0, 1) f16.

Tensor layout conventions (an input format, not a computation):

* ``wqkv``  ``[(n_heads + 2*n_kv_heads) * head_dim, hidden]`` - rows q | k | v.
* ``wo``    ``[hidden, n_heads * head_dim]``
* ``wgu``   ``[2 * intermediate, hidden]`` - rows gate | up.
* ``wd``    ``[hidden, intermediate]``
* ``embed`` ``[vocab, hidden]``, ``lm_head`` ``[vocab, hidden]``.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import numpy as np

__all__ = [
    "Config", "TINY", "QWEN3_8B", "qwen3_8b_layers", "TINY_MOE", "QWEN3_30B_A3B", "qwen3_30b_a3b_layers",
    "layer_tensor_names",
    "weights", "prompt_tokens", "kv_context", "fragmented_block_ids",
    "gemv_weight", "gemv_activations", "attention_case", "batched_lengths",
    "GEMV_SHAPES", "sub_rng", "device_tensor_fn",
]


@dataclass(frozen=True)
class Config:
    """Dimensions of a dense Qwen3-style decoder."""
    hidden: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    eps: float = 1e-6
    rope_theta: float = 1e6
    # routed experts (inferencelayer cuda_llm.rs, Cfg: "MoE (Qwen3-30B-A3B): 0 => dense", no
    # shared expert): num_experts 0 is a dense model
    num_experts: int = 0
    topk: int = 0
    moe_inter: int = 0
    norm_topk: bool = True

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim

    def as_dict(self) -> dict:
        return asdict(self)


#: hidden 256, 2 layers, 4/2 heads, head_dim 64, SwiGLU 768, vocab 1024.
TINY = Config(hidden=256, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=64,
              intermediate=768, vocab=1024)

#: Qwen3-8B-shaped: hidden 4096, 36 layers, 32/8 heads, head_dim 128, SwiGLU 12288.
QWEN3_8B = Config(hidden=4096, n_layers=36, n_heads=32, n_kv_heads=8, head_dim=128,
                  intermediate=12288, vocab=151936)


#: tiny routed-expert model: the tiny dense shape with 8 experts of SwiGLU width 128, top-2.
TINY_MOE = Config(hidden=256, n_layers=2, n_heads=4, n_kv_heads=2, head_dim=64, intermediate=0,
                  vocab=1024, num_experts=8, topk=2, moe_inter=128)

#: Qwen3-30B-A3B-shaped: hidden 2048, 48 layers, 32/4 heads, head_dim 128, 128 experts of SwiGLU
#: width 768, top-8 with the selected weights renormalised, vocab 151936.
QWEN3_30B_A3B = Config(hidden=2048, n_layers=48, n_heads=32, n_kv_heads=4, head_dim=128, intermediate=0,
                       vocab=151936, num_experts=128, topk=8, moe_inter=768)


def qwen3_30b_a3b_layers(n_layers: int) -> Config:
    """The A3B shape with fewer layers (full width, experts and vocab) for oracle-sized parity."""
    d = QWEN3_30B_A3B.as_dict()
    d["n_layers"] = n_layers
    return Config(**d)


def qwen3_8b_layers(n_layers: int) -> Config:
    """The 8B shape with fewer layers (full width and vocab) for oracle-sized parity."""
    d = QWEN3_8B.as_dict()
    d["n_layers"] = n_layers
    return Config(**d)


#: (rows, cols) of the q4_0 GEMV microbenchmark: q/o, k/v, fused gate|up, down,
#: lm_head, plus the fused qkv projection.
GEMV_SHAPES = [(4096, 4096), (1024, 4096), (24576, 4096), (4096, 12288),
               (151936, 4096), (6144, 4096)]


def sub_rng(seed: int, *path: int) -> np.random.Generator:
    """A PCG64 stream keyed by (seed, *path); independent of every other path."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *path])))


def _normal(rng: np.random.Generator, shape, std: float, mean: float = 0.0) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    a *= np.float32(std)
    if mean:
        a += np.float32(mean)
    return a


_LAYER_TENSORS = ("attn_norm", "ffn_norm", "q_norm", "k_norm", "wqkv", "wo", "wgu", "wd")
#: routed-expert layers: the router (f32 [E, hidden], not quantised), the experts' gate|up rows
#: (expert e owns rows [e 2mi, e 2mi + mi) gate and the next mi up) and their down rows (expert e
#: owns rows [e hidden, (e + 1) hidden))
_MOE_TENSORS = ("attn_norm", "ffn_norm", "q_norm", "k_norm", "wqkv", "wo", "router", "w1", "w2")


def layer_tensor_names(cfg: Config):
    return _MOE_TENSORS if cfg.num_experts else _LAYER_TENSORS


def _layer_shape(cfg: Config, name: str):
    return {
        "attn_norm": (cfg.hidden,),
        "ffn_norm": (cfg.hidden,),
        "q_norm": (cfg.head_dim,),
        "k_norm": (cfg.head_dim,),
        "wqkv": (cfg.qkv_rows, cfg.hidden),
        "wo": (cfg.hidden, cfg.n_heads * cfg.head_dim),
        "wgu": (2 * cfg.intermediate, cfg.hidden),
        "wd": (cfg.hidden, cfg.intermediate),
        "router": (cfg.num_experts, cfg.hidden),
        "w1": (cfg.num_experts * 2 * cfg.moe_inter, cfg.hidden),
        "w2": (cfg.num_experts * cfg.hidden, cfg.moe_inter),
    }[name]


def layer_tensor(cfg: Config, seed: int, layer: int, name: str) -> np.ndarray:
    """One layer tensor, f32, drawn from its own stream (so any one can be regenerated)."""
    k = _LAYER_TENSORS.index(name) if name in _LAYER_TENSORS else 10 + _MOE_TENSORS.index(name)
    rng = sub_rng(seed, 1, layer, k)
    shape = _layer_shape(cfg, name)
    if name.endswith("norm"):
        return _normal(rng, shape, 0.1, 1.0)
    return _normal(rng, shape, 0.02)


def weights(cfg: Config, seed: int = 0) -> dict:
    """All weights of a model as f32 numpy arrays (host memory: small configs only)."""
    w = {
        "embed": _normal(sub_rng(seed, 0, 0), (cfg.vocab, cfg.hidden), 0.02),
        "final_norm": _normal(sub_rng(seed, 0, 1), (cfg.hidden,), 0.1, 1.0),
        "lm_head": _normal(sub_rng(seed, 0, 2), (cfg.vocab, cfg.hidden), 0.02),
        "layers": [],
    }
    for li in range(cfg.n_layers):
        w["layers"].append({n: layer_tensor(cfg, seed, li, n) for n in layer_tensor_names(cfg)})
    return w


def device_tensor_fn(cfg: Config, seed: int):
    """Seeded draws of a model's tensors on the GPU (torch generators), with the same
    distributions as :func:`weights` (N(0, 0.02) matrices and embedding, 1 + N(0, 0.1) norm
    weights), one tensor at a time: ``fn(layer or None, name) -> f32 CUDA tensor``. For shapes
    too large to draw on the host; the values differ from :func:`weights`."""
    import torch

    names = ("attn_norm", "ffn_norm", "q_norm", "k_norm", "wqkv", "wo", "wgu", "wd", "router", "w1", "w2")
    shapes = {n: _layer_shape(cfg, n) for n in names}
    shapes.update({"embed": (cfg.vocab, cfg.hidden), "final_norm": (cfg.hidden,),
                   "lm_head": (cfg.vocab, cfg.hidden)})

    def fn(layer, name):
        key = (seed * 1000003 + (0 if layer is None else layer + 1) * 101
               + (names.index(name) if name in names else 50 + len(name))) & 0x7FFFFFFF
        g = torch.Generator(device="cuda")
        g.manual_seed(key)
        t = torch.randn(shapes[name], generator=g, device="cuda", dtype=torch.float32)
        if name.endswith("norm"):
            return t.mul_(0.1).add_(1.0)
        return t.mul_(0.02)
    return fn


def prompt_tokens(n: int, vocab: int, seed: int = 1) -> np.ndarray:
    """n token ids uniform in [0, vocab)."""
    return sub_rng(seed, 0).integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def kv_context(n_layers: int, n_kv_heads: int, head_dim: int, n_pos: int, seed: int = 4,
               slot: int = 0):
    """A pre-filled context: K and V, each ``[n_layers, n_kv_heads, n_pos, head_dim]`` f16 N(0,1)."""
    rng = sub_rng(seed, slot)
    shape = (n_layers, n_kv_heads, n_pos, head_dim)
    k = rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16)
    v = rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16)
    return k, v


def fragmented_block_ids(num_blocks: int, seed: int = 5) -> np.ndarray:
    """A random permutation of physical block ids 0..num_blocks-1 (fragmented tables)."""
    return sub_rng(seed, 0).permutation(num_blocks).astype(np.int32)


def gemv_weight(rows: int, cols: int, seed: int = 2) -> np.ndarray:
    """A GEMV weight matrix ``[rows, cols]`` f32 N(0, 0.02)."""
    return _normal(sub_rng(seed, rows, cols), (rows, cols), 0.02)


def gemv_activations(batch: int, cols: int, seed: int = 3) -> np.ndarray:
    """GEMV activations ``[batch, cols]`` f16 N(0, 1)."""
    rng = sub_rng(seed, batch, cols)
    return rng.standard_normal(size=(batch, cols), dtype=np.float32).astype(np.float16)


def batched_lengths(batch: int, lo: int, hi: int, seed: int = 6) -> np.ndarray:
    """Per-sequence context lengths uniform in [lo, hi]."""
    return sub_rng(seed, batch).integers(lo, hi + 1, size=batch).astype(np.int32)


def attention_case(batch: int, n_heads: int, n_kv_heads: int, head_dim: int,
                   lens, block_size: int = 16, seed: int = 4, spare_blocks: int = 0):
    """Paged attention inputs: q, K/V pools, fragmented block tables.

    Returns a dict with ``q`` ``[batch, n_heads, head_dim]`` f16, ``k_pool``/``v_pool``
    ``[num_blocks, n_kv_heads, block_size, head_dim]`` f16 (N(0,1)), ``block_tables``
    ``[batch, max_blocks]`` int32 (unused entries -1) and ``lens`` ``[batch]`` int32.
    Physical blocks are a random permutation of the pool, so every table is fragmented.
    """
    lens = np.asarray(lens, dtype=np.int32)
    nblk_seq = [(int(L) + block_size - 1) // block_size for L in lens]
    max_blocks = max(max(nblk_seq), 1)
    num_blocks = sum(nblk_seq) + spare_blocks
    rng = sub_rng(seed, batch, n_heads, head_dim, int(lens.sum()))
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((batch, max_blocks), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(nblk_seq):
        bt[b, :n] = perm[off:off + n]
        off += n
    shape = (num_blocks, n_kv_heads, block_size, head_dim)
    k_pool = rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16)
    v_pool = rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16)
    q = rng.standard_normal(size=(batch, n_heads, head_dim), dtype=np.float32).astype(np.float16)
    return {"q": q, "k_pool": k_pool, "v_pool": v_pool, "block_tables": bt, "lens": lens,
            "num_blocks": num_blocks, "max_blocks": max_blocks, "block_size": block_size}
