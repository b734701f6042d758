"""Device-resident model built on the libql C ABI (memory via PyTorch, compute in libql).

``DeviceModel`` owns the torch tensors that hold a model's q4_0 weights, norms, embedding and
paged KV pools, fills the ``ql_model_desc`` and drives ``ql_decode_step`` /
``ql_decode_graph_capture`` / ``ql_decode_graph_replay``. Weights arrive as f32 (host numpy
arrays or device tensors) and are quantised on the device by ``ql_q4_0_pack_device``.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import (LayerDesc, ModelDesc, Q4Matrix, QL_KV_F16, StepArgs, check, lib, ptr, stream_ptr)

BLOCK = 16


class Q4Tensor:
    """A q4_0 matrix on the device: ``scales`` int16 [rows, cols/32] (f16 bits), ``quants`` u8."""

    def __init__(self, rows: int, cols: int, device="cuda"):
        self.rows, self.cols = rows, cols
        self.scales = torch.empty((rows, cols // 32), dtype=torch.int16, device=device)
        self.quants = torch.empty((rows, cols // 32, 16), dtype=torch.uint8, device=device)

    @classmethod
    def pack(cls, w: torch.Tensor, stream=None) -> "Q4Tensor":
        """Quantise an f32 device matrix (``ql_q4_0_pack_device``)."""
        assert w.dtype == torch.float32 and w.is_cuda and w.is_contiguous()
        t = cls(w.shape[0], w.shape[1], w.device)
        check(lib().ql_q4_0_pack_device(ptr(w), t.rows, t.cols, ptr(t.scales), ptr(t.quants),
                                        stream_ptr(stream)))
        return t

    def desc(self) -> Q4Matrix:
        return Q4Matrix(ptr(self.scales), ptr(self.quants), self.rows, self.cols)

    def nbytes(self) -> int:
        return self.scales.numel() * 2 + self.quants.numel()


def _moe(cfg) -> bool:
    return getattr(cfg, "num_experts", 0) > 0


def _matrices(cfg):
    """The layer's q4_0 matrices: q|k|v, o and the dense gate|up, down, or the experts' w1, w2."""
    return ("wqkv", "wo", "w1", "w2") if _moe(cfg) else ("wqkv", "wo", "wgu", "wd")


def _dev(a, device="cuda") -> torch.Tensor:
    if isinstance(a, torch.Tensor):
        return a.to(device=device, dtype=torch.float32).contiguous()
    return torch.from_numpy(a).to(device=device, dtype=torch.float32).contiguous()


class DeviceModel:
    """A dense Qwen3-style model resident on one GPU, plus its paged KV pools."""

    def __init__(self, cfg, weights: dict, num_blocks: int, max_batch: int,
                 max_blocks_per_seq: int, device="cuda", kv_format: int = QL_KV_F16):
        self.cfg = cfg
        self.device = device
        self.kv_format = kv_format
        self.num_blocks = num_blocks
        self.max_batch = max_batch
        self.max_blocks_per_seq = max_blocks_per_seq
        torch.cuda.synchronize()
        self.embed = _dev(weights["embed"], device)
        self.final_norm = _dev(weights["final_norm"], device)
        self.lm_head = Q4Tensor.pack(_dev(weights["lm_head"], device))
        self.layers = []
        for lw in weights["layers"]:
            L = {n: _dev(lw[n], device) for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm")}
            for n in _matrices(cfg):
                L[n] = Q4Tensor.pack(_dev(lw[n], device))
            if _moe(cfg):
                L["router"] = _dev(lw["router"], device)
            self.layers.append(L)
        torch.cuda.synchronize()
        check(lib().ql_check_device_error(None))
        self._alloc_pools()
        self._create()

    def _alloc_pools(self):
        """KV pools: f16 K and V [n_layers, num_blocks, n_kv, 16, hd], or the quantised records
        [n_layers, num_blocks, n_kv, ql_kvq_record_bytes(hd)] (u8)."""
        cfg = self.cfg
        if self.kv_format == QL_KV_F16:
            shape = (cfg.n_layers, self.num_blocks, cfg.n_kv_heads, BLOCK, cfg.head_dim)
            self.k_pool = torch.zeros(shape, dtype=torch.float16, device=self.device)
            self.v_pool = torch.zeros(shape, dtype=torch.float16, device=self.device)
            self.kvq_pool = None
        else:
            rec = int(lib().ql_kvq_record_bytes(cfg.head_dim))
            self.k_pool = self.v_pool = None
            self.kvq_pool = torch.zeros((cfg.n_layers, self.num_blocks, cfg.n_kv_heads, rec), dtype=torch.uint8,
                                        device=self.device)

    @classmethod
    def from_layer_fn(cls, cfg, tensor_fn, num_blocks, max_batch, max_blocks_per_seq, device="cuda",
                      kv_format: int = QL_KV_F16):
        """Build from ``tensor_fn(layer or None, name) -> f32 device tensor``, one tensor at a
        time (for models too large to hold as f32 anywhere)."""
        self = cls.__new__(cls)
        self.cfg, self.device, self.kv_format = cfg, device, kv_format
        self.num_blocks, self.max_batch, self.max_blocks_per_seq = num_blocks, max_batch, max_blocks_per_seq
        self.embed = tensor_fn(None, "embed")
        self.final_norm = tensor_fn(None, "final_norm")
        self.lm_head = Q4Tensor.pack(tensor_fn(None, "lm_head"))
        self.layers = []
        for li in range(cfg.n_layers):
            L = {n: tensor_fn(li, n) for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm")}
            for n in _matrices(cfg):
                w = tensor_fn(li, n)
                L[n] = Q4Tensor.pack(w)
                del w
            if _moe(cfg):
                L["router"] = tensor_fn(li, "router")
            self.layers.append(L)
        torch.cuda.synchronize()
        check(lib().ql_check_device_error(None))
        self._alloc_pools()
        self._create()
        return self

    def sibling(self, num_blocks: int, max_batch: int, max_blocks_per_seq: int,
                kv_format: int | None = None) -> "DeviceModel":
        """Another model handle over the same weight tensors, with its own KV pools, batch bound,
        block-table width and KV format (for example a batched workload next to a batch-1 one).
        The weights must outlive both handles."""
        other = DeviceModel.__new__(DeviceModel)
        other.cfg, other.device = self.cfg, self.device
        other.kv_format = self.kv_format if kv_format is None else kv_format
        other.num_blocks, other.max_batch, other.max_blocks_per_seq = num_blocks, max_batch, max_blocks_per_seq
        other.embed, other.final_norm, other.lm_head, other.layers = self.embed, self.final_norm, self.lm_head, self.layers
        other._alloc_pools()
        other._create()
        return other

    def _create(self):
        cfg = self.cfg
        self._layer_descs = (LayerDesc * cfg.n_layers)()
        empty = Q4Matrix(None, None, 0, 0)
        for i, L in enumerate(self.layers):
            if _moe(cfg):
                self._layer_descs[i] = LayerDesc(ptr(L["attn_norm"]), ptr(L["ffn_norm"]), ptr(L["q_norm"]),
                                                 ptr(L["k_norm"]), L["wqkv"].desc(), L["wo"].desc(), empty, empty,
                                                 ptr(L["router"]), L["w1"].desc(), L["w2"].desc())
            else:
                self._layer_descs[i] = LayerDesc(ptr(L["attn_norm"]), ptr(L["ffn_norm"]), ptr(L["q_norm"]),
                                                 ptr(L["k_norm"]), L["wqkv"].desc(), L["wo"].desc(),
                                                 L["wgu"].desc(), L["wd"].desc(), None, empty, empty)
        d = ModelDesc()
        d.hidden, d.n_layers, d.n_heads = cfg.hidden, cfg.n_layers, cfg.n_heads
        d.n_kv_heads, d.head_dim, d.intermediate, d.vocab = cfg.n_kv_heads, cfg.head_dim, cfg.intermediate, cfg.vocab
        d.eps, d.rope_theta = cfg.eps, cfg.rope_theta
        d.embed, d.final_norm, d.lm_head = ptr(self.embed), ptr(self.final_norm), self.lm_head.desc()
        d.layers = self._layer_descs
        d.k_pool, d.v_pool = ptr(self.k_pool), ptr(self.v_pool)
        d.num_blocks, d.block_size = self.num_blocks, BLOCK
        d.max_batch, d.max_blocks_per_seq = self.max_batch, self.max_blocks_per_seq
        d.kv_format, d.kvq_pool = self.kv_format, ptr(self.kvq_pool)
        d.num_experts, d.topk, d.moe_inter = cfg.num_experts, cfg.topk, cfg.moe_inter
        d.norm_topk = 1 if cfg.norm_topk else 0
        self._desc = d
        h = ctypes.c_void_p()
        check(lib().ql_model_create(ctypes.byref(d), ctypes.byref(h)))
        self.handle = h.value

    def weight_bytes(self) -> int:
        """Bytes of every q4_0 weight (and router) of the model."""
        n = self.lm_head.nbytes()
        for L in self.layers:
            n += sum(L[k].nbytes() for k in _matrices(self.cfg))
            if _moe(self.cfg):
                n += L["router"].numel() * 4
        return n

    def step_weight_bytes(self) -> int:
        """Weight bytes one batch-1 decode step reads: every dense matrix, or for routed experts
        the attention matrices, the router and topk experts' rows per layer."""
        if not _moe(self.cfg):
            return self.weight_bytes()
        cfg = self.cfg
        n = self.lm_head.nbytes()
        for L in self.layers:
            n += L["wqkv"].nbytes() + L["wo"].nbytes() + L["router"].numel() * 4
            n += cfg.topk * (L["w1"].nbytes() + L["w2"].nbytes()) // cfg.num_experts
        return n

    @staticmethod
    def step_args(tokens, positions, block_tables, next_tokens, active=None, logits=None,
                  out_tokens=None) -> StepArgs:
        a = StepArgs()
        a.batch = tokens.numel()
        a.tokens, a.positions, a.block_tables = ptr(tokens), ptr(positions), ptr(block_tables)
        a.active, a.logits, a.next_tokens = ptr(active), ptr(logits), ptr(next_tokens)
        a.out_tokens = ptr(out_tokens)
        a.out_stride = out_tokens.shape[1] if out_tokens is not None else 0
        return a

    def ql_model_set_option(self, option: int, value: int):
        check(lib().ql_model_set_option(self.handle, option, value))

    def ql_model_persistent_max_batch(self) -> int:
        return int(lib().ql_model_persistent_max_batch(self.handle))

    def ql_decode_step(self, args: StepArgs, stream=None):
        check(lib().ql_decode_step(self.handle, ctypes.byref(args), stream_ptr(stream)))

    def ql_decode_graph_capture(self, args: StepArgs, stream):
        check(lib().ql_decode_graph_capture(self.handle, ctypes.byref(args), stream_ptr(stream)))

    def ql_decode_graph_replay(self, batch: int, n_steps: int, stream=None):
        check(lib().ql_decode_graph_replay(self.handle, batch, n_steps, stream_ptr(stream)))

    def ql_decode_graph_step_host(self, batch: int, h_tokens, h_next_tokens, stream=None):
        """One replayed step from host buffers (int32 CPU tensors, pinned for asynchronous
        copies): h_tokens in, the step's greedy tokens out in h_next_tokens on return."""
        assert h_tokens.device.type == "cpu" and h_next_tokens.device.type == "cpu"
        check(lib().ql_decode_graph_step_host(self.handle, batch, h_tokens.data_ptr(), h_next_tokens.data_ptr(),
                                              stream_ptr(stream)))

    def ql_prefill_chunk(self, tokens, position, block_table, logits=None, next_token=None, stream=None):
        """Run the prompt tokens ``tokens`` (int32 [T] device, T <= 32) of one sequence as one
        chunk at ``position`` (int32 [1] device, advanced by T) through the sequence's
        ``block_table`` (int32 [max_blocks_per_seq] device)."""
        check(lib().ql_prefill_chunk(self.handle, ptr(tokens), tokens.numel(), ptr(position), ptr(block_table),
                                     ptr(logits), ptr(next_token), stream_ptr(stream)))

    def ql_check_device_error(self):
        check(lib().ql_check_device_error(self.handle))

    def write_context(self, slot_blocks, k_ctx, v_ctx):
        """Place a pre-filled context ``[n_layers, n_kv, n_pos, hd]`` into the pools through a
        slot's block list (stands in for prefill): f16 pools take the values as f16; the quantised
        pool takes them quantised on the device (``ql_kvq_write``, per layer)."""
        n = k_ctx.shape[2]
        if self.kv_format != QL_KV_F16:
            cfg = self.cfg
            pos = torch.arange(n, device=self.device)
            blocks = torch.as_tensor(list(slot_blocks), dtype=torch.int64, device=self.device)
            slots = (blocks[pos // BLOCK] * BLOCK + pos % BLOCK).contiguous()
            for li in range(cfg.n_layers):
                kl = torch.as_tensor(k_ctx[li], device=self.device).float().permute(1, 0, 2).contiguous()
                vl = torch.as_tensor(v_ctx[li], device=self.device).float().permute(1, 0, 2).contiguous()
                check(lib().ql_kvq_write(ptr(kl), ptr(vl), ptr(slots), n, cfg.n_kv_heads, cfg.head_dim,
                                         ptr(self.kvq_pool[li]), self.num_blocks, stream_ptr(None)))
            return
        kc = torch.as_tensor(k_ctx, dtype=torch.float16, device=self.device)
        vc = torch.as_tensor(v_ctx, dtype=torch.float16, device=self.device)
        for i, blk in enumerate(slot_blocks):
            lo, hi = i * BLOCK, min(n, (i + 1) * BLOCK)
            if lo >= n:
                break
            self.k_pool[:, blk, :, : hi - lo] = kc[:, :, lo:hi]
            self.v_pool[:, blk, :, : hi - lo] = vc[:, :, lo:hi]

    def close(self):
        if getattr(self, "handle", None):
            lib().ql_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
