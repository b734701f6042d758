#!/usr/bin/env python
"""Decode benchmark: Qwen3-8B-shaped q4_0 model, batch 1, 2048-token context, greedy steps.

One "step" is one whole decode step (embed, 36 layers of RMSNorm / q4_0 qkv GEMV / qk-norm +
RoPE + paged KV append / split-K paged GQA attention / o GEMV + residual / RMSNorm / gate|up
GEMV + SiLU*up / down GEMV + residual, final RMSNorm, lm_head GEMV + greedy argmax, position
advance) for every sequence of the batch, replayed as one CUDA graph.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ql|reference] [--config e1|e32]

Prints one JSON line. ``--impl reference`` times the f64 CPU oracle on the host cores on a
bounded sample of the same workload. Under torchrun each rank runs an independent replica
(the decode step does not shard) and rank 0 reports the aggregate.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import ql_inputs  # noqa: E402

METRIC = "decode tokens/s at 1 GB300; q4_0 GEMV + paged attn achieved HBM GB/s vs peak"
CTX = 2048


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_peaks_tflops():
    """The measured dense bf16 burst peak (TFLOP/s), or None."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return None


# ----------------------------------------------------------------------------- distributed
def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def graph_ms(fn, stream, reps: int, warm: int = 1) -> float:
    """Capture ``fn`` (a sequence of library launches on ``stream``) into a CUDA graph and time
    ``reps`` replays with CUDA events on that stream; returns ms per replay. Replaying a graph
    keeps host launch overhead out of the kernel timings."""
    import torch
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn()
    with torch.cuda.stream(stream):   # the warm replays on the timed stream, finished before e0
        for _ in range(warm):
            graph.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    ms = e0.elapsed_time(e1) / reps
    del graph
    return ms


# ----------------------------------------------------------------------------- GPU arm
device_tensor_fn = ql_inputs.device_tensor_fn

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the batch-1 tile
# stream GEMV at the gate|up shape (24576 x 4096, plain epilogue), from one ncu capture. It is
# reported only while the kernel's source files hash to the value recorded with it: any change
# to the kernel makes it null until the counters are taken again.
GU_TRAFFIC_BYTES = 57192192
GU_TRAFFIC_SOURCES = ("ql_persist.cuh", "ql_persist.cu", "ql_internal.h")
GU_TRAFFIC_SHA16 = "96f7f477bb83a1db"


def kernel_source_sha16(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "quantized_transformer_decode_ql_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemv_bytes(rows, cols, B, epilogue):
    """Algorithmic bytes of one GEMV launch: q4_0 weights, f16 activations in, the output (f32,
    or f16 halves for SiLU*up), and the residual read of the in-place add."""
    out = B * (rows // 2) * 2 if epilogue == "silu" else B * rows * 4
    return rows * cols * 18 // 32 + B * cols * 2 + out + (B * rows * 4 if epilogue == "resid" else 0)


def gemv_kinds(gm, cfg, B, s, g):
    """Each of the step's GEMV kinds alone, as the step runs them at batch 1-2 (tile stream
    layout; f16 activations in), over enough layers' matrices in turn that the weights of one
    pass exceed 3x L2 (lm_head: two packed copies of its 350 MB); CUDA-event time per launch over 3
    graph replays."""
    import torch
    import quantized_transformer_decode_ql_gb300 as ql
    l2 = torch.cuda.get_device_properties(torch.cuda.current_device()).L2_cache_size
    kinds = [("qkv", "wqkv", "none"), ("o", "wo", "resid"), ("gate_up", "wgu", "silu"), ("down", "wd", "resid"),
             ("lm_head", None, "none")]
    epi = {"none": ql.QL_EPI_NONE, "resid": ql.QL_EPI_ADD_RESIDUAL, "silu": ql.QL_EPI_SILU_MUL}
    out = {}
    for name, key, e in kinds:
        # two packed copies of lm_head (350 MB each), so that no launch finds its matrix in L2
        mats = [gm.lm_head, gm.lm_head] if key is None else [L[key] for L in gm.layers]
        W = mats[0]
        one = W.rows * W.cols * 18 // 32
        n = len(mats) if key is None else min(len(mats), max(1, -(-3 * l2 // one)))
        silu = 1 if e == "silu" else 0
        bufs = []
        for Wl in mats[:n]:
            buf = torch.empty(ql.ql_q4_0_stream_bytes(Wl.rows, Wl.cols, silu), dtype=torch.uint8, device="cuda")
            ql.ql_q4_0_stream_pack(Wl.scales, Wl.quants, Wl.rows, Wl.cols, silu, buf, s)
            bufs.append(buf)
        x = torch.randn((B, W.cols), generator=g, device="cuda").half()
        y = (torch.empty((B, W.rows // 2), dtype=torch.float16, device="cuda") if silu
             else torch.zeros((B, W.rows), dtype=torch.float32, device="cuda"))
        s.synchronize()
        reps_per = 3 if key is None else 1

        def run():
            for buf in bufs:
                for _ in range(reps_per):
                    ql.ql_gemv_q4_0_stream(buf, W.rows, W.cols, x, B, y, epi[e], None, s)
        launches = len(bufs) * reps_per
        us = graph_ms(run, s, 3) * 1e3 / launches
        nbytes = gemv_bytes(W.rows, W.cols, B, e)
        out[name] = {"rows": W.rows, "cols": W.cols, "epilogue": e, "us_per_launch": round(us, 3),
                     "bytes_per_launch": nbytes, "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "matrices_rotated": len(bufs), "launches_timed": 3 * launches}
        del bufs
    return out


def gemm_gate_up_alone(gm, s, g, T=256):
    """The prompt GEMM (tcgen05) on the 8B gate|up matrices for a T-token chunk, SiLU*up epilogue
    as in prefill, over 8 layers' matrices in turn (> 3x L2); CUDA-event time per launch over 3
    graph replays; TFLOP/s against the measured dense bf16 peak (the tensor roofline)."""
    import torch
    import quantized_transformer_decode_ql_gb300 as ql
    mats = [L["wgu"] for L in gm.layers][:8]
    W = mats[0]
    bufs = []
    for Wl in mats:
        buf = torch.empty(ql.ql_q4_0_stream_bytes(Wl.rows, Wl.cols, 1), dtype=torch.uint8, device="cuda")
        ql.ql_q4_0_stream_pack(Wl.scales, Wl.quants, Wl.rows, Wl.cols, 1, buf, s)
        bufs.append(buf)
    x = torch.randn((T, W.cols), generator=g, device="cuda").half()
    y = torch.empty((T, W.rows // 2), dtype=torch.float16, device="cuda")
    s.synchronize()

    def run():
        for buf in bufs:
            ql.ql_gemm_q4_0_stream(buf, W.rows, W.cols, x, T, y, ql.QL_EPI_SILU_MUL, s)
    us = graph_ms(run, s, 3) * 1e3 / len(bufs)
    flops = 2.0 * T * W.rows * W.cols
    tf = flops / (us * 1e-6) / 1e12
    peak = load_peaks_tflops()
    del bufs
    return {"rows": W.rows, "cols": W.cols, "tokens": T, "epilogue": "silu", "us_per_launch": round(us, 3),
            "bound": "tensor", "flops_per_launch": flops, "achieved_tflops": round(tf, 1),
            "peak_tflops": peak, "peak_source": "measured bf16 burst (the f16 kind's rate)",
            "frac": round(tf / peak, 4) if peak else None, "matrices_rotated": len(mats)}


def attn_alone(B, lo, hi, s, g, seed=6, iters=10, kvq=False):
    """Paged GQA decode attention alone at the attention workload's shape (32/8 heads, head_dim
    128, 16-token blocks, randomly permuted block tables): B sequences with lengths uniform in
    [lo, hi]; L2 flushed (a 256 MB read) before every launch, the flush timed apart and taken out."""
    import torch
    import quantized_transformer_decode_ql_gb300 as ql
    nh, nkv, hd = 32, 8, 128
    lens = ql_inputs.batched_lengths(B, lo, hi, seed=seed)
    nblk = [(int(L) + 15) // 16 for L in lens]
    maxb, num_blocks = max(nblk), sum(nblk)
    perm = torch.from_numpy(ql_inputs.fragmented_block_ids(num_blocks, seed=5)).cuda()
    bt = torch.full((B, maxb), -1, dtype=torch.int32, device="cuda")
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += n
    if kvq:   # records quantised on the device from N(0,1) rows, 65536 positions at a time
        pool = torch.zeros((num_blocks, nkv, ql.ql_kvq_record_bytes(hd)), dtype=torch.uint8, device="cuda")
        for p0 in range(0, num_blocks * 16, 65536):
            n = min(65536, num_blocks * 16 - p0)
            slots = torch.arange(p0, p0 + n, dtype=torch.int64, device="cuda")
            k = torch.randn((n, nkv, hd), generator=g, device="cuda")
            v = torch.randn((n, nkv, hd), generator=g, device="cuda")
            ql.ql_kvq_write(k, v, slots, nkv, hd, pool, num_blocks)   # on the stream that made k, v
        torch.cuda.synchronize()
        del k, v
    else:
        kp = torch.randn((num_blocks, nkv, 16, hd), generator=g, device="cuda").half()
        vp = torch.randn((num_blocks, nkv, 16, hd), generator=g, device="cuda").half()
    q = torch.randn((B, nh, hd), generator=g, device="cuda").half()
    o = torch.empty((B, nh * hd), dtype=torch.float16, device="cuda")
    cl = torch.from_numpy(lens).cuda()
    ws = torch.zeros(ql.ql_paged_attn_workspace_bytes(B, nh, nkv, hd, 16, maxb), dtype=torch.uint8, device="cuda")
    flush = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    flush_sum = torch.zeros((), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()

    def run():
        if kvq:
            ql.ql_paged_attn_decode_kvq(q, pool, bt, cl, B, nh, nkv, hd, 16, maxb, num_blocks, 1 / math.sqrt(hd), o,
                                        ws, s)
        else:
            ql.ql_paged_attn_decode(q, kp, vp, bt, cl, B, nh, nkv, hd, 16, maxb, num_blocks, 1 / math.sqrt(hd), o,
                                    ws, s)
    with torch.cuda.stream(s):
        run()                       # first call outside capture (per-device set-up)
    s.synchronize()

    def flush_then_run():
        for _ in range(iters):
            flush_sum.copy_(flush.sum())
            run()

    def flush_only():
        for _ in range(iters):
            flush_sum.copy_(flush.sum())
    us = (graph_ms(flush_then_run, s, 3) - graph_ms(flush_only, s, 3)) * 1e3 / iters
    per_pos = nkv * 29 * hd / 16 if kvq else 2 * nkv * hd * 2   # K and V bytes of one position
    nbytes = int(sum(int(L) * per_pos + 4 * ((int(L) + 15) // 16) for L in lens) + B * nh * hd * 4)
    return {"batch": B, "lengths": f"uniform in [{lo}, {hi}] (seed {seed})", "sum_len": int(lens.sum()),
            "kv": "q8_0 K / q5_1 V records" if kvq else "f16",
            "us_per_launch": round(us, 2), "bytes_per_launch": int(nbytes),
            "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}


def prefill_context(gm, cfg, ids, n_pos, g):
    """Synthetic pre-filled context (stands in for prefill): N(0,1) K and V written straight
    into a slot's blocks of every layer and kv head: as f16 into an f16 pool, quantised on the
    device (ql_kvq_write) into a quantised one."""
    import torch
    import quantized_transformer_decode_ql_gb300 as ql
    nb = (n_pos + 15) // 16
    idx = torch.as_tensor(list(ids[:nb]), dtype=torch.long, device="cuda")
    if gm.kv_format != ql.QL_KV_F16:
        pos = torch.arange(n_pos, device="cuda")
        slots = (idx[pos // 16] * 16 + pos % 16).contiguous()
        for li in range(cfg.n_layers):
            k = torch.randn((n_pos, cfg.n_kv_heads, cfg.head_dim), generator=g, device="cuda")
            v = torch.randn((n_pos, cfg.n_kv_heads, cfg.head_dim), generator=g, device="cuda")
            ql.ql_kvq_write(k, v, slots, cfg.n_kv_heads, cfg.head_dim, gm.kvq_pool[li], gm.num_blocks)
        return
    shape = (cfg.n_layers, nb, cfg.n_kv_heads, 16, cfg.head_dim)
    gm.k_pool[:, idx] = torch.randn(shape, generator=g, device="cuda").half()
    gm.v_pool[:, idx] = torch.randn(shape, generator=g, device="cuda").half()


def kv_bytes_per_token(gm, cfg):
    """KV bytes one cached position costs over all layers: f16 K and V, or its share of the
    quantised records (29 head_dim bytes per 16 positions and kv head)."""
    import quantized_transformer_decode_ql_gb300 as ql
    if gm.kv_format == ql.QL_KV_F16:
        return cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim * 2
    return cfg.n_layers * cfg.n_kv_heads * 29 * cfg.head_dim / 16


def build_e1(cfg, steps, warmup):
    """The 8B-shaped model (seeded device draws, q4_0 on the device) with a batch-1 pool."""
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    max_ctx = CTX + warmup + steps + 2
    maxb = (max_ctx + 15) // 16
    num_blocks = maxb + 8
    gm = DeviceModel.from_layer_fn(cfg, device_tensor_fn(cfg, seed=0), num_blocks=num_blocks,
                                   max_batch=1, max_blocks_per_seq=maxb)
    return gm, maxb, num_blocks, max_ctx


def gpu_arm(args, rank, world, local_rank):
    import torch

    from quantized_transformer_decode_ql_gb300 import build as qbuild
    if rank == 0 or world == 1:
        qbuild.build()
    barrier(world)
    import quantized_transformer_decode_ql_gb300 as ql

    torch.cuda.set_device(local_rank)
    cfg = ql_inputs.QWEN3_8B
    if args.layers:   # profiling aid: the same layer shapes, fewer layers (not a bench line)
        cfg = dataclasses.replace(cfg, n_layers=args.layers)
    B = 1
    steps, warmup = args.steps, args.warmup
    t_setup = time.time()
    gm, maxb, num_blocks, max_ctx = build_e1(cfg, steps, warmup)
    gm.ql_model_set_option(ql.QL_OPT_STEP_KERNEL, STEP_KERNELS[args.step_kernel])
    persistent = args.step_kernel == "persistent" and B <= gm.ql_model_persistent_max_batch()
    streamed = not persistent and B <= gm.ql_model_persistent_max_batch()   # stream GEMVs in the step
    # fragmented block table; pre-filled synthetic context of CTX positions N(0,1) f16
    perm = torch.from_numpy(ql_inputs.fragmented_block_ids(num_blocks, seed=5)).cuda()
    bt = perm[:maxb].reshape(1, maxb).contiguous()
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    prefill_context(gm, cfg, bt[0].tolist(), CTX, g)
    first = torch.from_numpy(ql_inputs.prompt_tokens(B, cfg.vocab, seed=1)).cuda()
    tokens = first.clone()
    positions = torch.full((B,), CTX, dtype=torch.int32, device="cuda")
    out_tokens = torch.full((B, max_ctx + 1), -1, dtype=torch.int32, device="cuda")
    sargs = gm.step_args(tokens, positions, bt, tokens, out_tokens=out_tokens)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    gm.ql_decode_graph_capture(sargs, s)
    setup_s = time.time() - t_setup

    def reset():
        tokens.copy_(first)
        positions.fill_(CTX)

    # warm-up (untimed), then reset to the same starting state
    with torch.cuda.stream(s):
        reset()
        gm.ql_decode_graph_replay(B, warmup, s)
        reset()
    s.synchronize()
    gm.ql_check_device_error()

    # ---- timed region: K graph replays, device-timed with events on the launching stream
    clock = ClockSampler(local_rank)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        e0.record(s)
        gm.ql_decode_graph_replay(B, steps, s)
        e1.record(s)
    s.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    clocks = clock.stop()
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(ms, world)
    gm.ql_check_device_error()
    toks = out_tokens.cpu().numpy()
    phases = step_phases(gm, sargs, s, cfg) if persistent else launch_phases(gm, sargs, s, cfg)

    # ---- algorithmic bytes per step (weights + KV read/write + embedding row + logits)
    wbytes = gm.weight_bytes()
    kv_tok = cfg.n_layers * 2 * cfg.n_kv_heads * cfg.head_dim * 2
    ctx_avg = CTX + 1 + (steps - 1) / 2.0
    step_bytes = wbytes + B * (kv_tok * ctx_avg + kv_tok + cfg.hidden * 4 + cfg.vocab * 4)

    # ---- end to end through the C ABI with host buffers: per step one ql_decode_graph_step_host
    # call (H2D of the step's token ids from pinned memory, one graph replay, D2H of the next
    # tokens, stream sync), made as a C caller makes it (arguments bound once). A greedy loop
    # passes one pinned buffer as input and output: the step's tokens become the next input.
    import quantized_transformer_decode_ql_gb300._lib as qlib
    h_buf = torch.empty((B,), dtype=torch.int32, pin_memory=True)
    h_buf.copy_(first.cpu())
    with torch.cuda.stream(s):
        positions.fill_(CTX)
    s.synchronize()
    step_host = qlib.lib().ql_decode_graph_step_host
    call = (gm.handle, B, h_buf.data_ptr(), h_buf.data_ptr(), s.cuda_stream)
    t0 = time.perf_counter()
    for _ in range(steps):
        rc = step_host(*call)
        if rc != qlib.QL_OK:
            qlib.check(rc)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world)

    # ---- the kernels alone (untimed region over): every GEMV kind at this batch, the dominant
    # one (gate|up, the largest weight stream of a layer) is the roofline kernel; attention at
    # this context and on the attention workload (batch 32, lengths in [512, 32768])
    peak, peak_src = load_peaks()
    kernels = {}
    if streamed:
        kernels["gemv"] = gemv_kinds(gm, cfg, B, s, g)
    kernels["paged_attention_e1"] = attn_alone(1, int(ctx_avg), int(ctx_avg), s, g)
    if not args.layers:
        kernels["paged_attention_a_b32"] = attn_alone(32, 512, 32768, s, g)
        kernels["paged_attention_a_b32_kvq"] = attn_alone(32, 512, 32768, s, g, kvq=True)
    for k in kernels.values():
        for v in (k.values() if "qkv" in k else [k]):
            v["frac"] = round(v["achieved_gbs"] / peak, 4)
    if not args.layers and streamed:
        kernels["gemm_prefill_gate_up_t256"] = gemm_gate_up_alone(gm, s, g)

    tok_total = sum_over_ranks(float(B * steps), world)
    value = tok_total / (ms_max / 1e3)
    step_gbs = step_bytes * steps / (ms_max / 1e3) / 1e9
    kernels_per_step = 1 if persistent else 3 + 5 * cfg.n_layers   # embed, 5 per layer, lm_head, finalize
    roof = {"bound": "hbm", "peak": peak, "unit": "GB/s", "peak_source": peak_src}
    if streamed:
        gu = kernels["gemv"]["gate_up"]
        sha = kernel_source_sha16(GU_TRAFFIC_SOURCES)
        traffic = GU_TRAFFIC_BYTES if sha == GU_TRAFFIC_SHA16 else None
        roof.update({"kernel": "gemv_stream_kernel<1,16>: q4_0 GEMV over the tile stream layout, gate|up "
                               "24576 x 4096, SiLU*up epilogue, batch 1",
                     "achieved": gu["achieved_gbs"], "frac": round(gu["achieved_gbs"] / peak, 4),
                     "traffic": traffic, "algorithmic_bytes": gu["bytes_per_launch"],
                     "us_per_launch": gu["us_per_launch"],
                     "traffic_note": ("one ncu capture of this kernel source (sha %s), plain epilogue" % sha
                                      if traffic else "kernel source changed since the counters were taken")})
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": round(ms_max / steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "q4_0 weights; int16 fixed-point activations at batch 1-2 (dp2a, exact block sums); f16 KV; f32 accumulation",
        "data": "synthetic (seeded random-init weights, N(0,1) f16 KV context, random prompt token)",
        "config": {"workload": f"qwen3-8b-shaped q4_0 decode, batch {B}, {CTX}-token context, {steps} greedy steps",
                   "hidden": cfg.hidden, "layers": cfg.n_layers, "heads": f"{cfg.n_heads}/{cfg.n_kv_heads}",
                   "head_dim": cfg.head_dim, "intermediate": cfg.intermediate, "vocab": cfg.vocab,
                   "batch": B, "context": CTX, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (%.2f GB of q4_0 weights streamed per step)" % (wbytes / 1e9)},
        "roofline": roof,
        "step_roofline": {"bytes_per_step": int(step_bytes), "achieved_gbs": round(step_gbs, 1),
                          "frac": round(step_gbs / peak, 4),
                          "roofline_tokens_s": round(B * peak * 1e9 / step_bytes, 1)},
        "kernels": kernels,
        "clocks": clocks,
        "e2e": {"value": round(tok_total / e2e_s, 2), "unit": "tokens/s", "h2d_bytes_per_step": 4 * B,
                "d2h_bytes_per_step": 4 * B, "api": "ql_decode_graph_step_host (host token buffers)"},
        "gpu_launches": kernels_per_step * steps,
        "setup_s": round(setup_s, 1),
        "tokens_head": toks[0, CTX + 1: CTX + 9].tolist(),
        "step_kernel": "persistent (one cooperative launch per step)" if persistent else "one launch per phase",
    }
    if phases:
        line["step_phases_us"] = phases
    if not args.layers and not args.no_prefill:
        line["prefill_8b"] = prefill_run(gm, cfg, s)
        line["prefill_8b_chunk32"] = prefill_run(gm, cfg, s, chunk=32)
    if not args.layers and not args.no_moe:
        line["moe_a3b_b1"] = moe_run(min(steps, 64), 3, s, local_rank, world)
    if not args.layers and not args.no_e32:
        for key, fmt in (("e32", ql.QL_KV_F16), ("e32_kvq", ql.QL_KV_Q8_0_Q5_1)):
            gm32 = gm.sibling(**e32_pool(cfg, E32_STEPS, 3), kv_format=fmt)
            try:
                line[key] = e32_run(gm32, cfg, E32_STEPS, 3, s, local_rank, world)
            finally:
                gm32.close()
                del gm32
    gm.close()
    return line


def moe_run(steps, warmup, s, local_rank, world):
    """The Qwen3-30B-A3B-shaped routed-expert model (48 layers, 128 experts of 768, top-8,
    random-init, q4_0 on the device) at batch 1 over a 2048-token pre-filled context: `steps`
    greedy steps timed as graph replays. Step bytes: the attention matrices, the f32 router and
    the top-8 experts' rows of every layer, the lm_head, the KV read and written, the embedding
    row and the logits."""
    import torch
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.QWEN3_30B_A3B
    max_ctx = CTX + warmup + steps + 2
    maxb = (max_ctx + 15) // 16
    t0 = time.time()
    gm = DeviceModel.from_layer_fn(cfg, device_tensor_fn(cfg, seed=0), num_blocks=maxb + 8, max_batch=1,
                                   max_blocks_per_seq=maxb)
    try:
        bt = torch.from_numpy(ql_inputs.fragmented_block_ids(maxb + 8, seed=5)[:maxb]).cuda().reshape(1, maxb)
        g = torch.Generator(device="cuda")
        g.manual_seed(4)
        prefill_context(gm, cfg, bt[0].tolist(), CTX, g)
        first = torch.from_numpy(ql_inputs.prompt_tokens(1, cfg.vocab, seed=1)).cuda()
        tokens = first.clone()
        positions = torch.full((1,), CTX, dtype=torch.int32, device="cuda")
        sargs = gm.step_args(tokens, positions, bt, tokens)
        torch.cuda.synchronize()
        gm.ql_decode_graph_capture(sargs, s)
        setup_s = time.time() - t0
        with torch.cuda.stream(s):
            gm.ql_decode_graph_replay(1, warmup, s)
            tokens.copy_(first)
            positions.fill_(CTX)
        s.synchronize()
        gm.ql_check_device_error()
        clock = ClockSampler(local_rank)
        time.sleep(0.3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            gm.ql_decode_graph_replay(1, steps, s)
            e1.record(s)
        s.synchronize()
        clocks = clock.stop()
        gm.ql_check_device_error()
        ms = max_over_ranks(e0.elapsed_time(e1), world)
        phases = launch_phases(gm, sargs, s, cfg)
        peak, peak_src = load_peaks()
        kv_tok = kv_bytes_per_token(gm, cfg)
        ctx_avg = CTX + 1 + (steps - 1) / 2.0
        step_bytes = gm.step_weight_bytes() + kv_tok * ctx_avg + kv_tok + cfg.hidden * 4 + cfg.vocab * 4
        gbs = step_bytes * steps / (ms / 1e3) / 1e9
        return {"value": round(sum_over_ranks(float(steps), world) / (ms / 1e3), 2), "unit": "tokens/s",
                "steps": steps, "warmup": warmup, "ms_per_step": round(ms / steps, 4),
                "workload": f"qwen3-30b-a3b-shaped routed-expert q4_0 decode (48 layers, 128 experts of 768, "
                            f"top-8), batch 1, {CTX}-token context, {steps} greedy steps",
                "weights_gb": round(gm.weight_bytes() / 1e9, 2),
                "step_roofline": {"bytes_per_step": int(step_bytes), "achieved_gbs": round(gbs, 1),
                                  "frac": round(gbs / peak, 4), "peak": peak, "peak_source": peak_src,
                                  "roofline_tokens_s": round(peak * 1e9 / step_bytes, 1)},
                "clocks": clocks, "gpu_launches": (3 + 7 * cfg.n_layers) * steps, "setup_s": round(setup_s, 1),
                **({"step_phases_us": phases} if phases else {})}
    finally:
        gm.close()


PREFILL_CHUNK = 256


def prefill_run(gm, cfg, s, n_prompt=2048, chunk=PREFILL_CHUNK):
    """Chunked prefill of one n_prompt-token prompt on the 8B shape (a sibling handle with batch
    bound `chunk` over the same weights): n_prompt / chunk calls of ql_prefill_chunk timed with
    CUDA events on the launching stream, against the weights streamed once per chunk (above 32
    tokens the chunk's projections are the tcgen05 GEMM, below the batched GEMVs)."""
    import torch
    maxb = (n_prompt + 15) // 16 + 1
    gp = gm.sibling(num_blocks=maxb + 8, max_batch=chunk, max_blocks_per_seq=maxb)
    try:
        bt = torch.from_numpy(ql_inputs.fragmented_block_ids(maxb + 8, seed=5)[:maxb].copy()).cuda()
        prompt = torch.from_numpy(ql_inputs.prompt_tokens(n_prompt, cfg.vocab, seed=1)).cuda()
        position = torch.zeros(1, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")

        def run():
            for c0 in range(0, n_prompt, chunk):
                gp.ql_prefill_chunk(prompt[c0:c0 + chunk], position, bt, next_token=nxt, stream=s)
        with torch.cuda.stream(s):
            run()                       # warm-up pass over the whole prompt
            position.zero_()
        s.synchronize()
        gp.ql_check_device_error()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            run()
            e1.record(s)
        s.synchronize()
        gp.ql_check_device_error()
        ms = e0.elapsed_time(e1)
        n_chunks = -(-n_prompt // chunk)
        wbytes = gp.weight_bytes()
        return {"value": round(n_prompt / (ms / 1e3), 1), "unit": "prompt tokens/s", "prompt": n_prompt,
                "chunk": chunk, "ms": round(ms, 3), "ms_per_chunk": round(ms / n_chunks, 4),
                "workload": f"qwen3-8b-shaped q4_0 prefill of one {n_prompt}-token prompt in chunks of {chunk}",
                "weights_gbs": round(wbytes * n_chunks / (ms / 1e3) / 1e9, 1)}
    finally:
        gp.close()


E32_STEPS = 128
E32_FRESH = 128


def e32_pool(cfg, steps, warmup):
    lens0 = ql_inputs.batched_lengths(32, 128, 8192, seed=7)
    cap = int(max(lens0.max(), E32_FRESH)) + warmup + steps + 2
    maxb = (cap + 15) // 16
    need = (sum((int(L) + warmup + steps + 2 + 15) // 16 for L in lens0)
            + 32 * ((E32_FRESH + steps + 2 + 15) // 16) + 16)
    return {"num_blocks": need, "max_batch": 32, "max_blocks_per_seq": maxb}


def e32_run(gm, cfg, steps, warmup, s, local_rank, world):
    """Batched decode: 32 sequences with initial context lengths uniform in [128, 8192], fragmented
    block tables from the library's block allocator, `steps` greedy steps; every sequence finishes
    at a random step and is replaced by a fresh 128-position context in newly allocated blocks.
    The replacement work runs between graph replays and is excluded from the decode time
    (reported separately). Each step is timed with CUDA events on the launching stream."""
    import torch
    import quantized_transformer_decode_ql_gb300 as ql
    B = 32
    lens0 = ql_inputs.batched_lengths(B, 128, 8192, seed=7)
    finish = ql_inputs.sub_rng(8, B).integers(0, steps, size=B)
    need, maxb = gm.num_blocks, gm.max_blocks_per_seq
    pool = ql.BlockPool(need)
    order = [pool.alloc() for _ in range(need)]
    pool.free([order[i] for i in ql_inputs.fragmented_block_ids(need, seed=5)])
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    bt_host = np.zeros((B, maxb), np.int32)
    owned = [None] * B

    def place(b, n_pos, n_total):
        ids = [pool.alloc() for _ in range((n_total + 15) // 16)]
        owned[b] = ids
        bt_host[b, :] = 0
        bt_host[b, :len(ids)] = ids
        prefill_context(gm, cfg, ids, n_pos, g)

    for b in range(B):
        place(b, int(lens0[b]), int(lens0[b]) + warmup + steps + 2)
    bt = torch.from_numpy(bt_host).cuda()
    tokens = torch.from_numpy(ql_inputs.prompt_tokens(B, cfg.vocab, seed=1)).cuda()
    positions = torch.from_numpy(lens0.astype(np.int32)).cuda()
    sargs = gm.step_args(tokens, positions, bt, tokens)
    torch.cuda.synchronize()
    gm.ql_decode_graph_capture(sargs, s)
    with torch.cuda.stream(s):
        gm.ql_decode_graph_replay(B, warmup, s)
    s.synchronize()
    gm.ql_check_device_error()

    clock = ClockSampler(local_rank)
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    kv_tok = kv_bytes_per_token(gm, cfg)
    live_len = positions.cpu().numpy().astype(np.int64) + 1
    step_bytes = []
    repl_s = 0.0
    for i in range(steps):
        step_bytes.append(gm.weight_bytes() + kv_tok * int(live_len.sum()) + B * (kv_tok + cfg.hidden * 4 + cfg.vocab * 4))
        with torch.cuda.stream(s):
            ev[i][0].record(s)
            gm.ql_decode_graph_replay(B, 1, s)
            ev[i][1].record(s)
        live_len += 1
        done = np.flatnonzero(finish == i)
        if len(done):
            t0 = time.perf_counter()
            s.synchronize()
            pos_h = positions.cpu().numpy()
            for b in done:
                pool.free(owned[b])
                place(int(b), E32_FRESH, E32_FRESH + steps + 2)
                pos_h[b] = E32_FRESH
                live_len[b] = E32_FRESH + 1
            bt.copy_(torch.from_numpy(bt_host))
            positions.copy_(torch.from_numpy(pos_h))
            torch.cuda.synchronize()
            repl_s += time.perf_counter() - t0
    s.synchronize()
    clocks = clock.stop()
    gm.ql_check_device_error()
    ms = sum(a.elapsed_time(b) for a, b in ev)
    ms = max_over_ranks(ms, world)
    phases = launch_phases(gm, sargs, s, cfg)   # untimed, after the timed region
    peak, peak_src = load_peaks()
    value = sum_over_ranks(float(B * steps), world) / (ms / 1e3)
    gbs = sum(step_bytes) / (ms / 1e3) / 1e9
    return {
        "value": round(value, 2), "unit": "tokens/s", "steps": steps, "warmup": warmup,
        "ms_per_step": round(ms / steps, 4),
        "workload": f"qwen3-8b-shaped q4_0 batched decode, 32 sequences, contexts uniform in [128, 8192], "
                    f"{steps} greedy steps, finished sequences replaced by fresh {E32_FRESH}-position contexts, "
                    + ("f16 KV cache" if gm.kv_format == ql.QL_KV_F16 else "q8_0 K / q5_1 V cache"),
        "kv_bytes_per_token": kv_tok,
        "step_roofline": {"bytes_per_step_avg": int(np.mean(step_bytes)), "achieved_gbs": round(gbs, 1),
                          "frac": round(gbs / peak, 4), "peak": peak, "peak_source": peak_src,
                          "roofline_tokens_s": round(B * peak * 1e9 / float(np.mean(step_bytes)), 1)},
        "replacement_s_excluded": round(repl_s, 3), "replacements": int((finish < steps).sum()),
        "clocks": clocks, "gpu_launches": launches_per_step(cfg, B) * steps,
        **({"step_phases_us": phases} if phases else {}),
    }


def gpu_arm_e32(args, rank, world, local_rank):
    """The batched workload as its own bench line (``--config e32``)."""
    import torch

    from quantized_transformer_decode_ql_gb300 import build as qbuild
    if rank == 0 or world == 1:
        qbuild.build()
    barrier(world)
    from quantized_transformer_decode_ql_gb300.model import DeviceModel

    torch.cuda.set_device(local_rank)
    cfg = ql_inputs.QWEN3_8B
    t_setup = time.time()
    import quantized_transformer_decode_ql_gb300 as ql
    gm = DeviceModel.from_layer_fn(cfg, device_tensor_fn(cfg, seed=0), **e32_pool(cfg, args.steps, args.warmup),
                                   kv_format=ql.QL_KV_Q8_0_Q5_1 if args.kv == "q8q5" else ql.QL_KV_F16)
    setup_s = time.time() - t_setup
    s = torch.cuda.Stream()
    r = e32_run(gm, cfg, args.steps, args.warmup, s, local_rank, world)
    gm.close()
    line = {"metric": METRIC, "value": r.pop("value"), "unit": r.pop("unit"), "n_gpus": world,
            "steps": r.pop("steps"), "warmup": r.pop("warmup"), "ms_per_step": r.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "q4_0 weights, f16 act/KV, f32 accum",
            "data": "synthetic (seeded random-init weights, N(0,1) f16 KV contexts, random tokens)",
            "config": {"workload": r.pop("workload"), "batch": 32, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (%.2f GB of weights + KV per step on average)"
                             % (r["step_roofline"]["bytes_per_step_avg"] / 1e9)},
            "setup_s": round(setup_s, 1)}
    line.update(r)
    return line


def gpu_arm_prefill(args, rank, world, local_rank):
    """The chunked prefill workload as its own line (``--config prefill``): one 2048-token prompt
    in chunks of --chunk tokens on the 8B shape, timed as in the default line's prefill_8b key."""
    import torch

    from quantized_transformer_decode_ql_gb300 import build as qbuild
    if rank == 0 or world == 1:
        qbuild.build()
    barrier(world)
    from quantized_transformer_decode_ql_gb300.model import DeviceModel

    torch.cuda.set_device(local_rank)
    cfg = ql_inputs.QWEN3_8B
    gm = DeviceModel.from_layer_fn(cfg, device_tensor_fn(cfg, seed=0), num_blocks=16, max_batch=1,
                                   max_blocks_per_seq=4)
    s = torch.cuda.Stream()
    clock = ClockSampler(local_rank)
    chunk = args.chunk
    r = prefill_run(gm, cfg, s, chunk=chunk)
    clocks = clock.stop()
    gm.close()
    value = sum_over_ranks(r.pop("value"), world)
    line = {"metric": f"prefill prompt tokens/s at 1 GB300 (q4_0 weights, chunks of {chunk})", "value": value,
            "unit": r.pop("unit"), "n_gpus": world, "steps": -(-2048 // chunk), "warmup": -(-2048 // chunk),
            "ms_per_step": r["ms_per_chunk"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "q4_0 weights, f16 act/KV, f32 accum", "data": "synthetic (seeded random-init weights, random prompt)",
            "config": {"workload": r.pop("workload"), "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (4.6 GB of weights streamed per chunk)"},
            "clocks": clocks}
    line.update(r)
    return line


STEP_KERNELS = {"auto": 0, "launches": 1, "persistent": 2}


def gemv_passes(cols, batch):
    """Launches of one q4_0 GEMV call: the batch goes in passes of as many columns as the
    kernel's 100 KB activation staging holds (at most 8)."""
    nblk = cols // 32
    fixed = nblk * 8 * 4 + 8 * 32 * 16
    nb_max = min(8, (100 * 1024 - fixed) // ((nblk * 4 + 4) * 16))
    return -(-batch // nb_max)


def launches_per_step(cfg, B):
    """Kernel launches of one step in the one-launch-per-phase form. Batch 1-2: embed, per layer
    qkv / attention / o / gate_up / down GEMVs over the tile stream layout, lm_head, finalize.
    Batch 3-32 (the mma.sync form): each GEMV is the split-K kernel plus its merge kernel; the
    RMSNorm is folded into the merges, so only layer 0's q|k|v GEMV gets an RMSNorm kernel first
    (every RMSNorm'd GEMV does with QL_BATCHED_NORM_FOLD=0). Above 32: row-major passes."""
    if B <= 2:
        return 3 + 5 * cfg.n_layers
    if B <= 32:
        if os.environ.get("QL_BATCHED_NORM_FOLD", "1").strip() == "0":
            return 5 + 11 * cfg.n_layers   # an RMSNorm before q|k|v and gate|up, and before lm_head
        return 5 + 9 * cfg.n_layers
    per_layer = (gemv_passes(cfg.hidden, B) * 2 + gemv_passes(cfg.n_heads * cfg.head_dim, B)
                 + gemv_passes(cfg.intermediate, B) + 1)
    return 2 + per_layer * cfg.n_layers + gemv_passes(cfg.hidden, B)


def ns_relative(raw, nstamps, base=None):
    """The trace as float64 with its first `nstamps` words (globaltimer ns, ~1.8e18) taken
    relative to the earliest stamp (or to `base`), in int64 first: float64 cannot hold the
    absolute values to better than 256 ns. Unwritten (zero) stamps stay zero, written ones are
    >= 1."""
    import numpy as np
    out = raw.astype(np.float64)
    ts = raw[..., :nstamps]
    if (ts > 0).any():
        if base is None:
            base = ts[ts > 0].min() - 1
        out[..., :nstamps] = np.where(ts > 0, ts - base, 0).astype(np.float64)
    return out


def launch_phases(gm, sargs, s, cfg):
    """Per-GEMV phase times of a step of separate launches (batch 1-2) from the GEMV kernels'
    globaltimer trace (untimed eager steps after the timed region). Per matrix kind, means over
    layers, in us: "gap" = first CTA start minus the previous GEMV's last CTA end (covers the
    launches in between, e.g. attention before o), "wait" = last CTA past its wait on the
    predecessor minus first CTA start, "stage" / "loop" / "finish" = per-CTA mean durations of
    activation staging, the unit loop and the epilogues, "tail" = last CTA end minus the mean
    CTA end, "span" = last end minus first start."""
    import numpy as np
    import torch
    import quantized_transformer_decode_ql_gb300 as ql
    grid = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    rows = 4 * cfg.n_layers + 1
    B = int(sargs.batch) if hasattr(sargs, "batch") else 1
    buf = torch.zeros((rows + cfg.n_layers) * grid * 8, dtype=torch.int64, device="cuda")
    # batch 3-32: the merge launch after each split-K GEMV, [rows][grid CTAs][4]
    mbuf = torch.zeros(rows * grid * 4, dtype=torch.int64, device="cuda") if B > 2 else None
    gm.ql_model_set_option(ql.QL_OPT_STEP_TRACE, buf.data_ptr())
    if mbuf is not None:
        gm.ql_model_set_option(ql.QL_OPT_MERGE_TRACE, mbuf.data_ptr())
    try:   # a graph captured with the trace on, replayed as the timed graph is (2 steps: one warm)
        gm.ql_decode_graph_capture(sargs, s)
        with torch.cuda.stream(s):
            gm.ql_decode_graph_replay(B, 1, s)
        s.synchronize()
        buf.zero_()
        if mbuf is not None:
            mbuf.zero_()
        with torch.cuda.stream(s):
            gm.ql_decode_graph_replay(B, 1, s)
        s.synchronize()
    finally:
        gm.ql_model_set_option(ql.QL_OPT_STEP_TRACE, 0)
        gm.ql_model_set_option(ql.QL_OPT_MERGE_TRACE, 0)
        gm.ql_decode_graph_capture(sargs, s)
    gm.ql_check_device_error()
    raw = buf.cpu().numpy().reshape(rows + cfg.n_layers, grid, 8)
    stamped = raw[..., :6][raw[..., :6] > 0]
    base = stamped.min() - 1 if stamped.size else None
    ta = ns_relative(raw, 6, base)
    t, tat = ta[:rows], ta[rows:]
    tm = ns_relative(mbuf.cpu().numpy().reshape(rows, grid, 4), 4, base) if mbuf is not None else None
    if not (t[:, 0, 0] > 0).all():
        return None   # another GEMV form ran (not traced)
    kinds = [k for _ in range(cfg.n_layers) for k in ("qkv", "o", "gate_up", "down")] + ["lm_head"]
    acc = {}
    for k in range(rows):
        r = t[k][t[k][:, 0] > 0]   # the launch's CTAs (a grid may be smaller than the SM count)
        prev_end = t[k - 1][t[k - 1][:, 0] > 0][:, 5].max() if k > 0 else float("nan")
        v = {"gap": (r[:, 0].min() - prev_end) if k > 0 else float("nan"),
             "wait": r[:, 1].max() - r[:, 0].min(),
             "first_past_wait": (r[:, 1].min() - prev_end) if k > 0 else float("nan"),
             "stage": (r[:, 2] - r[:, 1]).mean(), "loop": (r[:, 3] - r[:, 2]).mean(),
             "finish": (r[:, 5] - r[:, 3]).mean(), "sync": (r[:, 4] - r[:, 3]).mean(),
             "epilogue": (r[:, 5] - r[:, 4]).mean(), "tail": r[:, 5].max() - r[:, 5].mean(),
             "span": r[:, 5].max() - r[:, 0].min(),
             "ring_wait_frac": r[:, 6].sum() / max(r[:, 7].sum(), 1.0)}
        a = acc.setdefault(kinds[k], [])
        a.append(v)
    out = {}
    for n, lst in acc.items():
        out[n] = {key: round(float(np.nanmean([d[key] for d in lst])) / (1.0 if key == "ring_wait_frac" else 1e3), 3)
                  for key in lst[0]}
    # attention (layer l between GEMV rows 4l and 4l+1), from the qkv GEMV's last CTA end:
    # first CTA start, last CTA past its wait, means of q ready / blocks / ticket per CTA, the
    # merging CTAs' merge, last CTA end; then the o GEMV's last CTA past its wait
    att = []
    for l in range(cfg.n_layers):
        r = tat[l][tat[l][:, 5] > 0]
        if len(r) == 0:
            continue
        qkv_end = t[4 * l][t[4 * l][:, 0] > 0][:, 5].max()
        o = t[4 * l + 1][t[4 * l + 1][:, 0] > 0]
        mg = r[r[:, 6] == 1]
        att.append({"first_start": r[:, 0].min() - qkv_end, "first_past_wait": r[:, 1].min() - qkv_end,
                    "last_past_wait": r[:, 1].max() - qkv_end,
                    "q_ready": (r[:, 2] - r[:, 1]).mean(), "blocks": (r[:, 3] - r[:, 2]).mean(),
                    "ticket": (r[:, 4] - r[:, 3]).mean(),
                    "merge": (mg[:, 5] - mg[:, 4]).mean() if len(mg) else float("nan"),
                    "last_end": r[:, 5].max() - qkv_end, "o_past_wait": o[:, 1].max() - qkv_end})
    if att:
        out["attention"] = {k: round(float(np.nanmean([a[k] for a in att])) / 1e3, 3) for k in att[0]}
    # the merges (batch 3-32), from their GEMV's last CTA end: first CTA start, first and last
    # CTA past the wait, last CTA done with its outputs, last CTA end, and the next launch's
    # first CTA past its wait (attention after q|k|v, else the next GEMV)
    if tm is not None and (tm[:, :, 0] > 0).any():
        mg = {}
        for k in range(rows):
            m = tm[k][tm[k][:, 0] > 0]
            if len(m) == 0:
                continue
            g_end = t[k][t[k][:, 0] > 0][:, 5].max()
            kind = kinds[k]
            if kind == "qkv":
                a = tat[k // 4]
                a = a[a[:, 5] > 0]
                nxt = a[:, 1].min() if len(a) else float("nan")
            elif k + 1 < rows:
                nxt = t[k + 1][t[k + 1][:, 0] > 0][:, 1].min()
            else:
                nxt = float("nan")
            mg.setdefault(kind, []).append({
                "first_start": m[:, 0].min() - g_end, "first_past_wait": m[:, 1].min() - g_end,
                "last_past_wait": m[:, 1].max() - g_end, "last_done": m[:, 2].max() - g_end,
                "last_end": m[:, 3].max() - g_end, "next_past_wait": nxt - g_end})
        out["merge"] = {n: {key: round(float(np.nanmean([d[key] for d in lst])) / 1e3, 3) for key in lst[0]}
                        for n, lst in mg.items()}
    out["total_step_us"] = round((t[rows - 1][:, 5].max() - t[0][t[0][:, 0] > 0][:, 0].min()) / 1e3, 1)
    return out


def step_phases(gm, sargs, s, cfg):
    """Per-phase times of the persistent step from its globaltimer trace (untimed eager steps
    after the timed region): for each phase kind the mean over layers of the critical work time
    (last CTA arriving at the phase's barrier minus the last CTA leaving the previous one) and of
    the barrier time (last exit minus last arrival), plus the mean per-CTA work time."""
    import numpy as np
    import torch
    import quantized_transformer_decode_ql_gb300 as ql
    grid = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    rows = 3 + 5 * cfg.n_layers
    buf = torch.zeros(rows * grid * 8, dtype=torch.int64, device="cuda")
    gm.ql_model_set_option(ql.QL_OPT_STEP_TRACE, buf.data_ptr())
    try:
        for _ in range(2):
            gm.ql_decode_step(sargs, s)
        s.synchronize()
        buf.zero_()   # stamps of the last step only (a CTA stamps only the phases it works in)
        gm.ql_decode_step(sargs, s)
        s.synchronize()
    finally:
        gm.ql_model_set_option(ql.QL_OPT_STEP_TRACE, 0)
    gm.ql_check_device_error()
    t = ns_relative(buf.cpu().numpy().reshape(rows, grid, 8), 8)
    arrive, leave = t[:, :, 0], t[:, :, 1]
    kinds = ["embed"] + [k for _ in range(cfg.n_layers) for k in ("qkv", "attn", "o", "gate_up", "down")] + ["lm_head"]
    acc = {}
    for k in range(1, rows):
        name = kinds[k - 1]
        work = arrive[k].max() - leave[k - 1].max()
        bar = leave[k].max() - arrive[k].max()
        mean_cta = (arrive[k] - leave[k - 1]).mean()
        # steps inside the phase (mean over the CTAs that stamped them), from the previous exit
        st = []
        for i in range(2, 6):
            v = t[k, :, i]
            ok = v > 0
            st.append(float((v[ok] - leave[k - 1][ok]).mean()) if ok.any() else float("nan"))
        a = acc.setdefault(name, [0.0, 0.0, 0.0, 0, np.zeros(4)])
        a[0] += work; a[1] += bar; a[2] += mean_cta; a[3] += 1; a[4] += np.array(st)
    out = {n: {"work": round(a[0] / a[3] / 1e3, 2), "barrier": round(a[1] / a[3] / 1e3, 2),
               "mean_cta_work": round(a[2] / a[3] / 1e3, 2), "count": a[3],
               "steps": [round(x / a[3] / 1e3, 2) for x in a[4]]} for n, a in acc.items()}
    # GEMV phases: warp 0's share of its unit loop spent waiting for ring slots (clock cycles)
    for n in ("qkv", "o", "gate_up", "down", "lm_head"):
        ks = [k for k in range(1, rows) if kinds[k - 1] == n]
        wait = t[ks, :, 6].sum()
        loop = t[ks, :, 7].sum()
        if loop > 0:
            out[n]["ring_wait_frac"] = round(float(wait / loop), 3)
    out["total_step_us"] = round((leave[rows - 1].max() - leave[0].min()) / 1e3, 1)
    return out


# ----------------------------------------------------------------------------- CPU oracle arm
def oracle_sample(budget_s: float = 20.0):
    """Time the f64 oracle on a bounded sample of the batch-1 8B-shaped decode: one full decode
    step of layer 0 (attention over a 2048-position f16 context) and the lm_head on a slice of
    rows, then scale to one token (36 layers + the whole vocabulary). Returns (tokens/s, info)."""
    from oracle import decode, ops

    cfg = ql_inputs.QWEN3_8B
    lm_rows = 8192
    one = ql_inputs.Config(**{**cfg.as_dict(), "n_layers": 1, "vocab": lm_rows})
    w = {"embed": ql_inputs._normal(ql_inputs.sub_rng(0, 0, 0), (lm_rows, cfg.hidden), 0.02),
         "final_norm": ql_inputs.layer_tensor(cfg, 0, 0, "attn_norm"),
         "lm_head": ql_inputs.gemv_weight(lm_rows, cfg.hidden, seed=2),
         "layers": [{n: ql_inputs.layer_tensor(cfg, 0, 0, n) for n in
                     ("attn_norm", "ffn_norm", "q_norm", "k_norm", "wqkv", "wo", "wgu", "wd")}]}
    model = decode.Q4Model(one, w)
    k, v = ql_inputs.kv_context(1, cfg.n_kv_heads, cfg.head_dim, CTX, seed=4)
    cache = decode.KVCache(one, 1, CTX + 64)
    cache.preload(0, k, v)
    hf = np.random.default_rng(0).standard_normal((1, cfg.hidden))
    t_layer, t_lm, n = [], [], 0
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        decode.decode_step(model, cache, [1], [CTX + n])          # layer 0 + lm_head slice
        t1 = time.perf_counter()
        ops.gemv(model.dense(model.lm_head), hf)                   # the lm_head slice alone
        t2 = time.perf_counter()
        t_layer.append((t1 - t0) - (t2 - t1))
        t_lm.append(t2 - t1)
        n += 1
        if time.perf_counter() - t_start > budget_s or n >= 8:
            break
    tl, tm = statistics.median(t_layer), statistics.median(t_lm)
    t_token = cfg.n_layers * tl + tm * (cfg.vocab / lm_rows)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    info = {"kind": "oracle", "cores": cores,
            "sample": (f"{n} oracle decode steps of layer 0 (2048-position f16 context) + lm_head on "
                       f"{lm_rows} of {cfg.vocab} rows, scaled to 36 layers + full vocab; "
                       f"{tl:.2f} s/layer, {tm:.2f} s per lm_head slice"),
            "s_per_token": t_token}
    return 1.0 / t_token, info


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    budget = max(10.0, min(120.0, 6.0 * (args.steps + args.warmup)))
    tps, info = oracle_sample(budget_s=budget)
    cpu = {"value": round(tps, 6), "unit": "tokens/s", "cores": info["cores"], "kind": "oracle",
           "sample": info["sample"]}
    return {
        "metric": METRIC, "value": round(tps, 6), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 / tps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": f"qwen3-8b-shaped q4_0 decode, batch 1, {CTX}-token context, {args.steps} greedy steps"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(tps, 6), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- kernel microbenchmarks
def micro_gemv(shapes, batches, iters):
    """q4_0 GEMV alone on the projection shapes; rotates weight copies totalling > 3x L2."""
    import torch
    from quantized_transformer_decode_ql_gb300 import build as qbuild
    qbuild.build()
    import quantized_transformer_decode_ql_gb300 as ql
    from quantized_transformer_decode_ql_gb300.model import Q4Tensor
    peak, src = load_peaks()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    s = torch.cuda.Stream()
    g = torch.Generator(device="cuda")
    g.manual_seed(2)
    out = []
    for rows, cols in shapes:
        one = rows * cols * 18 // 32
        copies = max(1, min(64, -(-3 * l2 // one)))
        Ws = []
        for c in range(copies):
            w = torch.randn((rows, cols), generator=g, device="cuda").mul_(0.02)
            Ws.append(Q4Tensor.pack(w))
            del w
        torch.cuda.synchronize()      # packing runs on the default stream; time nothing before it ends
        for B in batches:
            x = torch.randn((B, cols), generator=g, device="cuda").half()
            y = torch.empty((B, rows), dtype=torch.float32, device="cuda")

            def run(n):
                for i in range(n):
                    W = Ws[i % copies]
                    ql.ql_gemv_q4_0(W.scales, W.quants, rows, cols, x, B, y, 0, 0, None, s)
            n = max(iters, copies)
            with torch.cuda.stream(s):
                run(1)                  # first call outside capture (per-device set-up)
            s.synchronize()
            us = graph_ms(lambda: run(n), s, 3) * 1e3 / n
            nbytes = one + B * cols * 2 + B * rows * 4
            gbs = nbytes / (us * 1e-6) / 1e9
            out.append({"kernel": "ql_gemv_q4_0", "rows": rows, "cols": cols, "batch": B,
                        "us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                        "peak": peak, "peak_source": src, "copies": copies})
            print(json.dumps(out[-1]), flush=True)
        del Ws
    return out


def micro_gemv_stream(shapes, batches, iters):
    """q4_0 GEMV over the tile stream layout alone (batch 1-2: the CUDA-core stream kernel,
    3-32: the split-K tensor-core kernel plus its merge), plain epilogue; rotates weight copies
    totalling > 3x L2."""
    import torch
    from quantized_transformer_decode_ql_gb300 import build as qbuild
    qbuild.build()
    import quantized_transformer_decode_ql_gb300 as ql
    from quantized_transformer_decode_ql_gb300.model import Q4Tensor
    peak, src = load_peaks()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    s = torch.cuda.Stream()
    g = torch.Generator(device="cuda")
    g.manual_seed(2)
    out = []
    for rows, cols in shapes:
        one = rows * cols * 18 // 32
        copies = max(1, min(64, -(-3 * l2 // one)))
        Ws = []
        for c in range(copies):
            w = torch.randn((rows, cols), generator=g, device="cuda").mul_(0.02)
            W = Q4Tensor.pack(w)
            del w
            buf = torch.empty(ql.ql_q4_0_stream_bytes(rows, cols, 0), dtype=torch.uint8, device="cuda")
            ql.ql_q4_0_stream_pack(W.scales, W.quants, rows, cols, 0, buf)
            del W
            Ws.append(buf)
        torch.cuda.synchronize()
        for B in batches:
            x = torch.randn((B, cols), generator=g, device="cuda").half()
            y = torch.empty((B, rows), dtype=torch.float32, device="cuda")
            ws = None
            if B > 2:
                ws = torch.zeros(ql.ql_gemv_q4_0_stream_workspace_bytes(rows, cols, 0), dtype=torch.uint8,
                                 device="cuda")

            def run(n):
                for i in range(n):
                    ql.ql_gemv_q4_0_stream(Ws[i % copies], rows, cols, x, B, y, ql.QL_EPI_NONE, ws, s)
            n = max(iters, copies)
            with torch.cuda.stream(s):
                run(1)                  # first call outside capture (per-device set-up)
            s.synchronize()
            us = graph_ms(lambda: run(n), s, 3) * 1e3 / n
            nbytes = one + B * cols * 2 + B * rows * 4
            gbs = nbytes / (us * 1e-6) / 1e9
            out.append({"kernel": "ql_gemv_q4_0_stream", "rows": rows, "cols": cols, "batch": B,
                        "us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                        "peak": peak, "peak_source": src, "copies": copies})
            print(json.dumps(out[-1]), flush=True)
        del Ws
    return out


def micro_gemm(shapes, tokens, iters):
    """The prompt-chunk q4_0 GEMM (tcgen05) alone: T tokens x the tile stream copy, plain
    epilogue; rotates weight copies totalling > 3x L2. Reports us per call, the weight bytes'
    rate and TFLOP/s (2 T rows cols flops) against the measured bf16 peak."""
    import torch
    from quantized_transformer_decode_ql_gb300 import build as qbuild
    qbuild.build()
    import quantized_transformer_decode_ql_gb300 as ql
    from quantized_transformer_decode_ql_gb300.model import Q4Tensor
    peak, src = load_peaks()
    tf_peak = load_peaks_tflops()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    s = torch.cuda.Stream()
    g = torch.Generator(device="cuda")
    g.manual_seed(2)
    out = []
    for rows, cols in shapes:
        one = rows * cols * 18 // 32
        copies = max(1, min(64, -(-3 * l2 // one)))
        Ws = []
        for c in range(copies):
            w = torch.randn((rows, cols), generator=g, device="cuda").mul_(0.02)
            W = Q4Tensor.pack(w)
            del w
            buf = torch.empty(ql.ql_q4_0_stream_bytes(rows, cols, 0), dtype=torch.uint8, device="cuda")
            ql.ql_q4_0_stream_pack(W.scales, W.quants, rows, cols, 0, buf)
            del W
            Ws.append(buf)
        torch.cuda.synchronize()
        for T in tokens:
            x = torch.randn((T, cols), generator=g, device="cuda").half()
            y = torch.empty((T, rows), dtype=torch.float32, device="cuda")

            def run(n):
                for i in range(n):
                    ql.ql_gemm_q4_0_stream(Ws[i % copies], rows, cols, x, T, y, ql.QL_EPI_NONE, s)
            n = max(iters, copies)
            with torch.cuda.stream(s):
                run(1)
            s.synchronize()
            us = graph_ms(lambda: run(n), s, 3) * 1e3 / n
            tflops = 2.0 * T * rows * cols / (us * 1e-6) / 1e12
            gbs = one / (us * 1e-6) / 1e9
            out.append({"kernel": "ql_gemm_q4_0_stream", "rows": rows, "cols": cols, "tokens": T,
                        "us": round(us, 2), "TFLOP/s": round(tflops, 1),
                        "tflops_frac_of_bf16": round(tflops / tf_peak, 4) if tf_peak else None,
                        "weight_GB/s": round(gbs, 1), "copies": copies})
            print(json.dumps(out[-1]), flush=True)
        del Ws
    return out


def micro_attn(batches, iters, ctx=0):
    """Paged GQA decode attention alone: 32/8 heads, hd 128, lengths uniform in [512, 32768]
    (ctx > 0: every sequence ctx tokens long)."""
    import torch
    from quantized_transformer_decode_ql_gb300 import build as qbuild
    qbuild.build()
    import quantized_transformer_decode_ql_gb300 as ql
    peak, src = load_peaks()
    nh, nkv, hd = 32, 8, 128
    s = torch.cuda.Stream()
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    for B in batches:
        lens = ql_inputs.batched_lengths(B, 512, 32768, seed=6) if ctx <= 0 else np.full(B, ctx, dtype=np.int32)
        nblk = [(int(L) + 15) // 16 for L in lens]
        maxb = max(nblk)
        num_blocks = sum(nblk)
        perm = torch.from_numpy(ql_inputs.fragmented_block_ids(num_blocks, seed=5)).cuda()
        bt = torch.full((B, maxb), -1, dtype=torch.int32, device="cuda")
        off = 0
        for b, n in enumerate(nblk):
            bt[b, :n] = perm[off:off + n]
            off += n
        kp = torch.randn((num_blocks, nkv, 16, hd), generator=g, device="cuda").half()
        vp = torch.randn((num_blocks, nkv, 16, hd), generator=g, device="cuda").half()
        q = torch.randn((B, nh, hd), generator=g, device="cuda").half()
        o = torch.empty((B, nh * hd), dtype=torch.float16, device="cuda")
        cl = torch.from_numpy(lens).cuda()
        ws = torch.zeros(ql.ql_paged_attn_workspace_bytes(B, nh, nkv, hd, 16, maxb), dtype=torch.uint8, device="cuda")
        flush = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
        flush_sum = torch.zeros((), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()

        def run():
            ql.ql_paged_attn_decode(q, kp, vp, bt, cl, B, nh, nkv, hd, 16, maxb, num_blocks,
                                    1 / math.sqrt(hd), o, ws, s)
        with torch.cuda.stream(s):
            run()                       # first call outside capture (per-device set-up)
        s.synchronize()

        def flush_then_run():
            for _ in range(iters):
                flush_sum.copy_(flush.sum())   # read 256 MB: evicts the KV from L2, leaves no dirty lines
                run()

        def flush_only():
            for _ in range(iters):
                flush_sum.copy_(flush.sum())
        us = (graph_ms(flush_then_run, s, 3) - graph_ms(flush_only, s, 3)) * 1e3 / iters
        nbytes = sum(2 * int(L) * nkv * hd * 2 + 4 * ((int(L) + 15) // 16) for L in lens) + B * nh * hd * 4
        gbs = nbytes / (us * 1e-6) / 1e9
        print(json.dumps({"kernel": "ql_paged_attn_decode", "batch": B, "sum_len": int(lens.sum()),
                          "us": round(us, 2), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
                          "peak": peak, "peak_source": src}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ql", choices=["ql", "reference"])
    ap.add_argument("--config", default="e1", choices=["e1", "e32", "prefill"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e32", action="store_true", help="leave the batch-32 sub-results out of the default line")
    ap.add_argument("--kv", default="f16", choices=["f16", "q8q5"], help="--config e32: KV cache format")
    ap.add_argument("--no-moe", action="store_true", help="leave the routed-expert sub-result out of the default line")
    ap.add_argument("--no-prefill", action="store_true", help="leave the prefill sub-result out of the default line")
    ap.add_argument("--chunk", type=int, default=256, help="--config prefill: prompt tokens per chunk (1-256)")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling aid: run the 8B-shaped step with this many layers (default: all 36)")
    ap.add_argument("--step-kernel", default="auto", choices=["auto", "persistent", "launches"],
                    help="decode step implementation (auto: persistent when the batch allows it)")
    ap.add_argument("--micro", choices=["gemv", "gemv_stream", "gemm", "attn"], help="time one kernel family alone")
    ap.add_argument("--shape", default=None, help="micro gemv: ROWSxCOLS (default: all shapes)")
    ap.add_argument("--batch", default=None, help="micro: comma-separated batch sizes")
    ap.add_argument("--iters", type=int, default=50)
    ap.add_argument("--ctx", type=int, default=0, help="micro attn: one context length for every sequence")
    args = ap.parse_args()
    if args.micro == "gemv":
        shapes = [tuple(int(v) for v in args.shape.split("x"))] if args.shape else ql_inputs.GEMV_SHAPES
        batches = [int(b) for b in args.batch.split(",")] if args.batch else [1, 4, 16, 64]
        micro_gemv(shapes, batches, args.iters)
        return
    if args.micro == "gemv_stream":
        shapes = [tuple(int(v) for v in args.shape.split("x"))] if args.shape else ql_inputs.GEMV_SHAPES
        batches = [int(b) for b in args.batch.split(",")] if args.batch else [1, 2, 8, 32]
        micro_gemv_stream(shapes, batches, args.iters)
        return
    if args.micro == "gemm":
        shapes = [tuple(int(v) for v in args.shape.split("x"))] if args.shape else ql_inputs.GEMV_SHAPES
        tokens = [int(b) for b in args.batch.split(",")] if args.batch else [128, 256]
        micro_gemm(shapes, tokens, args.iters)
        return
    if args.micro == "attn":
        batches = [int(b) for b in args.batch.split(",")] if args.batch else [1, 2, 4, 8, 16, 32, 64]
        micro_attn(batches, args.iters, args.ctx)
        return
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        line = reference_arm(args, rank, 1 if rank == 0 else world)
        if line is not None:
            line["n_gpus"] = args.gpus
            print(json.dumps(line), flush=True)
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"
    if args.config == "e32":
        line = gpu_arm_e32(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.config == "prefill":
        line = gpu_arm_prefill(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    line = gpu_arm(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            tps, info = oracle_sample(budget_s=20.0)
            line["cpu_baseline"] = {"value": round(tps, 6), "unit": "tokens/s", "cores": info["cores"],
                                    "kind": "oracle", "sample": info["sample"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
