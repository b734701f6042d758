"""Host-side helpers of ``bench.py`` (no GPU): the trace-stamp conversion and the launch count
that the benchmark line claims."""
import dataclasses

import numpy as np

import bench
import ql_inputs


def test_trace_stamps_keep_nanoseconds():
    # globaltimer values near 1.8e18 ns: float64 alone would round them to 256 ns
    base = 1_800_000_000_000_000_123
    raw = np.zeros((2, 3, 8), dtype=np.int64)
    raw[0, 0, :3] = [base, base + 7, base + 1001]
    raw[1, 2, :2] = [base + 5, base + 6]
    raw[..., 6] = 11   # a statistics word, not a stamp
    out = bench.ns_relative(raw, 6)
    assert out.dtype == np.float64
    assert out[0, 0, 0] == 1.0                        # the earliest stamp becomes 1
    assert out[0, 0, 1] - out[0, 0, 0] == 7.0         # differences exact to the nanosecond
    assert out[0, 0, 2] - out[0, 0, 0] == 1001.0
    assert out[1, 2, 1] - out[1, 2, 0] == 1.0
    assert (out[0, 1, :6] == 0).all() and out[0, 0, 3] == 0   # unwritten stamps stay zero
    assert (out[..., 6] == 11).all()                  # other words untouched


def test_launches_per_step(monkeypatch):
    monkeypatch.delenv("QL_BATCHED_NORM_FOLD", raising=False)
    cfg = ql_inputs.QWEN3_8B
    L = cfg.n_layers
    # batch 1-2: embed, per layer q|k|v, attention, o, gate|up, down, then lm_head, finalize
    assert bench.launches_per_step(cfg, 1) == 3 + 5 * L
    assert bench.launches_per_step(cfg, 2) == 3 + 5 * L
    # batch 3-32: every GEMV plus its merge and the attention (9 per layer); embed, layer 0's
    # RMSNorm, lm_head and its merge, finalize. The ncu launch list of the batch-32 step has,
    # per 36-layer step, 144 + 1 GEMVs, as many merges, 36 attentions and 1 RMSNorm.
    assert bench.launches_per_step(cfg, 32) == 5 + 9 * L
    assert 5 + 9 * 36 == 1 + 1 + 36 * (4 + 4 + 1) + 2 + 1
    small = dataclasses.replace(cfg, n_layers=2)
    assert bench.launches_per_step(small, 1) == 13
    # with the fold switched off every RMSNorm'd GEMV (q|k|v, gate|up, lm_head) gets its kernel
    monkeypatch.setenv("QL_BATCHED_NORM_FOLD", "0")
    assert bench.launches_per_step(cfg, 32) == 5 + 11 * L
