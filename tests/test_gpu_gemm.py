"""The q4_0 GEMM for prompt chunks over the tile stream layout (ql_gemm_q4_0_stream, tcgen05).

Against the oracle: the f64 dense product of the dequantised weights (the definition of the
GEMV, one output per token). The kernel's arithmetic is the batch 3-32 GEMV's: f16 activations,
(q - 8) d rounded once to f16, products and sums in f32, so the bar is the same:
``|y - y_ref| <= 1e-2 * rms(y_ref) + 1e-2 * |y_ref|``. Shapes cover partial row blocks (rows
not a multiple of 128, tiles past the matrix), partial token tiles (n_tokens not a multiple of
128) and every epilogue; a second call must give the same bits (one accumulator per output, K
in order).
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import ops, q4_0 as oq

from gpu_util import lib, dev, q4_dev, rel_err

pytestmark = pytest.mark.gpu


def packed(w, silu):
    ql = lib()
    rows, cols = w.shape
    s, q = oq.quantize(w)
    ds, dq = q4_dev(s, q)
    buf = torch.full((ql.ql_q4_0_stream_bytes(rows, cols, silu),), 0xAB, dtype=torch.uint8, device="cuda")
    ql.ql_q4_0_stream_pack(ds, dq, rows, cols, silu, buf)
    torch.cuda.synchronize()
    return s, q, buf


def run(w, x, epilogue, residual=None):
    ql = lib()
    rows, cols = w.shape
    silu = 1 if epilogue == ql.QL_EPI_SILU_MUL else 0
    s, q, buf = packed(w, silu)
    ref = ops.gemv(oq.dequantize(s, q), x.astype(np.float64))
    T = x.shape[0]
    if epilogue == ql.QL_EPI_SILU_MUL:
        y = torch.full((T, rows // 2), float("nan"), dtype=torch.float16, device="cuda")
    elif epilogue == ql.QL_EPI_ADD_RESIDUAL:
        y = dev(residual.astype(np.float32))
    else:
        y = torch.full((T, rows), float("nan"), dtype=torch.float32, device="cuda")
    y0 = y.clone()
    xd = dev(x)
    ql.ql_gemm_q4_0_stream(buf, rows, cols, xd, T, y, epilogue)
    torch.cuda.synchronize()
    y2 = y0.clone()
    ql.ql_gemm_q4_0_stream(buf, rows, cols, xd, T, y2, epilogue)
    torch.cuda.synchronize()
    assert torch.equal(y, y2), "two calls differ"
    ql.ql_check_device_error()
    return y.float().cpu().numpy().astype(np.float64), ref


def check_close(got, want, what):
    rms = np.sqrt(np.mean(want * want))
    err = np.abs(got - want)
    bad = err > 1e-2 * rms + 1e-2 * np.abs(want)
    assert not np.any(np.isnan(got)), what
    assert not bad.any(), f"{what}: {bad.sum()} outside tolerance, max rel err {rel_err(got, want):.3e}"


@pytest.mark.parametrize("rows,cols", [(37, 256), (128, 128), (200, 384), (1000, 1024), (6144, 4096), (96, 12288)])
@pytest.mark.parametrize("n_tokens", [1, 33, 128, 129, 256])
def test_gemm_plain(rows, cols, n_tokens):
    ql = lib()
    w = ql_inputs.gemv_weight(rows, cols, seed=31)
    x = ql_inputs.gemv_activations(n_tokens, cols, seed=32)
    got, ref = run(w, x, ql.QL_EPI_NONE)
    check_close(got, ref, f"gemm {rows}x{cols} T{n_tokens}")


@pytest.mark.parametrize("n_tokens", [40, 200])
def test_gemm_residual_and_silu(n_tokens):
    ql = lib()
    w = ql_inputs.gemv_weight(300, 2048, seed=33)
    x = ql_inputs.gemv_activations(n_tokens, 2048, seed=34)
    res = np.random.default_rng(3).standard_normal((n_tokens, 300))
    got, ref = run(w, x, ql.QL_EPI_ADD_RESIDUAL, residual=res)
    check_close(got, ref + res.astype(np.float32).astype(np.float64), "gemm residual")
    wg = ql_inputs.gemv_weight(2 * 700, 1024, seed=35)
    xg = ql_inputs.gemv_activations(n_tokens, 1024, seed=36)
    got, ref = run(wg, xg, ql.QL_EPI_SILU_MUL)
    check_close(got, ops.swiglu(ref[:, :700], ref[:, 700:]), "gemm silu_mul")


def test_gemm_full_width_gate_up():
    """The 8B gate|up shape (24576 x 4096, SiLU*up) for a 256-token chunk, on sampled rows."""
    ql = lib()
    rows, cols, T = 24576, 4096, 256
    w = ql_inputs.gemv_weight(rows, cols, seed=37)
    x = ql_inputs.gemv_activations(T, cols, seed=38)
    s, q, buf = packed(w, 1)
    y = torch.full((T, rows // 2), float("nan"), dtype=torch.float16, device="cuda")
    ql.ql_gemm_q4_0_stream(buf, rows, cols, dev(x), T, y, ql.QL_EPI_SILU_MUL)
    torch.cuda.synchronize()
    ql.ql_check_device_error()
    got = y.float().cpu().numpy().astype(np.float64)
    assert not np.isnan(got).any()
    pick = np.random.default_rng(4).choice(rows // 2, 64, replace=False)
    wd = oq.dequantize(s, q)
    g = ops.gemv(wd[pick], x.astype(np.float64))
    u = ops.gemv(wd[rows // 2 + pick], x.astype(np.float64))
    check_close(got[:, pick], ops.swiglu(g, u), "gate|up 256 tokens")


def test_gemm_rejects_bad_arguments():
    ql = lib()
    t = torch.zeros(8192, dtype=torch.uint8, device="cuda")
    x = torch.zeros((4, 256), dtype=torch.float16, device="cuda")
    y = torch.zeros((4, 16), dtype=torch.float32, device="cuda")
    for args in ((t, 16, 200, x, 4, y, ql.QL_EPI_NONE),      # cols % 128
                 (t, 16, 256, x, 0, y, ql.QL_EPI_NONE),      # no tokens
                 (t, 15, 256, x, 4, y, ql.QL_EPI_SILU_MUL),  # odd rows with SiLU*up
                 (t, 16, 256, x, 4, y, 7)):                  # unknown epilogue
        with pytest.raises(ql.QLError) as e:
            ql.ql_gemm_q4_0_stream(*args)
        assert e.value.status == ql.QL_EINVAL
