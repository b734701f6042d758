"""q4_0 GEMV on the GPU against the oracle (f64 dense product of the dequantised weights).

Tolerance, from the kernel's arithmetic: activations are staged in f16 (exact here, since the
tests give f16 activations; x/16 for the high nibbles is exact too). Each weight enters the
tensor-core MMA as an exact f16 (1024 + q or 1024 + 16 q), every product is exact in f32 and the
MMA sums them in f32; the 1032 / 1152 offsets are taken out in f32 with the block's sum of
activations and the block's f16 scale d multiplies the result. The largest rounding is the
cancellation of that offset, about 1032 * 2^-24 * sum|x| per block, so for N(0, 0.02) weights and
N(0, 1) activations the expected error is ~1e-4 of the output rms and the bar
``|y - y_ref| <= 1e-2 * rms(y_ref) + 1e-2 * |y_ref|`` leaves room for f16 outputs' own rounding.
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import ops, q4_0 as oq

from gpu_util import lib, dev, q4_dev, rel_err

pytestmark = pytest.mark.gpu


def run_gemv(w, x, epilogue=0, y_dtype=0, residual=None):
    ql = lib()
    rows, cols = w.shape
    batch = x.shape[0]
    s, q = oq.quantize(w)
    ref = ops.gemv(oq.dequantize(s, q), x.astype(np.float64))
    ds, dq = q4_dev(s, q)
    dx = dev(x)
    out_rows = rows // 2 if epilogue == ql.QL_EPI_SILU_MUL else rows
    tdt = torch.float16 if y_dtype == ql.QL_DTYPE_F16 else torch.float32
    y = torch.full((batch, out_rows), float("nan"), dtype=tdt, device="cuda")
    dres = None
    if residual is not None:
        dres = dev(residual.astype(np.float32))
        y = dres if y_dtype == 0 else y
    ql.ql_gemv_q4_0(ds, dq, rows, cols, dx, batch, y, y_dtype, epilogue, dres)
    torch.cuda.synchronize()
    return y.float().cpu().numpy().astype(np.float64), ref


def check_close(got, want, what):
    rms = np.sqrt(np.mean(want * want))
    err = np.abs(got - want)
    bad = err > 1e-2 * rms + 1e-2 * np.abs(want)
    assert not np.any(np.isnan(got)), what
    assert not bad.any(), f"{what}: {bad.sum()} outside tolerance, max rel err {rel_err(got, want):.3e}"


SHAPES = [(8, 32), (37, 96), (256, 256), (512, 768), (1000, 4096), (4099, 1024), (96, 12288)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("batch", [1, 2, 3, 4, 5, 8, 9, 16, 33, 64])
def test_gemv_plain(rows, cols, batch):
    w = ql_inputs.gemv_weight(rows, cols, seed=2)
    x = ql_inputs.gemv_activations(batch, cols, seed=3)
    got, ref = run_gemv(w, x)
    check_close(got, ref, f"gemv {rows}x{cols} b{batch}")


@pytest.mark.parametrize("batch", [1, 3, 8])
def test_gemv_f16_out_and_residual(batch):
    ql = lib()
    w = ql_inputs.gemv_weight(300, 512, seed=5)
    x = ql_inputs.gemv_activations(batch, 512, seed=6)
    got, ref = run_gemv(w, x, y_dtype=ql.QL_DTYPE_F16)
    check_close(got, ref, "f16 out")
    res = np.random.default_rng(1).standard_normal((batch, 300))
    got, ref = run_gemv(w, x, epilogue=ql.QL_EPI_ADD_RESIDUAL, residual=res)
    want = ref + res.astype(np.float32).astype(np.float64)
    check_close(got, want, "residual")


@pytest.mark.parametrize("batch", [1, 2, 5, 16])
@pytest.mark.parametrize("inter", [96, 768, 1000])
def test_gemv_silu_mul(batch, inter):
    ql = lib()
    w = ql_inputs.gemv_weight(2 * inter, 256, seed=7)
    x = ql_inputs.gemv_activations(batch, 256, seed=8)
    for ydt in (ql.QL_DTYPE_F32, ql.QL_DTYPE_F16):
        got, ref = run_gemv(w, x, epilogue=ql.QL_EPI_SILU_MUL, y_dtype=ydt)
        want = ops.swiglu(ref[:, :inter], ref[:, inter:])
        check_close(got, want, f"silu_mul dtype {ydt}")


def test_gemv_zero_and_extreme_blocks():
    # all-zero rows (d = 0), single large outlier per block, codes at both ends
    w = np.zeros((64, 256), np.float32)
    w[1, ::32] = 5.0
    w[2, 5::32] = -3.0
    w[3] = np.linspace(-1, 1, 256, dtype=np.float32)
    w[4:] = ql_inputs.gemv_weight(60, 256, seed=9)
    x = ql_inputs.gemv_activations(2, 256, seed=10)
    got, ref = run_gemv(w, x)
    assert np.all(got[:, 0] == 0.0)
    check_close(got, ref, "extreme blocks")


_FULL = {}


def full_size_matrix(rows, cols):
    """Weights of one microbenchmark shape, packed by the library's host codec (cached)."""
    if (rows, cols) not in _FULL:
        ql = lib()
        _FULL.clear()
        w = ql_inputs.gemv_weight(rows, cols, seed=2)
        s = np.empty((rows, cols // 32), np.uint16)
        q = np.empty((rows, cols // 32, 16), np.uint8)
        ql.ql_q4_0_pack(w, s, q)
        _FULL[(rows, cols)] = (w, q4_dev(s, q))
    return _FULL[(rows, cols)]


@pytest.mark.slow
@pytest.mark.parametrize("rows,cols", [(151936, 4096), (24576, 4096), (4096, 12288)])
@pytest.mark.parametrize("batch", [1, 4, 16, 64])
def test_gemv_full_size_sampled_rows(rows, cols, batch):
    """The microbenchmark shapes at full size: the GPU computes every row from the product
    packer's codes; the oracle quantises and computes 256 sampled rows on its own."""
    ql = lib()
    w, (ds, dq) = full_size_matrix(rows, cols)
    x = ql_inputs.gemv_activations(batch, cols, seed=3)
    y = torch.empty((batch, rows), dtype=torch.float32, device="cuda")
    ql.ql_gemv_q4_0(ds, dq, rows, cols, dev(x), batch, y)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    idx = np.sort(np.random.default_rng(rows).choice(rows, 256, replace=False))
    idx[-1] = rows - 1
    so, qo = oq.quantize(w[idx])
    ref = ops.gemv(oq.dequantize(so, qo), x.astype(np.float64))
    check_close(got[:, idx], ref, f"full {rows}x{cols} b{batch}")
