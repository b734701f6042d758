"""The q4_0 GEMV over the tile stream layout, batch 1-32 (ql_q4_0_stream_pack, ql_gemv_q4_0_stream).

Layout: bit-exact against a NumPy restatement of the documented layout (16-row tiles, units of
4 blocks x 16 rows of codes then the rows' 4 scales, gate/up row pairing for SiLU*up, zero
rows past the matrix).

GEMV: against the oracle (f64 dense product of the dequantised weights). Tolerance, from the
kernel's arithmetic. Batch 1-2: activations become 16-bit fixed point with a power-of-two scale
per 32-element block (rounding error at most 2^-16 of the block's largest |x| per element), and
the products and each block's sum are exact integers. Batch 3-32: activations f16, (q - 8) d
rounded once to f16, tensor-core products and sums in f32. Blocks are scaled and summed in f32.
For N(0, 0.02) weights and N(0, 1) activations that is ~1e-3 of the output rms or less, so the
bar is
``|y - y_ref| <= 1e-2 * rms(y_ref) + 1e-2 * |y_ref|``, the same as the row-major GEMV.
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import ops, q4_0 as oq

from gpu_util import lib, dev, q4_dev, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["mma_sync", "tcgen05"])
def form(request):
    """Both tensor-core forms of the batch 3-32 GEMV (restored afterwards)."""
    ql = lib()
    f = ql.QL_BATCHED_MMA_SYNC if request.param == "mma_sync" else ql.QL_BATCHED_TCGEN05
    prev = ql.ql_set_batched_gemv_form(f)
    yield request.param
    ql.ql_set_batched_gemv_form(prev)


def tile_rows(rows, silu, tile):
    """Global rows of tile rows 0..15 (-1: past the matrix)."""
    if silu:
        half = rows // 2
        i = tile * 8 + np.arange(8)
        gate = np.where(i < half, i, -1)
        up = np.where(i < half, half + i, -1)
        return np.concatenate([gate, up])
    r = tile * 16 + np.arange(16)
    return np.where(r < rows, r, -1)


def expected_stream(scales, quants, silu):
    """The documented tile stream layout, restated with NumPy from the q4_0 arrays."""
    rows, nblk = scales.shape
    ntile = (rows // 2 + 7) // 8 if silu else (rows + 15) // 16
    nst = nblk // 4
    out = np.zeros((ntile, nst, 1152), np.uint8)
    sbytes = scales.view(np.uint8).reshape(rows, nblk, 2)
    for tile in range(ntile):
        rr = tile_rows(rows, silu, tile)
        for k in range(nst):
            unit = out[tile, k]
            for q in range(4):
                for r in range(16):
                    if rr[r] >= 0:
                        unit[(q * 16 + r) * 16:(q * 16 + r + 1) * 16] = quants[rr[r], 4 * k + q]
            for r in range(16):
                if rr[r] >= 0:
                    unit[1024 + r * 8:1024 + r * 8 + 8] = sbytes[rr[r], 4 * k:4 * k + 4].reshape(8)
    return out.reshape(-1)


def packed(w, silu):
    ql = lib()
    rows, cols = w.shape
    s, q = oq.quantize(w)
    ds, dq = q4_dev(s, q)
    n = ql.ql_q4_0_stream_bytes(rows, cols, silu)
    buf = torch.full((n,), 0xAB, dtype=torch.uint8, device="cuda")
    ql.ql_q4_0_stream_pack(ds, dq, rows, cols, silu, buf)
    torch.cuda.synchronize()
    return s, q, buf


@pytest.mark.parametrize("rows,cols,silu", [(16, 128, 0), (37, 256, 0), (200, 384, 1), (18, 128, 1)])
def test_stream_layout_bit_exact(rows, cols, silu):
    w = ql_inputs.gemv_weight(rows, cols, seed=21)
    s, q, buf = packed(w, silu)
    want = expected_stream(s, q, silu)
    assert np.array_equal(buf.cpu().numpy(), want)


def run(w, x, epilogue, residual=None):
    ql = lib()
    rows, cols = w.shape
    silu = 1 if epilogue == ql.QL_EPI_SILU_MUL else 0
    s, q, buf = packed(w, silu)
    ref = ops.gemv(oq.dequantize(s, q), x.astype(np.float64))
    B = x.shape[0]
    if epilogue == ql.QL_EPI_SILU_MUL:
        y = torch.full((B, rows // 2), float("nan"), dtype=torch.float16, device="cuda")
    elif epilogue == ql.QL_EPI_ADD_RESIDUAL:
        y = dev(residual.astype(np.float32))
    else:
        y = torch.full((B, rows), float("nan"), dtype=torch.float32, device="cuda")
    ws = None
    if B > 2:   # scratch, zero-filled before its first use (the calls keep it valid)
        ws = torch.zeros((ql.ql_gemv_q4_0_stream_workspace_bytes(rows, cols, silu),), dtype=torch.uint8,
                         device="cuda")
    y0 = y.clone()
    ql.ql_gemv_q4_0_stream(buf, rows, cols, dev(x), B, y, epilogue, ws)
    torch.cuda.synchronize()
    if ws is not None:
        # a second call on the same workspace gives the same bits (a fixed summation order)
        y2 = y0.clone()
        ql.ql_gemv_q4_0_stream(buf, rows, cols, dev(x), B, y2, epilogue, ws)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)
    return y.float().cpu().numpy().astype(np.float64), ref


def check_close(got, want, what):
    rms = np.sqrt(np.mean(want * want))
    err = np.abs(got - want)
    bad = err > 1e-2 * rms + 1e-2 * np.abs(want)
    assert not np.any(np.isnan(got)), what
    assert not bad.any(), f"{what}: {bad.sum()} outside tolerance, max rel err {rel_err(got, want):.3e}"


@pytest.mark.parametrize("rows,cols", [(16, 128), (37, 256), (1000, 4096), (4099, 1024), (96, 12288), (6144, 4096)])
@pytest.mark.parametrize("batch", [1, 2])
def test_stream_gemv_plain(rows, cols, batch):
    ql = lib()
    w = ql_inputs.gemv_weight(rows, cols, seed=2)
    x = ql_inputs.gemv_activations(batch, cols, seed=3)
    got, ref = run(w, x, ql.QL_EPI_NONE)
    check_close(got, ref, f"stream gemv {rows}x{cols} b{batch}")


@pytest.mark.parametrize("batch", [1, 2])
def test_stream_gemv_residual(batch):
    ql = lib()
    w = ql_inputs.gemv_weight(300, 512, seed=5)
    x = ql_inputs.gemv_activations(batch, 512, seed=6)
    res = np.random.default_rng(1).standard_normal((batch, 300))
    got, ref = run(w, x, ql.QL_EPI_ADD_RESIDUAL, residual=res)
    check_close(got, ref + res.astype(np.float32).astype(np.float64), "residual")


@pytest.mark.parametrize("batch", [1, 2])
@pytest.mark.parametrize("inter", [8, 100, 768, 12288])
def test_stream_gemv_silu_mul(batch, inter):
    ql = lib()
    w = ql_inputs.gemv_weight(2 * inter, 256, seed=7)
    x = ql_inputs.gemv_activations(batch, 256, seed=8)
    got, ref = run(w, x, ql.QL_EPI_SILU_MUL)
    want = ops.swiglu(ref[:, :inter], ref[:, inter:])
    check_close(got, want, f"silu_mul {inter}")


def test_stream_gemv_zero_and_extreme_blocks():
    ql = lib()
    w = np.zeros((64, 256), np.float32)
    w[1, ::32] = 5.0
    w[2, 5::32] = -3.0
    w[3] = np.linspace(-1, 1, 256, dtype=np.float32)
    w[4:] = ql_inputs.gemv_weight(60, 256, seed=9)
    x = ql_inputs.gemv_activations(2, 256, seed=10)
    got, ref = run(w, x, ql.QL_EPI_NONE)
    assert np.all(got[:, 0] == 0.0)
    check_close(got, ref, "extreme blocks")


@pytest.mark.parametrize("rows,cols", [(37, 256), (200, 384), (1000, 1024), (6144, 4096), (96, 12288)])
@pytest.mark.parametrize("batch", [3, 5, 8, 17, 32])
def test_stream_gemv_batched(rows, cols, batch, form):
    """Batches 3-32: every weight streamed once, K in windows of 1024 columns."""
    ql = lib()
    w = ql_inputs.gemv_weight(rows, cols, seed=12)
    x = ql_inputs.gemv_activations(batch, cols, seed=13)
    got, ref = run(w, x, ql.QL_EPI_NONE)
    check_close(got, ref, f"batched {rows}x{cols} b{batch}")


@pytest.mark.parametrize("batch", [3, 16, 32])
def test_stream_gemv_batched_epilogues(batch, form):
    ql = lib()
    w = ql_inputs.gemv_weight(300, 2048, seed=14)
    x = ql_inputs.gemv_activations(batch, 2048, seed=15)
    res = np.random.default_rng(2).standard_normal((batch, 300))
    got, ref = run(w, x, ql.QL_EPI_ADD_RESIDUAL, residual=res)
    check_close(got, ref + res.astype(np.float32).astype(np.float64), "batched residual")
    wg = ql_inputs.gemv_weight(2 * 700, 1024, seed=16)
    xg = ql_inputs.gemv_activations(batch, 1024, seed=17)
    got, ref = run(wg, xg, ql.QL_EPI_SILU_MUL)
    check_close(got, ops.swiglu(ref[:, :700], ref[:, 700:]), "batched silu_mul")


def test_stream_gemv_rejects_bad_arguments():
    ql = lib()
    t = torch.zeros(8192, dtype=torch.uint8, device="cuda")
    x = torch.zeros((33, 1152), dtype=torch.float16, device="cuda")
    y = torch.zeros((33, 16), dtype=torch.float32, device="cuda")
    for args in ((16, 128, 33), (16, 96, 1), (15, 128, 1), (16, 1152, 3)):
        rows, cols, batch = args
        epi = ql.QL_EPI_SILU_MUL if rows % 2 else ql.QL_EPI_NONE
        with pytest.raises(ql.QLError) as e:
            ql.ql_gemv_q4_0_stream(t, rows, cols, x, batch, y, epi)
        assert e.value.status == ql.QL_EINVAL
    # batches above 2 need a workspace of the size the shape asks for
    need = ql.ql_gemv_q4_0_stream_workspace_bytes(16, 1024, 0)
    assert need > 0
    for ws in (None, torch.zeros(need - 256, dtype=torch.uint8, device="cuda")):
        with pytest.raises(ql.QLError) as e:
            ql.ql_gemv_q4_0_stream(t, 16, 1024, x, 3, y, ql.QL_EPI_NONE, ws)
        assert e.value.status == ql.QL_EINVAL


def test_stream_gemv_batched_shared_workspace(form):
    """Matrices of different shapes take turns on one workspace (as the decode step's projections
    do): the results equal those of separate workspaces, bit for bit."""
    ql = lib()
    B = 8
    shapes = [(6144, 4096, 0), (1400, 1024, 1), (4096, 12288, 0), (300, 2048, 0)]
    mats, outs_sep, xs = [], [], []
    for i, (rows, cols, silu) in enumerate(shapes):
        w = ql_inputs.gemv_weight(rows, cols, seed=40 + i)
        _, _, buf = packed(w, silu)
        x = dev(ql_inputs.gemv_activations(B, cols, seed=50 + i))
        mats.append((rows, cols, silu, buf))
        xs.append(x)

    def call(k, ws):
        rows, cols, silu, buf = mats[k]
        epi = ql.QL_EPI_SILU_MUL if silu else ql.QL_EPI_NONE
        y = torch.zeros((B, rows // 2), dtype=torch.float16, device="cuda") if silu else \
            torch.zeros((B, rows), dtype=torch.float32, device="cuda")
        ql.ql_gemv_q4_0_stream(buf, rows, cols, xs[k], B, y, epi, ws)
        return y

    for k, (rows, cols, silu, _) in enumerate(mats):
        ws = torch.zeros(ql.ql_gemv_q4_0_stream_workspace_bytes(rows, cols, silu), dtype=torch.uint8, device="cuda")
        outs_sep.append(call(k, ws))
    shared = torch.zeros(max(ql.ql_gemv_q4_0_stream_workspace_bytes(r, c, s) for r, c, s, _ in mats),
                         dtype=torch.uint8, device="cuda")
    for _ in range(3):
        got = [call(k, shared) for k in range(len(mats))]
        torch.cuda.synchronize()
        for k in range(len(mats)):
            assert torch.equal(got[k], outs_sep[k]), f"matrix {k}"
