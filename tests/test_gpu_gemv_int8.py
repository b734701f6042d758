"""The int8 absmax activation form of the batch 1-2 q4_0 GEMV (ql_set_gemv_activation_form).

inferencelayer ``cuda_llm.rs``: ``CudaQwen3::absmax`` fills ``xs = [max|x|, 1/max|x|]`` before
every GEMV, which then reads its activation vector with that one scale. The oracle states that
form in ``oracle.act8`` (codes decided in f32, as on the page). Here:

* GEMV: the GPU against the oracle's dense product of the dequantised weights with the oracle's
  int8-dequantised activations. The inputs are f16 (exact in both), so both sides take the same
  codes, the products and block sums are exact integers on the GPU, and only the f32 scaling and
  summation of the blocks differ: the bar is ``1e-5 rms(y) + 1e-5 |y|`` (f32 outputs; SiLU*up is
  rounded to f16, ``2e-3 |y| + 1e-4 rms``). The same outputs also lie within the form's own
  error bound against the exact product, ``sum_k |w_k| max|x| / 254``.
* Decode step (tiny model, RMSNorm'd inputs): against the oracle's decode with every GEMV input
  taken through the same int8 form. The GPU decides each code from its own input vector (the
  RMSNorm in f32, the attention and SiLU*up outputs rounded to f16), the oracle from the f64
  value; where the two straddle a rounding boundary the code differs by one, which moves that
  product by a whole step (max|x| / 127), a larger jump than any rounding of the default form.
  The bar is therefore twice the step tolerance, ``4e-2 + 2e-2 |ref|``; the greedy token must
  match where the oracle's top-2 margin exceeds it.
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import act8, decode, ops, q4_0 as oq

from gpu_util import lib, dev, q4_dev

pytestmark = pytest.mark.gpu


@pytest.fixture
def int8_form():
    ql = lib()
    prev = ql.ql_set_gemv_activation_form(ql.QL_GEMV_ACT_INT8)
    yield
    ql.ql_set_gemv_activation_form(prev)


def stream(w, silu):
    ql = lib()
    rows, cols = w.shape
    s, q = oq.quantize(w)
    ds, dq = q4_dev(s, q)
    buf = torch.empty(ql.ql_q4_0_stream_bytes(rows, cols, silu), dtype=torch.uint8, device="cuda")
    ql.ql_q4_0_stream_pack(ds, dq, rows, cols, silu, buf)
    return s, q, buf


@pytest.mark.parametrize("rows,cols", [(16, 128), (37, 256), (1000, 4096), (96, 12288), (6144, 4096)])
@pytest.mark.parametrize("batch", [1, 2])
@pytest.mark.parametrize("epi", ["none", "resid", "silu"])
def test_int8_gemv_matches_oracle(int8_form, rows, cols, batch, epi):
    ql = lib()
    if epi == "silu" and rows % 2:
        rows += 1
    w = ql_inputs.gemv_weight(rows, cols, seed=2)
    x = ql_inputs.gemv_activations(batch, cols, seed=3)
    silu = 1 if epi == "silu" else 0
    s, q, buf = stream(w, silu)
    W = oq.dequantize(s, q)
    xh = act8.absmax_dequant(x.astype(np.float64))
    y8 = ops.gemv(W, xh)                                  # the int8 form's exact value
    resid = ql_inputs.gemv_activations(batch, rows, seed=9).astype(np.float32) if epi == "resid" else None
    if epi == "silu":
        h = rows // 2
        want = ops.swiglu(y8[:, :h], y8[:, h:])
        y = torch.full((batch, h), float("nan"), dtype=torch.float16, device="cuda")
        e = ql.QL_EPI_SILU_MUL
    elif epi == "resid":
        want = resid.astype(np.float64) + y8
        y = dev(resid)
        e = ql.QL_EPI_ADD_RESIDUAL
    else:
        want = y8
        y = torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda")
        e = ql.QL_EPI_NONE
    ql.ql_gemv_q4_0_stream(buf, rows, cols, dev(x), batch, y, e, None)
    torch.cuda.synchronize()
    got = y.float().cpu().numpy().astype(np.float64)
    assert not np.isnan(got).any()
    rms = np.sqrt(np.mean(want * want))
    tol = (2e-3 * np.abs(want) + 1e-4 * rms) if epi == "silu" else (1e-5 * rms + 1e-5 * np.abs(want))
    err = np.abs(got - want)
    assert (err <= tol).all(), f"max err {err.max():.3e} vs rms {rms:.3e}"
    if epi == "none":
        # the form's own bound against the exact product: half a code step per element
        exact = ops.gemv(W, x.astype(np.float64))
        m = np.abs(x.astype(np.float32)).max(axis=1).astype(np.float64)
        bound = (np.abs(W).sum(axis=1)[None, :] * (m[:, None] / 254.0)) * (1 + 1e-4) + 1e-6 * rms
        assert (np.abs(got - exact) <= bound).all()


def test_int8_decode_step_matches_oracle_int8_form(int8_form):
    lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    cfg = ql_inputs.TINY
    w = ql_inputs.weights(cfg, seed=0)
    gm = DeviceModel(cfg, w, num_blocks=16, max_batch=1, max_blocks_per_seq=4)
    try:
        om = decode.Q4Model(cfg, w)
        cache = decode.KVCache(cfg, 1, 64)
        bt = dev(ql_inputs.fragmented_block_ids(16, seed=5)[:4].reshape(1, 4).copy())
        tokens = torch.zeros(1, dtype=torch.int32, device="cuda")
        positions = torch.zeros(1, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
        logits = torch.zeros((1, cfg.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, bt, nxt, logits=logits)
        tok = int(ql_inputs.prompt_tokens(1, cfg.vocab, seed=1)[0])
        for step in range(12):
            want = decode.decode_step(om, cache, [tok], [step], act=act8.absmax_dequant)[0]
            tokens.fill_(tok)
            gm.ql_decode_step(args)
            torch.cuda.synchronize()
            got = logits.cpu().numpy()[0].astype(np.float64)
            err = np.abs(got - want)
            assert (err <= 4e-2 + 2e-2 * np.abs(want)).all(), f"step {step}: max err {err.max():.3e}"
            top = np.sort(want)[-2:]
            if top[1] - top[0] > 4e-2 + 2e-2 * abs(top[1]):
                assert int(nxt.item()) == int(decode.greedy(want))
            tok = int(decode.greedy(want))
        gm.ql_check_device_error()
    finally:
        gm.close()
