"""The full Qwen3-8B shape in the benchmark's decode configurations: 36 layers, the full
151,936-row vocabulary, batch 1 (the tile stream GEMVs) and batch 32 (the split-K tensor-core
GEMVs with the RMSNorm folded into their merges).

The f64 oracle cannot hold 36 layers of these weights, so the element-by-element comparison
with it is made at two layers of the same width (test_gpu_decode_full.py). At the full depth the
step is checked through properties that hold at any size:
* the replayed graph gives the eager step's logits and tokens bit for bit;
* identical sequences within a batch give identical logits bit for bit (2 at batch 2, 32 at
  batch 32). Across batch sizes the o GEMV's grid changes (it leaves one SM per attention merge,
  batch x kv heads of them), so its tiles' partial sums are grouped differently. Batch 2 then
  agrees with batch 1 within the step's logit tolerance (|d| <= 2e-2 + 1e-2 |w|).
* every greedy token is the argmax of the logits the step wrote (the first index among equal
  maxima).
The weights are seeded device draws (as in bench.py); every slot holds the same synthetic
N(0, 1) context in its own blocks of a fragmented pool.
"""
import numpy as np
import pytest
import torch

import ql_inputs

from oracle import decode

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu

CFG = ql_inputs.QWEN3_8B
N_POS = 256


def _model(max_batch):
    """A full-depth model whose every slot holds the same N_POS-position context."""
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    maxb = (N_POS + 8 + 15) // 16
    nb = max_batch * maxb
    gm = DeviceModel.from_layer_fn(CFG, ql_inputs.device_tensor_fn(CFG, seed=0), num_blocks=nb,
                                   max_batch=max_batch, max_blocks_per_seq=maxb)
    bt = ql_inputs.fragmented_block_ids(nb, seed=5).reshape(max_batch, maxb).copy()
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    nblk = (N_POS + 15) // 16
    shape = (CFG.n_layers, nblk, CFG.n_kv_heads, 16, CFG.head_dim)
    k = torch.randn(shape, generator=g, device="cuda").half()
    v = torch.randn(shape, generator=g, device="cuda").half()
    for b in range(max_batch):
        idx = torch.as_tensor(bt[b, :nblk], dtype=torch.long, device="cuda")
        gm.k_pool[:, idx] = k
        gm.v_pool[:, idx] = v
    return gm, bt


def _step(gm, bt, B, token, graph=False):
    """One decode step of B slots (the first B rows of bt), all with `token` at position N_POS;
    returns (logits [B, vocab], next tokens [B])."""
    tokens = torch.full((B,), token, dtype=torch.int32, device="cuda")
    positions = torch.full((B,), N_POS, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    logits = torch.zeros((B, CFG.vocab), dtype=torch.float32, device="cuda")
    args = gm.step_args(tokens, positions, dev(bt[:B].copy()), nxt, logits=logits)
    if graph:
        s = torch.cuda.Stream()
        gm.ql_decode_graph_capture(args, s)
        positions.fill_(N_POS)
        tokens.fill_(token)
        with torch.cuda.stream(s):
            gm.ql_decode_graph_replay(B, 1, s)
        s.synchronize()
    else:
        gm.ql_decode_step(args)
    torch.cuda.synchronize()
    gm.ql_check_device_error()
    return logits.cpu().numpy().copy(), nxt.cpu().numpy().copy()


def _argmax_first(row):
    return int(np.flatnonzero(row == row.max())[0])


@pytest.mark.parametrize("B", [1, 32])
def test_full_depth_graph_equals_eager_and_identical_slots_agree(B):
    lib()
    gm, bt = _model(B)
    try:
        token = int(ql_inputs.prompt_tokens(1, CFG.vocab, seed=1)[0])
        le, te = _step(gm, bt, B, token)
        lg, tg = _step(gm, bt, B, token, graph=True)
        assert np.isfinite(le).all()
        assert np.array_equal(le, lg), "graph replay differs from the eager step"
        assert np.array_equal(te, tg)
        for b in range(B):
            assert np.array_equal(le[b], le[0]), f"slot {b} differs from slot 0 on identical inputs"
            assert int(te[b]) == _argmax_first(le[b]), f"slot {b}: the token is not the logits' argmax"
    finally:
        gm.close()


def test_full_depth_two_identical_slots_equal_batch_one():
    lib()
    gm, bt = _model(2)
    try:
        token = int(ql_inputs.prompt_tokens(1, CFG.vocab, seed=1)[0])
        l1, t1 = _step(gm, bt, 1, token)
        l2, t2 = _step(gm, bt, 2, token)
        assert np.array_equal(l2[1], l2[0]), "two identical slots differ"
        assert decode.logits_close(l2[0].astype(np.float64), l1[0].astype(np.float64)).all()
        assert int(t2[0]) == int(t2[1]) == _argmax_first(l2[0])
        assert int(t1[0]) == _argmax_first(l1[0])
        if decode.greedy_must_agree(l1[0].astype(np.float64)):
            assert int(t2[0]) == int(t1[0])
    finally:
        gm.close()
