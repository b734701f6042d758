"""Whole decode step on the GPU (ql_decode_step / graphs) against the oracle.

Tiny config (hidden 256, 2 layers, 4/2 heads, hd 64, SwiGLU 768, vocab 1024): 16 prompt tokens
fed as sequential decode, then 16 greedy steps, teacher-forced with the oracle's tokens (a
legitimate near-tie flip cannot derail later steps). Bar: logits within 2e-2 + 1e-2 |ref|, and
the greedy token equal to the oracle's wherever the top-2 margin exceeds that tolerance.

The step has two implementations, selected with QL_OPT_STEP_KERNEL: one cooperative kernel for
the whole step (batches up to 2) and one launch per phase (any batch); the step tests run on
both.
"""
import numpy as np
import pytest
import torch

import ql_inputs
from oracle import decode

from gpu_util import lib, dev

pytestmark = pytest.mark.gpu

CFG = ql_inputs.TINY


MODES = ("persistent", "launches")


@pytest.fixture(scope="module")
def tiny_model():
    lib()
    from quantized_transformer_decode_ql_gb300.model import DeviceModel
    w = ql_inputs.weights(CFG, seed=0)
    gm = DeviceModel(CFG, w, num_blocks=64, max_batch=8, max_blocks_per_seq=4)
    om = decode.Q4Model(CFG, w)
    yield gm, om
    gm.close()


@pytest.fixture
def tiny(tiny_model):
    """The tiny model with the default step selection, restored after each test."""
    ql = lib()
    yield tiny_model
    tiny_model[0].ql_model_set_option(ql.QL_OPT_STEP_KERNEL, ql.QL_STEP_AUTO)
    tiny_model[0].ql_model_set_option(ql.QL_OPT_BARRIER_TIMEOUT_NS, 2_000_000_000)
    tiny_model[0].ql_model_set_option(ql.QL_OPT_TEST_BARRIER_EXTRA, 0)


def set_mode(gm, mode):
    ql = lib()
    gm.ql_model_set_option(ql.QL_OPT_STEP_KERNEL,
                           ql.QL_STEP_PERSISTENT if mode == "persistent" else ql.QL_STEP_LAUNCHES)


def test_persistent_kernel_is_available(tiny):
    gm, _ = tiny
    assert gm.ql_model_persistent_max_batch() == 2


def slot_tables(B, maxb, seed=5, num_blocks=64):
    ids = ql_inputs.fragmented_block_ids(num_blocks, seed=seed)
    return ids[: B * maxb].reshape(B, maxb).copy()


@pytest.mark.parametrize("mode", MODES)
def test_tiny_teacher_forced_32_steps(tiny, mode):
    gm, om = tiny
    set_mode(gm, mode)
    prompt = ql_inputs.prompt_tokens(16, CFG.vocab, seed=1)
    cache = decode.KVCache(CFG, 1, 32)
    bt = dev(slot_tables(1, 4))
    tokens = torch.zeros(1, dtype=torch.int32, device="cuda")
    positions = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    logits = torch.zeros((1, CFG.vocab), dtype=torch.float32, device="cuda")
    args = gm.step_args(tokens, positions, bt, nxt, logits=logits)
    tok = int(prompt[0])
    agreed = 0
    for step in range(32):
        want = decode.decode_step(om, cache, [tok], [step])[0]
        tokens.fill_(tok)
        gm.ql_decode_step(args)
        torch.cuda.synchronize()
        got = logits.cpu().numpy()[0].astype(np.float64)
        ok = decode.logits_close(got, want)
        assert ok.all(), f"step {step}: {np.sum(~ok)} logits off, max err {np.abs(got - want).max():.3e}"
        assert int(positions.item()) == step + 1
        g_tok = int(nxt.item())
        o_tok = int(decode.greedy(want))
        if decode.greedy_must_agree(want):
            assert g_tok == o_tok, f"step {step}"
            agreed += 1
        tok = int(prompt[step + 1]) if step + 1 < 16 else o_tok
    gm.ql_check_device_error()
    assert agreed >= 24


@pytest.mark.parametrize("B", (2, 3))   # 2: the persistent kernel; 3: one launch per phase
def test_graph_replay_equals_eager(tiny, B):
    gm, _ = tiny
    start = ql_inputs.prompt_tokens(B, CFG.vocab, seed=9)
    runs = []
    for mode in ("eager", "graph"):
        tokens = dev(start.astype(np.int32))
        positions = torch.zeros(B, dtype=torch.int32, device="cuda")
        out = torch.full((B, 64), -1, dtype=torch.int32, device="cuda")
        bt = dev(slot_tables(B, 4, seed=21))
        logits = torch.zeros((B, CFG.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, bt, tokens, logits=logits, out_tokens=out)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            if mode == "eager":
                for _ in range(12):
                    gm.ql_decode_step(args, s)
            else:
                gm.ql_decode_graph_capture(args, s)   # captured, not executed
                gm.ql_decode_graph_replay(B, 12, s)
        s.synchronize()
        runs.append((out.cpu().numpy(), logits.cpu().numpy(), positions.cpu().numpy()))
    assert np.array_equal(runs[0][0], runs[1][0])
    assert np.array_equal(runs[0][1], runs[1][1])
    assert np.all(runs[0][2] == 12)
    assert np.all(runs[0][0][:, 1:13] >= 0)


def test_graph_step_from_host_buffers(tiny):
    """ql_decode_graph_step_host (token ids in from pinned host memory, next tokens back) gives
    the same tokens, step for step, as replays of the same graph on device buffers, also with
    one host buffer as both input and output."""
    gm, _ = tiny
    B = 2
    start = ql_inputs.prompt_tokens(B, CFG.vocab, seed=11).astype(np.int32)
    seqs = []
    for mode in ("device", "host", "host_in_place"):
        tokens = dev(start)
        positions = torch.zeros(B, dtype=torch.int32, device="cuda")
        bt = dev(slot_tables(B, 4, seed=23))
        args = gm.step_args(tokens, positions, bt, tokens)
        s = torch.cuda.Stream()
        gm.ql_decode_graph_capture(args, s)
        got = []
        if mode == "device":
            for _ in range(10):
                gm.ql_decode_graph_replay(B, 1, s)
                s.synchronize()
                got.append(tokens.cpu().numpy().copy())
        elif mode == "host":
            h_in = torch.from_numpy(start.copy()).pin_memory()
            h_out = torch.zeros(B, dtype=torch.int32).pin_memory()
            for _ in range(10):
                gm.ql_decode_graph_step_host(B, h_in, h_out, s)
                got.append(h_out.numpy().copy())
                h_in.copy_(h_out)
        else:   # one buffer in and out: each step's tokens are the next input
            h_buf = torch.from_numpy(start.copy()).pin_memory()
            for _ in range(10):
                gm.ql_decode_graph_step_host(B, h_buf, h_buf, s)
                got.append(h_buf.numpy().copy())
        seqs.append(np.stack(got))
        assert np.all(positions.cpu().numpy() == 10)
    assert np.array_equal(seqs[0], seqs[1])
    assert np.array_equal(seqs[0], seqs[2])
    gm.ql_check_device_error()


def test_identical_slots_equal_batch_one(tiny):
    """Identical slots give bit-identical logits within a batch (the step treats the batch
    columns independently); across batch sizes and step kernels the f32 sums are taken in
    another order, so batch 1 and batches 2 and 4 agree within the logits tolerance."""
    gm, om = tiny
    tok0 = int(ql_inputs.prompt_tokens(1, CFG.vocab, seed=3)[0])
    res = {}
    for B in (1, 2, 4):
        tokens = torch.full((B,), tok0, dtype=torch.int32, device="cuda")
        positions = torch.zeros(B, dtype=torch.int32, device="cuda")
        bt = dev(slot_tables(B, 4, seed=31))
        logits = torch.zeros((B, CFG.vocab), dtype=torch.float32, device="cuda")
        args = gm.step_args(tokens, positions, bt, tokens, logits=logits)
        for _ in range(5):
            gm.ql_decode_step(args)
        torch.cuda.synchronize()
        res[B] = logits.cpu().numpy()
    for B in (2, 4):
        for b in range(B):
            assert np.array_equal(res[B][b], res[B][0])
        assert decode.logits_close(res[B][0].astype(np.float64), res[1][0].astype(np.float64)).all()


@pytest.mark.parametrize("mode", MODES)
def test_inactive_slot_is_frozen(tiny, mode):
    gm, _ = tiny
    set_mode(gm, mode)
    B = 2
    tokens = dev(np.array([5, 7], np.int32))
    positions = dev(np.array([0, 3], np.int32))
    active = dev(np.array([1, 0], np.int32))
    bt_np = slot_tables(B, 4, seed=41)
    bt = dev(bt_np)
    before = gm.k_pool[:, bt_np[1]].clone()
    args = gm.step_args(tokens, positions, bt, tokens, active=active)
    gm.ql_decode_step(args)
    torch.cuda.synchronize()
    assert positions.cpu().tolist() == [1, 3]
    assert int(tokens[1].item()) == 7
    assert torch.equal(gm.k_pool[:, bt_np[1]], before)


@pytest.mark.parametrize("mode", MODES)
def test_device_error_on_bad_token_and_block(tiny, mode):
    ql = lib()
    gm, _ = tiny
    set_mode(gm, mode)
    tokens = dev(np.array([CFG.vocab + 5], np.int32))
    positions = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = dev(np.array([[0, 1, 2, 3]], np.int32))
    args = gm.step_args(tokens, positions, bt, torch.zeros(1, dtype=torch.int32, device="cuda"))
    gm.ql_decode_step(args)
    with pytest.raises(ql.QLError) as e:
        gm.ql_check_device_error()
    assert e.value.status == ql.QL_EDEVICE and "vocabulary" in str(e.value)
    gm.ql_check_device_error()          # the record is cleared once read
    tokens.fill_(1)
    bad_bt = dev(np.array([[9999, 1, 2, 3]], np.int32))
    positions.fill_(0)
    args = gm.step_args(tokens, positions, bad_bt, torch.zeros(1, dtype=torch.int32, device="cuda"))
    gm.ql_decode_step(args)
    with pytest.raises(ql.QLError) as e:
        gm.ql_check_device_error()
    assert "block id" in str(e.value)


def test_replay_before_capture_is_an_error(tiny):
    ql = lib()
    gm, _ = tiny
    with pytest.raises(ql.QLError) as e:
        gm.ql_decode_graph_replay(7, 1)
    assert e.value.status == ql.QL_ESTATE


@pytest.mark.parametrize("B,form", [(2, "mma_sync"), (3, "mma_sync"), (3, "tcgen05")])
def test_batched_slots_with_replacement(tiny, B, form):
    """Slots at different context lengths (pre-filled f16 contexts in fragmented blocks from
    the library's block allocator) decode together; after four steps slot 1 finishes, its
    blocks go back to the pool and it restarts on a fresh 7-position context in newly allocated
    blocks. Every step's logits of every slot match the oracle decoding each slot on its own
    (batch 3: with either tensor-core form of the batched GEMV)."""
    import quantized_transformer_decode_ql_gb300 as ql
    prev = ql.ql_set_batched_gemv_form(ql.QL_BATCHED_TCGEN05 if form == "tcgen05" else ql.QL_BATCHED_MMA_SYNC)
    try:
        _slots_with_replacement(tiny, B)
    finally:
        ql.ql_set_batched_gemv_form(prev)


def _slots_with_replacement(tiny, B):
    import quantized_transformer_decode_ql_gb300 as ql
    gm, om = tiny
    maxb = 4
    pool = ql.BlockPool(64)
    order = [pool.alloc() for _ in range(64)]
    pool.free(list(np.random.default_rng(3).permutation(order)))   # fragmented reuse order
    lens = [5, 20, 33][:B]
    cache = decode.KVCache(CFG, B, maxb * 16)
    bt = np.full((B, maxb), 0, np.int32)
    blocks = [None] * B

    def place(slot, n_pos, seed):
        ids = [pool.alloc() for _ in range(maxb)]
        blocks[slot] = ids
        bt[slot] = ids
        k, v = ql_inputs.kv_context(CFG.n_layers, CFG.n_kv_heads, CFG.head_dim, n_pos, seed=seed)
        gm.write_context(ids, k, v)
        cache.k[slot] = 0.0
        cache.v[slot] = 0.0
        cache.preload(slot, k, v)

    for b in range(B):
        place(b, lens[b], seed=40 + b)
    tokens = dev(ql_inputs.prompt_tokens(B, CFG.vocab, seed=17).astype(np.int32))
    positions = dev(np.array(lens, np.int32))
    logits = torch.zeros((B, CFG.vocab), dtype=torch.float32, device="cuda")
    d_bt = dev(bt)
    args = gm.step_args(tokens, positions, d_bt, tokens, logits=logits)
    toks = tokens.cpu().numpy().copy()
    pos = np.array(lens)
    for step in range(8):
        if step == 4:
            pool.free(blocks[1])
            place(1, 7, seed=99)
            d_bt.copy_(torch.from_numpy(bt))
            pos[1] = 7
            positions.copy_(torch.from_numpy(pos.astype(np.int32)))
        want = decode.decode_step(om, cache, toks, pos)
        tokens.copy_(torch.from_numpy(toks.astype(np.int32)))
        gm.ql_decode_step(args)
        torch.cuda.synchronize()
        got = logits.cpu().numpy().astype(np.float64)
        for b in range(B):
            ok = decode.logits_close(got[b], want[b])
            assert ok.all(), f"step {step} slot {b}: max err {np.abs(got[b] - want[b]).max():.3e}"
        toks = decode.greedy(want)          # teacher forcing with the oracle's tokens
        pos = pos + 1
        assert positions.cpu().numpy().tolist() == pos.tolist()
    gm.ql_check_device_error()
    assert pool.in_use() == B * maxb   # slots 0 (and 2) plus the replacement of slot 1


def test_persistent_barrier_wait_is_bounded(tiny):
    """A grid barrier whose wait runs out (every barrier made to wait for one arrival that
    never comes, bound 1 ms) ends the step on every CTA without a fault: the device error says
    which barrier, the position does not advance, and the next step without the missing
    arrival is correct again."""
    ql = lib()
    gm, om = tiny
    set_mode(gm, "persistent")
    tok = int(ql_inputs.prompt_tokens(1, CFG.vocab, seed=11)[0])
    tokens = dev(np.array([tok], np.int32))
    positions = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    logits = torch.zeros((1, CFG.vocab), dtype=torch.float32, device="cuda")
    args = gm.step_args(tokens, positions, dev(slot_tables(1, 4, seed=51)), nxt, logits=logits)
    gm.ql_model_set_option(ql.QL_OPT_BARRIER_TIMEOUT_NS, 1_000_000)
    gm.ql_model_set_option(ql.QL_OPT_TEST_BARRIER_EXTRA, 1)
    gm.ql_decode_step(args)
    with pytest.raises(ql.QLError) as e:
        gm.ql_check_device_error()
    assert e.value.status == ql.QL_EDEVICE and "barrier" in str(e.value)
    assert int(positions.item()) == 0 and int(nxt.item()) == -5
    gm.ql_model_set_option(ql.QL_OPT_TEST_BARRIER_EXTRA, 0)
    gm.ql_model_set_option(ql.QL_OPT_BARRIER_TIMEOUT_NS, 2_000_000_000)
    for _ in range(2):   # the interrupted step left nothing behind (counters, tickets, keys)
        positions.fill_(0)
        gm.ql_decode_step(args)
        torch.cuda.synchronize()
        gm.ql_check_device_error()
        want = decode.decode_step(om, decode.KVCache(CFG, 1, 64), [tok], [0])[0]
        assert decode.logits_close(logits.cpu().numpy()[0].astype(np.float64), want).all()
        assert int(positions.item()) == 1


def test_persistent_rejects_larger_batches(tiny):
    ql = lib()
    gm, _ = tiny
    set_mode(gm, "persistent")
    B = 3
    tokens = torch.zeros(B, dtype=torch.int32, device="cuda")
    positions = torch.zeros(B, dtype=torch.int32, device="cuda")
    args = gm.step_args(tokens, positions, dev(slot_tables(B, 4, seed=61)), tokens)
    with pytest.raises(ql.QLError) as e:
        gm.ql_decode_step(args)
    assert e.value.status == ql.QL_EINVAL


@pytest.mark.parametrize("B", (1, 3))   # 1: stream GEMVs; 3: split-K GEMVs (+ merge kernels)
def test_launch_trace_stamps(tiny, B):
    """QL_OPT_STEP_TRACE on the one-launch-per-phase step: every GEMV launch row has its CTAs'
    stamps in order (start <= past the wait <= staged <= units done <= end), each GEMV starts
    no earlier than the previous one started, and each layer's attention row is stamped in
    order for the CTAs that took part. QL_OPT_MERGE_TRACE: at batch 3 every GEMV's merge row
    is stamped in order (start <= past the wait <= outputs written <= end), and no merge CTA
    passes its wait before the GEMV's last CTA has ended; at batch 1 (no merges) it stays
    untouched. Turning the options off leaves both buffers untouched."""
    ql = lib()
    gm, _ = tiny
    set_mode(gm, "launches")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = CFG.n_layers
    buf = torch.zeros((5 * L + 1) * sms * 8, dtype=torch.int64, device="cuda")
    mbuf = torch.zeros((4 * L + 1) * sms * 4, dtype=torch.int64, device="cuda")
    tokens = torch.zeros(B, dtype=torch.int32, device="cuda")
    positions = torch.full((B,), 3, dtype=torch.int32, device="cuda")
    bt = dev(slot_tables(B, 4, seed=11))
    args = gm.step_args(tokens, positions, bt, torch.zeros(B, dtype=torch.int32, device="cuda"))
    gm.ql_model_set_option(ql.QL_OPT_STEP_TRACE, buf.data_ptr())
    gm.ql_model_set_option(ql.QL_OPT_MERGE_TRACE, mbuf.data_ptr())
    try:
        gm.ql_decode_step(args)
        torch.cuda.synchronize()
    finally:
        gm.ql_model_set_option(ql.QL_OPT_STEP_TRACE, 0)
        gm.ql_model_set_option(ql.QL_OPT_MERGE_TRACE, 0)
    gm.ql_check_device_error()
    t = buf.cpu().numpy().reshape(5 * L + 1, sms, 8)
    starts = []
    for k in range(4 * L + 1):
        r = t[k][t[k][:, 0] > 0]
        assert len(r) > 0, f"GEMV launch {k} not stamped"
        for a, b in ((0, 1), (1, 2), (2, 3), (3, 5)):
            assert (r[:, a] <= r[:, b]).all(), f"GEMV launch {k}: stamp {a} after {b}"
        starts.append(r[:, 0].min())
    assert all(a <= b for a, b in zip(starts, starts[1:]))
    for l in range(L):
        r = t[4 * L + 1 + l]
        r = r[r[:, 5] > 0]
        assert len(r) > 0, f"attention of layer {l} not stamped"
        for a, b in ((0, 1), (1, 2), (2, 3), (3, 4), (4, 5)):
            assert (r[:, a] <= r[:, b]).all()
    m = mbuf.cpu().numpy().reshape(4 * L + 1, sms, 4)
    if B <= 2:
        assert not m.any(), "the batch 1-2 step has no merge launches"
    else:
        for k in range(4 * L + 1):
            r = m[k][m[k][:, 0] > 0]
            assert len(r) == sms, f"merge of GEMV launch {k}: {len(r)} CTAs stamped"
            for a, b in ((0, 1), (1, 2), (2, 3)):
                assert (r[:, a] <= r[:, b]).all(), f"merge {k}: stamp {a} after {b}"
            g_end = t[k][t[k][:, 0] > 0][:, 5].max()
            assert r[:, 1].min() >= g_end, f"merge {k} passed its wait before GEMV {k} ended"
    before, mbefore = buf.clone(), mbuf.clone()
    gm.ql_decode_step(args)
    torch.cuda.synchronize()
    assert torch.equal(buf, before) and torch.equal(mbuf, mbefore)
