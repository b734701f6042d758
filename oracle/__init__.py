"""The oracle: a plain, slow, f64 CPU statement of what the decode hot path computes.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. The CUDA library never calls it and it never
calls the CUDA library; the two share no code. The only thing both consume is the seeded
input arrays of ``ql_inputs``.

Sources (public web pages; cited by page and item):

* inferencelayer ``cuda_llm.rs`` - the dense Qwen3 decode engine: ``Q4Dev`` (q4_0 matrix,
  32-weight blocks, one f16 scale, 16 bytes of nibbles), ``CudaQwen3::step`` (the decode
  dataflow), ``Cfg`` (qk_norm, rope_theta, eps), ``rope_inv_freq`` (theta^(-2i/hd)).
* ferrum-kernels ``cuda_decode.rs`` - ``attention_paged`` / ``paged_decode_attention``
  (16-token blocks, block table, valid length = current length + 1, scale 1/sqrt(hd)),
  ``alloc_block`` (free list then bump, "pool exhausted").
* memra-engine ``qwen4exp_gpu.rs`` - ``host_rms_norm`` and ``host_rope_at`` twins
  (RMSNorm with effective weights; NeoX split-half rotation); the quantised-cache storage
  (q8_0 key rows, q5_1 value rows) and its host twins ``host_quant_q8_row``,
  ``host_deq_q8_rows``, ``host_quant_q5_row``, ``host_deq_q5_rows``.

Modules: :mod:`oracle.q4_0` (codec), :mod:`oracle.ops` (per-op definitions),
:mod:`oracle.decode` (decode step, full recomputation, greedy decoding),
:mod:`oracle.blockpool` (the block allocator rule), :mod:`oracle.kvq` (the quantised KV-row
codecs and attention over a quantised pool).

Pins: every function here is pinned in ``tests/test_oracle_*.py`` against closed forms,
invariants, brute force on tiny inputs and hand-derived fixtures in ``tests/golden/``.
The absolute end-to-end logits of a random-init model have no printed value on the
pages; they are pinned only through the invariants (incremental decode equals full
recomputation; identical batch slots equal batch 1) and the per-op pins.
"""
