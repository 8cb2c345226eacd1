"""CPU oracle of the CSA2 compressed-sparse-attention layer step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its CPU-baseline leg and ``--impl reference``) may import this
package.  The product path (``compressed_sparse_attention_05_gb300``) never
imports, calls or links anything here, and this package shares no code with
it: both sides only read the seeded inputs of ``csa2_inputs``.

Plain, slow, float64 numpy, one function per step of the method, each
citing the passage it follows:

  formats    E2M1 / E4M3 codes, MXFP4 (E4M3 scale per 16 channels) and the
             per-token FP8 window format, bf16 rounding
  compress   a1 4:1 linear compression, a2 RMSNorm + RoPE, a3 MXFP4 pack,
             a4 indexer-key projection
  indexer    a5 index scores, a6 Top-K, a7 block pool, a8 Reindex, a9 Reuse
  attention  a10/a11 sparse MQA attention over selected entries + window,
             and an independent dense masked form
  replay     SWA Bounded Replay: window rows rebuilt from the replayed
             tokens' hidden states, and the window cut at the replay start
  layer      the layer schedule (Full / Reindex / Reuse) for sampled tokens

Pins (tests/test_oracle_*.py, run with ``-m "not gpu"``) tie every function
to something other than itself: the constants the pages print
(tests/golden/page_constants.json), the published format definitions
(tests/golden/ocp_formats.json), library routines (torch float8 / bf16
casts, torch scaled_dot_product_attention, torch.topk on distinct values),
closed forms and invariants (norm of RMSNorm output, norm preservation and
relative-position property of RoPE, selection/averaging compression maps,
attention with one key or equal logits), brute force on tiny inputs (rank
counting for Top-K, walking entries for the pool) and planted mistakes that
the pins must catch.  No function is left without a pin.
"""
