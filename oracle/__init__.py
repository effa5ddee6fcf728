"""Reference oracle for one continuous-batching decode step over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 CPU
restatement of what the decode step computes.  Only the test suite, the smoke
check in ``__graft_entry__`` and the CPU legs of ``bench.py`` (``cpu_baseline``
and ``--impl reference``) may import it.  The product path (the CUDA library
and its Python binding) never imports, links or executes anything in here, and
this package imports nothing from the product: the two share no code, tables or
constants.

Sources (the three web pages the method is taken from):

* "feat(neuron): continuous batching -- batched decode + engine" (helexa issue
  121), slice 1: per-row RoPE positions gathered per batch row and applied with
  the rotate-half convention; keys stored after RoPE; the additive (B,1,1,S)
  decode mask over each row's padding gap.
* "neurogrid releases", v0.7.0 "Paged KV Cache": fixed 16-token blocks, an O(1)
  block allocator with per-sequence block tables, an attention kernel that reads
  K/V through block-table indirection with GQA; v0.8.0: ``kv_len = position + 1``.
* "cortex-engine writeup", section on the block-sparse cross-attention kernel:
  the guard that makes a row with zero normaliser emit zeros rather than NaN.

Modules
-------
``numerics``   rounding of float64 values onto the float32 / bfloat16 grids.
``rope``       rotate-half rotary embedding at an arbitrary position.
``attention``  exact softmax attention of one decode row, gathered through a
               block table (parity pinned by the tests in
               ``tests/test_oracle_pins.py``).
``allocator``  model of the host block allocator (LIFO free stack).
``step``       one whole decode step (RoPE, slot append, attention) and the
               joiners' prefix write (RoPE of each prefix key, slot write).
``dense``      the right-padded dense batch: assemble, extract a row, gap mask.

Every function is pinned by tests in ``tests/test_oracle_pins.py`` against
closed forms, hand-worked values, library routines or brute force.
"""
