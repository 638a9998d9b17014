"""CPU oracle for the ring-attention hot path.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import anything here.  The product path (the CUDA library and
its Python binding) never imports, calls or links this package, and this
package never imports the product.

Everything is plain numpy in float64 (the pages' own example is float64
numpy).  Each function names the passage it follows:

* :mod:`oracle.attention` -- full-row softmax attention, the result the ring
  method must reproduce exactly ("Interrogating parallelism, part 5", section
  "How does attention survive being split?": the merge is exact, not an
  approximation).
* :mod:`oracle.ring` -- the per-rank ring computation restated step by step:
  fixed queries, KV blocks visited hop by hop, running max / running sum /
  correction ("Ring Attention and Ulysses shard a sequence two different
  ways...", section "Ring Attention: point-to-point rotation, and an online
  softmax that never sees the whole row at once").
* :mod:`oracle.layout` -- contiguous and zigzag chunk assignment ("What breaks
  the load balance?": rank i holds chunks i and 2c-1-i).
* :mod:`oracle.merge` -- exact combination of two (output, log-sum-exp)
  partials over disjoint key sets.
* :mod:`oracle.work` -- per-rank causal work in chunk units, exact pairs and
  128x128 tiles.
* :mod:`oracle.docmask` -- attention over all-gathered keys and values under a
  document mask, causal inside each document ("Interrogating parallelism,
  part 5", section "Why did Llama 3 not use a ring?").
* :mod:`oracle.ulysses` -- Ulysses: the all-to-all from sequence shards to head
  shards and back, message by message, with full-sequence attention on each
  rank's heads in between ("Ring Attention and Ulysses shard a sequence two
  different ways...", section "Ulysses: an all-to-all relayout instead of a
  rotation").
* :mod:`oracle.backward` -- the exact gradient of that attention with respect
  to q, k and v, and the ring's backward (KV blocks travel with their dK, dV
  accumulators); the pages give only the forward, so the gradient is the
  definition.

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
brute force, library routines it does not call, or values the pages print.
"""
