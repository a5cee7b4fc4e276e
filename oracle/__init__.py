"""CPU oracle for prefix-tree packing and tree attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call,
link or execute anything under ``oracle/``; only ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.  It shares no code with the CUDA path.

It is a plain, slow restatement of the method as the prefix-tree-packing
pages describe it:

* ``oracle.pack``  -- the trie walk, tree-aware best-fit-decreasing placement
  (plus the in-order and per-group-tree placements used for comparison),
  and the materialization of packed rows.
* ``oracle.attn``  -- ancestor sets taken from parent pointers, the tile
  classes by brute force, and explicit ancestor-masked softmax attention
  with its analytic backward, in float64.
* ``oracle.index`` -- the tree-aware top-k indexer: scores over a query's
  ancestor candidates only, top k with ties to the smaller key index.
* ``oracle.logprob`` -- next-token log-probabilities read off packed rows
  where loss_mask is set, and the same quantity on unpacked sequences.
* ``oracle.gdn``   -- the Gated DeltaNet layer core (short convolution along
  each token's path, normalized heads, the gated delta rule) threaded over
  the packed tree token by token, and the same layer on one sequence.

Pins (in ``tests/test_oracle_*.py``) tie every function here to something
other than itself: the worked examples the pages print, closed forms,
brute force on tiny inputs, a library causal attention, and finite
differences.
"""
