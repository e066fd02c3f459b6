"""CPU oracle for the CSA / HCA attention hot path (DeepSeek-V4 report, §2.3).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, call or
execute anything in this package.  The CUDA product path never routes through
it, and it shares no code, header, table or helper with the CUDA sources.

Everything here is a plain, slow restatement of what the method computes, in
float64 unless the step itself fixes a narrower precision (the canonical
float32 index score, the storage codecs).  Each function cites the passage of
the pages it follows, by page title and section.

Parity status per function (what pins it is in ``tests/test_oracle.py``):

* ``codecs``: pinned (exhaustive code tables, RNE ties, saturation, and an
  independent library conversion where one exists).
* ``csa.compress``: pinned (identical tokens, equal logits -> mean, m = 1
  identity, weights sum to one).
* ``csa.index_scores`` / ``canon.index_scores_f32``: pinned (brute-force
  float64, one-hot head weights, a few-ulp bound between the two).
* ``csa.topk``: pinned (stable sort on the total order, k >= candidates,
  causality).
* ``csa.attend``: pinned (textbook causal MQA on tiny inputs, CSA with
  k >= blocks equals the dense HCA-style path, single visible entry,
  weights sum to one).
* ``decode.decode_step``: pinned (``tests/test_oracle_decode.py``): one
  step driven by the state cache equals the whole-sequence definitions above
  at t = L (block completion, window and tail slots, the new indexer key, BF16
  and FP4 keys, m = 4 and 128, L < W, L = 0), and planted mistakes in its
  bookkeeping fail those checks.
* Absolute model outputs of the pages: parity unpinned (no trained weights
  exist; inputs are synthetic).
"""
