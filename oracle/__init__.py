"""CPU oracle for the batched speculative-decoding draft-verify step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code, tables or helpers with the CUDA library; the only thing
both sides consume is the seeded input generator in
``speculative_decoding_verification_73_gb300.workloads``.

What it computes (plain float64, in the order the pages state it):

* ``philox``  -- Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
  Random Numbers: As Easy as 1, 2, 3", SC'11) and the uniform draw that
  the walk consumes.
* ``verify``  -- temperature softmax of each logit row, the Leviathan
  accept rule min(1, q/p), the residual (q-p)_+ / ||(q-p)_+||_1, the
  left-to-right chain with a correction at the first rejection or a bonus
  token from q_{N+1}, the greedy argmax-match path at temperature 0, and
  the committed KV length ("Speculative Decoding and EAGLE-3" lesson,
  sections "Invariant: Leviathan rejection sampling", "Build it" steps
  1-4 and "KV cache rollback").
* ``tree``    -- verification of a draft tree (EAGLE-2's dynamic draft tree
  in the same lesson's "Key terms", its tree-mask remark and exercise 3):
  the per-node Leviathan test of each child in turn against the residual
  left by its rejected elder siblings, descent on acceptance, a drawn
  token where every child is rejected or at a leaf, and the argmax path at
  temperature 0.
* ``fcnorm``  -- the drafter's input fusion of EAGLE-3 / EAGLE 3.1: the
  three target hidden states, each LayerNorm- or RMSNorm-normalised (or
  not), concatenated and projected by one FC layer.
* ``kv``      -- the KV-cache commit driven by out_kv_len (and a tree's
  out_path): copy the kept window entries from a scratch buffer, or move
  them together in place, and advance the logical length (section "KV
  cache rollback" and exercise 4).

Pins (see tests/test_oracle_*.py): exact Fraction enumeration of the
output law on tiny vocabularies, the acceptance identity sum_t min(p, q),
the E[accepted] closed form, brute-force greedy chains, textbook softmax
special cases, Philox known-answer vectors and a library Philox.
"""

from . import fcnorm, kv, philox, tree, verify  # noqa: F401
