"""CPU oracle for trie-constrained label scoring -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct implementation of what the CUDA path
computes, in float64 (numpy), written from the method's description:
  * "To Classify, Try a Trie Tree" (Quail blog): sec. 3.1 trie_decode,
    sec. 3.2 trie_tree (score, normalisation, prefix labels, evaluated
    positions, tree attention), sec. 3.3 letters, sec. 4.1 output head.
  * Quail "Execution" docs, section "Label scoring" (worked 0.8 x 0.6 example).

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline leg may import
this package. It shares no code with the CUDA path (trie_label_scoring_gb300)
and never imports it; the only common module is `synthetic`, which draws
input data and holds none of the method's arithmetic.

Modules:
  oracle.trie     -- label trie, decision depth d_m, evaluated set P
  oracle.model    -- the layer at an answer position (RMSNorm, q/k/v, RoPE,
                     attention over [document ; path], W_o, final norm, head)
  oracle.scoring  -- trie_tree scores and probabilities, prefix-label
                     correction, letters, greedy trie_decode, flat scoring

Parity status of each function is stated in its docstring; every function is
pinned by tests/test_oracle_pins.py (closed forms, worked examples from the
pages, brute force, library special cases).
"""
