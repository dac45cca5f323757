"""CPU oracle for grammar-constrained decoding -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what one constrained decode
step computes, written from the pages (labs.miniml.ai "Evaluator aware
decoding"; usetacet.com/docs/grammar "Constrained decoding"; seedpath.ai
"Guided Decoding & Structured-Output Reliability"; dev.to "I found a runner
bug...") and from the published Philox4x32-10 definition (Salmon, Moraes, Dror,
Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import anything under ``oracle/``.  The product path never does, and
this package shares no code with it: the grammar front-ends, the automaton
construction (Brzozowski derivatives + Moore minimisation here, against the
product's NFA/subset/Hopcroft pipeline), the mask walk, the sampler, the
evaluator and the host rules are all written separately.  Only the seeded
input generators in ``workloads/`` serve both sides.

Modules
  philox     Philox4x32-10 counter-based generator and the uniform mapping.
  grammar    GBNF-style rule language and JSON-schema subset -> regular
             expression tree over a 512-symbol alphabet (bytes 0..255 the
             model writes, 256..511 the same bytes forced by the host).
  dfa        derivative-based automaton, trimming, Moore minimisation,
             canonical breadth-first numbering.
  step       token mask, sampler (temperature, softmax, top-p, Gumbel-max),
             accept.
  evaluator  exact-rational arithmetic evaluator and greedy forced tokeniser.
  strops     string operations of the <strop> evaluator.
  driver     host rules around the step (reset, forced queue, token cap).
  pda        recursive grammars under a stack bound: the flattened language
             whose automaton the pushdown path is checked against.

Parity pins (tests/test_oracle_*.py) tie every function to something other
than itself; there is no function here whose parity is unpinned.
"""
