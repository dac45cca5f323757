"""Oracle of the pushdown-automaton path: recursive GBNF grammars under a stack
bound (test infrastructure: only tests, the smoke check and the benchmark's CPU
baseline use it).

usetacet.com/docs/grammar, "The guarantee": the automaton that masks the
logits at every step is a pushdown automaton.  The device keeps one stack per
row; its bound D is the number of frames of recursive rules open at once (a
frame opens at every reference to a rule that lies on a cycle of the
reference graph and closes when that rule's text ends).  The base frame, the
start rule, opens none.

The oracle runs no pushdown automaton.  With the stack bounded the language
is regular, so the oracle expands the rules with at most D frames open
(``gbnf_to_tree(..., nesting='stack')``) and builds the minimal trimmed DFA of
oracle.dfa.  Masks, accept flags and draft checks are then oracle.step's on
that DFA: a device configuration (state, stack) corresponds to the DFA state
that the same token sequence reaches from the start.

Parity of this definition is pinned in tests/test_oracle_pda.py against the
bounded-height Dyck counts (a closed recurrence), Python's json module on a
JSON grammar with its frame count written out per value, and the per-rule
bound for grammars with one recursive rule.
"""

from __future__ import annotations

from .dfa import OracleDFA, build_dfa
from .grammar import gbnf_rules, gbnf_to_tree, recursive_rules


def compile_pda(source: str, depth: int) -> OracleDFA:
    """The DFA of ``source``'s language with at most ``depth`` frames open."""
    return build_dfa(gbnf_to_tree(source, depth, nesting='stack'))


def frame_rules(source: str) -> set:
    """The rules whose references open a frame (the recursive ones)."""
    return recursive_rules(gbnf_rules(source))
