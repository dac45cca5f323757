"""Host rules around the step, and a multi-step oracle run (oracle side).

Per row, after each step's accept (the same order the product's driver uses):
  1. if the row's token was the forced one, it leaves the forced queue;
  2. a real token is appended to the row's text and counted;
  3. DONE, or ``max_tokens`` tokens without finishing (usetacet.com/docs/grammar,
     "A valid call also has to end": a 2048-token cap), resets the row: state
     <- start (0), empty text, empty queue, count 0;
  4. otherwise, FORCED_NEXT with an empty queue triggers the evaluator: the
     span is the text between the last ``span_open`` and the trailing
     ``span_close``; its result is formatted and tokenised greedily into the
     queue (labs.miniml.ai "Evaluator aware decoding", "The core idea",
     steps 1-4).
At the next step a row with a non-empty queue has its front as forced token.

Random start states: the row's draw r selects ``live[r mod len(live)]`` where
``live`` lists, in increasing id, the states that are neither finished
(accepting without successors) nor inside a forced region.
"""

from __future__ import annotations

import numpy as np

from .dfa import OracleDFA
from .evaluator import format_result, tokenize_greedy
from .step import (FLAG_DONE, FLAG_FORCED_NEXT, NO_TOKEN, VocabMatrix, accept,
                   onehot_mask, sample_row, token_mask)


def live_states(dfa: OracleDFA) -> np.ndarray:
    bad = dfa.sink() | dfa.forced_only()
    return np.flatnonzero(~bad)


class Row:
    def __init__(self, b: int, gid: int, state: int = 0):
        self.b = b
        self.gid = gid
        self.state = state
        self.text = b''
        self.queue: list[int] = []
        self.count = 0


class OracleRun:
    """Steps a set of rows through the oracle, each row on its own trajectory."""

    def __init__(self, dfas: list[OracleDFA], specs, tokens: list[bytes], max_tokens: int):
        self.dfas = dfas
        self.specs = specs
        self.tokens = tokens
        self.vm = VocabMatrix(tokens)
        self.max_tokens = max_tokens

    def step_row(self, row: Row, x: np.ndarray, temp: float, top_p: float, seed: int, step: int):
        """One step for one row; returns a record of what the step computed."""
        dfa = self.dfas[row.gid]
        V = self.vm.V
        forced = row.queue[0] if row.queue else -1
        state_in = row.state
        if forced >= 0:
            mask = onehot_mask(V, forced)
        else:
            mask = token_mask(dfa, self.vm, row.state)
        res = sample_row(x, mask, temp, top_p, seed, row.b, step)
        ns, flags = accept(dfa, row.state, res.tok, self.tokens, forced >= 0 and res.tok == forced)
        rec = dict(state_in=state_in, forced=forced, mask=mask, tok=res.tok, probs=res.probs,
                   gap=res.gap, margin=res.margin, state_out=ns, flags=flags,
                   nucleus=res.nucleus_size)
        # host rules
        if forced >= 0 and res.tok == forced:
            row.queue.pop(0)
        if res.tok != NO_TOKEN:
            row.text += self.tokens[res.tok]
            row.count += 1
        row.state = ns
        if (flags & FLAG_DONE) or row.count >= self.max_tokens:
            row.state = 0
            row.text = b''
            row.queue = []
            row.count = 0
        elif (flags & FLAG_FORCED_NEXT) and not row.queue:
            spec = self.specs[row.gid]
            text = row.text
            assert text.endswith(spec.span_close)
            end = len(text) - len(spec.span_close)
            start = text.rfind(spec.span_open, 0, end)
            span = text[start + len(spec.span_open):end] if start >= 0 else None
            row.queue = tokenize_greedy(format_result(span, spec.result_format), self.tokens)
        rec['state_after_host'] = row.state
        return rec
