"""Pins for the oracle's speculative draft verification (``accept_many``).

* The worked example of labs.miniml.ai "Evaluator aware decoding" ("The core
  idea"; "Where XGrammar-2 could take this"): a draft that writes
  ``<calc>17 * 23 + 91</calc>`` is accepted up to the closing tag and stops
  there (the result needs the evaluator); once the host pins the positions of
  ``<result>482</result>``, verifying them is exact matching against those ids:
  the right result passes, a wrong digit cuts the draft at that position.
* Against the mask by its definition: a step-by-step loop over the vectorised
  token mask (``token_mask``, pinned by brute force against the direct matcher
  in test_oracle_step) must accept the same prefix, from random states with
  random drafts mixing allowed and refused tokens.
* Counts and caps reset rows as ``accept`` does.
"""

import numpy as np

from oracle.dfa import DEAD
from oracle.evaluator import format_result, tokenize_greedy
from oracle.step import (FLAG_CAPPED, FLAG_DONE, FLAG_DRAFT_CUT, FLAG_FORCED_NEXT, FLAG_NO_TOKEN,
                         FLAG_REJECTED, VocabMatrix, accept, accept_many, token_mask)
from tests.oracle_cache import oracle_dfa, vocab


def _calc_setup():
    dfa = oracle_dfa("calc_eval")
    toks = [bytes([b]) for b in range(256)] + [b"<calc>", b"</calc>", b"<result>", b"</result>", b"17", b"482"]
    ids = {t: i for i, t in enumerate(toks)}
    return dfa, toks, ids


def _start_of_span(dfa, toks):
    """The state after the model has written the text before the span."""
    s = 0
    for b in b"The expression is ":
        s, _ = accept(dfa, s, b, toks, False)
        assert s != DEAD
    return s


def test_page_example_stops_where_the_evaluator_is_needed():
    dfa, toks, ids = _calc_setup()
    s0 = _start_of_span(dfa, toks)
    draft = [ids[b"<calc>"], ids[b"17"]] + list(b" * 23 + 91") + [ids[b"</calc>"], ids[b"<result>"]]
    r = accept_many(dfa, s0, draft, toks)
    assert r.n == len(draft) - 1                    # everything up to and including </calc>
    assert r.flags == FLAG_FORCED_NEXT              # the result span is the host's
    assert len(r.path) == r.n + 1 and r.path[0] == s0 and r.path[-1] == r.state


def test_page_example_pinned_result_is_exact_matching():
    dfa, toks, ids = _calc_setup()
    s0 = _start_of_span(dfa, toks)
    head = [ids[b"<calc>"], ids[b"17"]] + list(b" * 23 + 91") + [ids[b"</calc>"]]
    result = tokenize_greedy(format_result(b"17 * 23 + 91", "calc_tag"), toks)
    assert b"".join(toks[t] for t in result) == b"<result>482</result>"
    forced = [-1] * len(head) + result
    # the draft proposes exactly the pinned result: all accepted, then the tail continues
    r = accept_many(dfa, s0, head + result + list(b", ok"), toks, forced + [-1] * 4)
    assert r.n == len(head) + len(result) + 4 and not (r.flags & FLAG_DRAFT_CUT)
    # a wrong digit is cut at that position, whatever the grammar would allow there
    wrong = list(result)
    k = next(i for i, t in enumerate(wrong) if toks[t] == b"482")
    wrong[k] = ids[b"17"]
    r = accept_many(dfa, s0, head + wrong, toks, forced)
    assert r.n == len(head) + k and r.flags & FLAG_DRAFT_CUT
    assert r.state == r.path[-1]


def test_empty_draft_and_dead_row():
    dfa, toks, ids = _calc_setup()
    assert accept_many(dfa, 0, [], toks).flags == FLAG_NO_TOKEN
    r = accept_many(dfa, DEAD, [ids[b"17"]], toks)
    assert r.n == 0 and r.flags == FLAG_REJECTED and r.state == DEAD


def _loop_over_masks(dfa, vm, toks, s, draft):
    """Accepted prefix by the mask's definition, one position at a time, and
    whether it ended on a refused token."""
    n = 0
    for t in draft:
        if not token_mask(dfa, vm, s)[t]:
            return n, s, True
        s, fl = accept(dfa, s, t, toks, False)
        n += 1
        if fl & (FLAG_DONE | FLAG_FORCED_NEXT):
            break
    return n, s, False


def test_prefix_matches_the_mask_definition():
    rng = np.random.default_rng(3)
    for name, kind, V in (("calc_call", "tiny", 512), ("booking_200", "bpe", 2000)):
        dfa = oracle_dfa(name)
        toks = vocab(kind, V)
        vm = VocabMatrix(toks)
        live = np.flatnonzero(dfa.next.max(axis=1) >= 0)
        for _ in range(60):
            s = int(live[rng.integers(len(live))])
            draft, st = [], s
            for _ in range(int(rng.integers(1, 9))):
                m = token_mask(dfa, vm, st) if st >= 0 else np.zeros(V, bool)
                allowed = np.flatnonzero(m)
                if allowed.size and rng.random() < 0.85:
                    t = int(rng.choice(allowed))
                    st, _ = accept(dfa, st, t, toks, False)
                else:
                    t = int(rng.integers(V))
                draft.append(t)
            want_n, want_s, refused = _loop_over_masks(dfa, vm, toks, s, draft)
            r = accept_many(dfa, s, draft, toks)
            assert r.n == want_n, (name, s, draft)
            if not (r.flags & FLAG_DONE):
                assert r.state == want_s
            assert bool(r.flags & FLAG_DRAFT_CUT) == refused


def test_counts_and_cap():
    dfa, toks, ids = _calc_setup()
    s0 = _start_of_span(dfa, toks)
    draft = [ids[b"<calc>"], ids[b"17"]] + list(b" * 2")
    r = accept_many(dfa, s0, draft, toks, count=10, max_tokens=13)
    assert r.n == 3 and r.flags & FLAG_CAPPED and r.state == 0 and r.count == 0
    r = accept_many(dfa, s0, draft, toks, count=10, max_tokens=100)
    assert r.n == len(draft) and r.count == 10 + len(draft) and not (r.flags & FLAG_CAPPED)
