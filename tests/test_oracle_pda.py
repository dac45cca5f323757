"""Pins for the oracle of the pushdown path (oracle/pda.py): the language of a
recursive GBNF grammar with at most D frames of recursive rules open.

* bounded-height Dyck words: the number of accepted strings of each length
  equals the count of Dyck paths of height <= D (a recurrence over
  (length, height) written out here), D = 1..6, lengths up to 20;
* JSON: for random values the oracle accepts the canonical text iff the
  value's frame count (value 1, array +1, object +2 for object and member,
  written out per value below) is at most D; mutated texts the oracle accepts
  parse with Python's json module within the bound, and mutated texts that
  parse, are canonical and fit the bound are accepted;
* one recursive rule: the stack bound equals the per-rule bound of the
  flattened grammars (D for a recursive non-start rule, D + 1 when the start
  rule itself recurses) -- identical canonical tables;
* the recursive-rule sets of small grammars.
"""

import json
import random

import numpy as np
import pytest

from oracle.dfa import DEAD, build_dfa, walk
from oracle.grammar import gbnf_rules, gbnf_to_tree, recursive_rules
from oracle.pda import compile_pda, frame_rules
from workloads.grammars import JSON_NESTED

DYCK = r'''
root ::= pair*
pair ::= "(" pair* ")"
'''


def _count_by_length(dfa, n_max):
    """Accepted strings of each length 0..n_max, by stepping a vector of path
    counts through the transition table (any symbol with a transition)."""
    S = dfa.n_states
    v = np.zeros(S, dtype=object)
    v[0] = 1
    out = []
    for n in range(n_max + 1):
        out.append(int(sum(v[s] for s in range(S) if dfa.accept[s])))
        w = np.zeros(S, dtype=object)
        for s in range(S):
            if v[s]:
                for t in dfa.next[s]:
                    if t >= 0:
                        w[int(t)] += v[s]
        v = w
    return out


def _dyck_counts(n_max, h):
    """Dyck words of each length 0..n_max whose height never exceeds h:
    paths of +1/-1 steps from 0 back to 0 staying within [0, h]."""
    out = []
    for n in range(n_max + 1):
        ways = [1] + [0] * h
        for _ in range(n):
            nw = [0] * (h + 1)
            for y, c in enumerate(ways):
                if c:
                    if y + 1 <= h:
                        nw[y + 1] += c
                    if y - 1 >= 0:
                        nw[y - 1] += c
            ways = nw
        out.append(ways[0])
    return out


@pytest.mark.parametrize("D", [1, 2, 3, 4, 5, 6])
def test_dyck_counts_match_bounded_height_paths(D):
    dfa = compile_pda(DYCK, D)
    assert _count_by_length(dfa, 20) == _dyck_counts(20, D)


def test_dyck_depth_zero_is_the_empty_word_only():
    dfa = compile_pda(DYCK, 0)
    assert dfa.accept[0] and (dfa.next[0] < 0).all()


# ---------------------------------------------------------------------- JSON
_CHARS = " !#$%&'()*+,-./0123456789:;<=>?@ABCXYZ[]^_`abcxyz{|}~"


def _rand_value(rng, depth):
    k = rng.random()
    if depth == 0 or k < 0.35:
        c = rng.randrange(6)
        if c == 0:
            return rng.randrange(-10**6, 10**6)
        if c == 1:
            return "".join(rng.choice(_CHARS) for _ in range(rng.randrange(0, 6)))
        return [True, False, None, 0][c - 2]
    if k < 0.65:
        return [_rand_value(rng, depth - 1) for _ in range(rng.randrange(0, 4))]
    keys = rng.sample(["a", "b", "k y", "z!", "[x]", ""], rng.randrange(0, 4))
    return {key: _rand_value(rng, depth - 1) for key in keys}


def _frames(v):
    """Frames open at once while the JSON grammar derives v as a value: the
    value frame, then +1 for an array, +2 for an object (object and member)
    around the deepest child."""
    if isinstance(v, list):
        return 2 + max((_frames(x) for x in v), default=0)
    if isinstance(v, dict):
        return 2 + max((1 + _frames(x) for x in v.values()), default=0)
    return 1


def _canonical(v) -> bytes:
    return json.dumps(v, separators=(",", ":"), ensure_ascii=True).encode()


def _accepts(dfa, data: bytes) -> bool:
    s = walk(dfa, 0, list(data))
    return s != DEAD and bool(dfa.accept[s])


def _parse(data: bytes):
    """(True, value) when Python's json module parses data, else (False, None)."""
    try:
        return True, json.loads(data)
    except (ValueError, UnicodeDecodeError):
        return False, None


@pytest.mark.parametrize("D", [3, 5, 8])
def test_json_canonical_texts_accepted_iff_within_the_bound(D):
    dfa = compile_pda(JSON_NESTED, D)
    rng = random.Random(1000 + D)
    seen_in = seen_out = 0
    for _ in range(400):
        v = _rand_value(rng, 4)
        ok = _frames(v) <= D
        assert _accepts(dfa, _canonical(v)) == ok, (_canonical(v), _frames(v), D)
        seen_in += ok
        seen_out += not ok
    assert seen_in > 50 and seen_out > 50


@pytest.mark.parametrize("D", [4, 7])
def test_json_mutations_agree_with_the_json_module(D):
    dfa = compile_pda(JSON_NESTED, D)
    rng = random.Random(77 + D)
    alphabet = b'{}[]",:-0123456789tfnrulseax \\'
    n_acc = 0
    for _ in range(1500):
        data = bytearray(_canonical(_rand_value(rng, 3)))
        for _ in range(rng.randrange(1, 3)):
            op = rng.randrange(3) if data else 1
            if op == 1:
                data.insert(rng.randrange(len(data) + 1), rng.choice(alphabet))
            elif op == 0:
                data[rng.randrange(len(data))] = rng.choice(alphabet)
            else:
                del data[rng.randrange(len(data))]
        data = bytes(data)
        acc = _accepts(dfa, data)
        parsed, v = _parse(data)
        if acc:
            n_acc += 1
            assert parsed and _frames(v) <= D, data
        elif parsed and _canonical(v) == data and _frames(v) <= D:
            pytest.fail(f"valid canonical JSON refused: {data!r}")
    assert n_acc > 100


# ------------------------------------------------------- one recursive rule
def test_one_recursive_rule_matches_the_per_rule_bound():
    for D in range(1, 6):
        a = compile_pda(DYCK, D)
        b = build_dfa(gbnf_to_tree(DYCK, D))
        assert np.array_equal(a.next, b.next) and np.array_equal(a.accept, b.accept)
    rooted = r'''root ::= "(" root* ")" | "x"'''
    for D in range(0, 5):
        a = compile_pda(rooted, D)
        b = build_dfa(gbnf_to_tree(rooted, D + 1))
        assert np.array_equal(a.next, b.next) and np.array_equal(a.accept, b.accept)


def test_recursive_rule_sets():
    assert frame_rules(JSON_NESTED) == {"value", "object", "member", "array"}
    assert frame_rules(DYCK) == {"pair"}
    src = r'''
root ::= head body
head ::= "h" tail
tail ::= "t"?
body ::= "(" inner ")"
inner ::= body | "x"
'''
    assert recursive_rules(gbnf_rules(src)) == {"body", "inner"}
    assert recursive_rules(gbnf_rules(r'''root ::= "a" root | "b"''')) == {"root"}
