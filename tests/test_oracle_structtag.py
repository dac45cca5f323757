"""Pins for the oracle's structural-tag front-end (oracle.grammar.structtag_to_tree).

* The page's evaluated tag (labs.miniml.ai "Evaluator aware decoding", "Where
  XGrammar-2 could take this": begin "<calc>", regex content
  "[0-9+\\-*/(). ]+", end "</calc>", evaluator "arithmetic", result tags
  <result>...</result>) in the calc_eval framing compiles to exactly the
  minimal automaton of a hand-written GBNF for the same language (the GBNF
  front-end is pinned in test_oracle_grammar).
* The regex subset agrees with Python's ``re.fullmatch`` on every string up to
  a few bytes over a small alphabet, for patterns exercising each construct.
* The page's example walks through with the result injected, a model-written
  result is refused, a nested JSON-schema element behaves as that schema, and
  unsupported input fails closed.
"""

import itertools
import json
import re

import numpy as np
import pytest

from oracle.dfa import DEAD, build_dfa, compile_grammar, walk
from oracle.grammar import GrammarError, regex_to_tree
from tests.oracle_cache import oracle_dfa
from workloads import GRAMMARS, Bounds

_EQUIV_GBNF = r'''
root ::= "The expression is <calc>" content "</calc>" @forced( result ) tail
content ::= [0-9+\-*/(). ]+ & [\x00-\xff]{0,48}
result ::= "<result>" "-"? [0-9]{1,64} "</result>" | "<result_error>" [a-z_]{1,32} "</result_error>"
tail ::= [a-z ,]{0,24} "." & [\x00-\xff]{0,48}
'''


def test_page_evaluated_tag_equals_the_gbnf_automaton():
    st = oracle_dfa("calc_structtag")
    g = compile_grammar("gbnf", _EQUIV_GBNF, Bounds(max_len_default=48))
    assert st.n_states == g.n_states
    assert np.array_equal(st.next, g.next) and np.array_equal(st.accept, g.accept)


def test_page_example_walks_with_the_injected_result():
    d = oracle_dfa("calc_structtag")
    s = walk(d, 0, list(b"The expression is <calc>17 * 23 + 91</calc>"))
    assert s != DEAD and d.forced_only()[s]
    assert walk(d, s, list(b"<result>482</result>")) == DEAD           # the model may not write it
    s2 = walk(d, s, [b + 256 for b in b"<result>482</result>"])
    assert s2 != DEAD and walk(d, s2, list(b"ok.")) != DEAD
    assert walk(d, 0, list(b"The expression is <calc>17 x 23</calc>")) == DEAD


_PATTERNS = [
    "ab|c", "a*b+", "(ab)?c{2}", "[a-c]{1,3}", "[^ab]x", "a.c", r"\d+", r"[\-a]b", r"\.\*", "(a|bc)*",
    r"\w\s", "a{2,}", "[b-c]*a?", r"(\(|\))+", "x(y|)z",
]
_ALPHABET = b"abcx.*()-1 \n"


@pytest.mark.parametrize("pattern", _PATTERNS)
def test_regex_subset_agrees_with_re(pattern):
    dfa = build_dfa(regex_to_tree(pattern))
    rx = re.compile(pattern.encode())
    for n in range(0, 5):
        for t in itertools.product(_ALPHABET, repeat=n):
            s = bytes(t)
            st = walk(dfa, 0, list(s))
            ours = st != DEAD and bool(dfa.accept[st])
            assert ours == (rx.fullmatch(s) is not None), (pattern, s)


def test_nested_json_schema_element():
    schema = {"type": "object", "properties": {"n": {"type": "integer"}}, "required": ["n"]}
    src = json.dumps({"type": "sequence", "elements": [{"type": "literal", "text": "A:"},
                                                       {"type": "json_schema", "json_schema": schema}]})
    d = compile_grammar("structtag", src, Bounds())
    ok = walk(d, 0, list(b'A:{"n":-12}'))
    assert ok != DEAD and d.accept[ok]
    assert walk(d, 0, list(b'A:{"n":012}')) == DEAD
    assert walk(d, 0, list(b'{"n":1}')) == DEAD


@pytest.mark.parametrize("doc", [
    {"type": "bogus"},
    {"type": "literal", "text": "a", "extra": 1},
    {"type": "or", "elements": []},
    {"type": "regex", "pattern": "^a$"},
    {"type": "regex", "pattern": "(?:a)"},
    {"type": "regex", "pattern": "a)"},
    {"type": "evaluated_tag", "begin": "<c>", "content": {"type": "literal", "text": "1"}, "end": "</c>",
     "evaluator": "arithmetic", "result": {"begin": "<r>", "end": "</r>"}},
    {"type": "evaluated_tag", "begin": "<c>", "content": {"type": "literal", "text": "1"}, "end": "</c>",
     "evaluator": "python", "result": {"begin": "<result>", "end": "</result>"}},
])
def test_fails_closed(doc):
    with pytest.raises(GrammarError):
        compile_grammar("structtag", json.dumps(doc), Bounds())
    with pytest.raises(GrammarError):
        compile_grammar("structtag", "{not json", Bounds())


def test_workload_spec_is_registered():
    assert GRAMMARS["calc_structtag"].kind == "structtag"
