"""Pins for the oracle's string-operation evaluator (oracle.strops).

* The page's example (labs.miniml.ai "Evaluator aware decoding", "Not just
  arithmetic: string operations"): count("strawberry", "r") is 3 and the host
  forces <result>3</result>.
* Every operation against Python's own bytes methods and slicing on random
  strings (the oracle computes them with plain loops).
* The error codes of the reading, case by case.
* The strop grammar accepts the page-shaped text, refuses a result the model
  writes itself, and an evaluator-aware generation driven through the oracle's
  host rules produces the evaluated result.
"""

import random

import numpy as np
import pytest

from oracle.driver import OracleRun, Row
from oracle.evaluator import EvalError, format_result
from oracle.step import FLAG_DONE, accept
from oracle.strops import evaluate_strop
from tests.oracle_cache import oracle_dfa
from workloads import GRAMMARS


def test_page_example():
    assert evaluate_strop(b'count("strawberry", "r")') == b"3"
    assert format_result(b'count("strawberry", "r")', "strop_tag") == b"<result>3</result>"


def _quote(s: bytes) -> bytes:
    return b'"' + s.replace(b"\\", b"\\\\").replace(b'"', b'\\"') + b'"'


def _rand_bytes(rng, n):
    alphabet = b"abcrstwy RST.,!?'-\"\\0123456789"
    return bytes(rng.choice(alphabet) for _ in range(n))


def test_operations_against_python():
    rng = random.Random(5)
    for _ in range(3000):
        s = _rand_bytes(rng, rng.randint(0, 30))
        sub = _rand_bytes(rng, rng.randint(1, 3))
        i, j = rng.randint(-40, 40), rng.randint(-40, 40)
        assert evaluate_strop(b"count(" + _quote(s) + b", " + _quote(sub) + b")") == str(s.count(sub)).encode()
        assert evaluate_strop(b"len(" + _quote(s) + b")") == str(len(s)).encode()
        want = s[::-1]
        if b"<" not in want:
            assert evaluate_strop(b"reverse(" + _quote(s) + b")") == want
        assert evaluate_strop(b"upper(" + _quote(s) + b")") == s.upper()
        assert evaluate_strop(b"substr(" + _quote(s) + b", %d, %d)" % (i, j)) == s[i:j]


@pytest.mark.parametrize("span,code", [
    (b'count("abc")', "arity"), (b'len("a", "b")', "arity"), (b'substr("abc", "1", 2)', "arity"),
    (b'len(5)', "arity"), (b'count("abc", "")', "empty"), (b'lower("abc")', "unknown_op"),
    (b'len("abc"', "parse"), (b'len "abc")', "parse"), (b'len("abc") x', "parse"), (b'', "parse"),
    (b'len("a\\qb")', "parse"), (b'substr("a", 1234567890, 1)', "parse"), (b'Len("a")', "parse"),
    (b'upper("' + b"a" * 65 + b'")', "overflow"), (b'reverse("<a")', "bad_char"),
    (b'len("' + b"a" * 5000 + b'")', "overflow"),
])
def test_error_codes(span, code):
    with pytest.raises(EvalError) as e:
        evaluate_strop(span)
    assert e.value.code == code


def test_spaces_and_escapes():
    assert evaluate_strop(b'  len ( "a\\"b\\\\c" )  ') == b"5"
    assert evaluate_strop(b'substr("strawberry",-5,-1)') == b"berr"
    assert evaluate_strop(b'count("aaaa", "aa")') == b"2"          # non-overlapping


def _walk(dfa, s, data, injected=False):
    toks = [bytes([b]) for b in range(256)]
    for c in data:
        s, _ = accept(dfa, s, c, toks, injected)
        if s < 0:
            return s
    return s


def test_grammar_accepts_page_shape_and_refuses_model_written_result():
    dfa = oracle_dfa("strop_eval")
    s = _walk(dfa, 0, b'The answer is <strop>count("strawberry", "r")</strop>')
    assert s >= 0 and dfa.forced_only()[s]
    assert _walk(dfa, s, b"<result>3</result>") < 0                # the model may not write it
    s2 = _walk(dfa, s, b"<result>3</result>", injected=True)
    assert s2 >= 0 and _walk(dfa, s2, b"ok.") >= 0
    assert _walk(dfa, 0, b'The answer is <strop>count("straw"berry", "r")</strop>') < 0


def test_evaluator_aware_generation_end_to_end():
    spec = GRAMMARS["strop_eval"]
    dfa = oracle_dfa("strop_eval")
    toks = [bytes([b]) for b in range(256)] + [b"<result>", b"</result>", b"straw", b"berry"]
    run = OracleRun([dfa], [spec], toks, max_tokens=2048)
    row = Row(0, 0)
    target = b'The answer is <strop>count("strawberry", "r")</strop>'
    tail = b"ok."
    produced = b""
    script = list(target)
    for step in range(300):
        x = np.zeros(len(toks))
        if script:
            x[script[0]] = 10.0
        elif not row.queue:
            x[tail[len(produced) - len(target) - len(b"<result>3</result>")]] = 10.0
        rec = run.step_row(row, x, 0.0, 1.0, 0, step)
        if rec["forced"] < 0 and script:
            script.pop(0)
        produced += toks[rec["tok"]]
        if rec["flags"] & FLAG_DONE:
            break
    assert produced == target + b"<result>3</result>" + tail
