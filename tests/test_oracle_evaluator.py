"""Pins for the oracle's evaluator, forced tokeniser and host rules.

* 17 * 23 + 91 = 482 (labs.miniml.ai "Evaluator aware decoding", "The core idea");
* integer expressions against Python's own evaluator;
* expressions with division against Python's parser over exact Fraction literals;
* greedy tokenisation against a brute-force longest-prefix check;
* an end-to-end evaluator-aware generation driven through the host rules.
"""

import random
import re

import numpy as np
import pytest

from oracle.driver import OracleRun, Row
from oracle.evaluator import EvalError, evaluate, format_result, tokenize_greedy
from oracle.step import FLAG_DONE
from tests.oracle_cache import oracle_dfa
from workloads import GRAMMARS


def test_page_example():
    assert evaluate(b"17 * 23 + 91") == 482
    assert format_result(b"17 * 23 + 91", "calc_tag") == b"<result>482</result>"
    assert format_result(b"17 * 23 + 91", "json_answer") == b', "answer": 482}'


def _rand_expr(rng, depth=3, div=False):
    if depth == 0 or rng.random() < 0.3:
        return str(rng.randint(0, 999))
    ops = "+-*/" if div else "+-*"
    a = _rand_expr(rng, depth - 1, div)
    b = _rand_expr(rng, depth - 1, div)
    if rng.random() < 0.3:
        return f"({a} {rng.choice(ops)} {b})"
    return f"{a} {rng.choice(ops)} {b}"


def test_integer_expressions_against_python():
    rng = random.Random(11)
    for _ in range(2000):
        e = _rand_expr(rng)
        assert evaluate(e.encode()) == eval(e)


def test_division_against_python_fractions():
    """Python's own expression parser over exact Fraction literals."""
    from fractions import Fraction  # noqa: F401  (used by eval below)
    rng = random.Random(12)
    for _ in range(2000):
        e = _rand_expr(rng, div=True)
        exact = re.sub(r"(\d+)", r"Fraction(\1)", e)
        try:
            ref = eval(exact)
        except ZeroDivisionError:
            with pytest.raises(EvalError) as ex:
                evaluate(e.encode())
            assert ex.value.code == "div_zero"
            continue
        if ref.denominator == 1:
            assert evaluate(e.encode()) == ref
        else:
            with pytest.raises(EvalError) as ex:
                evaluate(e.encode())
            assert ex.value.code == "non_integer"


@pytest.mark.parametrize("span,out", [
    (b"8 - 2 - 1", 5), (b"2 * 3 + 4", 10), (b"2 + 3 * 4", 14), (b"-(3)", -3), (b"--2", 2),
    (b"1.5 * 2", 3), (b".5 * 4", 2), (b"7. * 2", 14), (b"(((1)))", 1), (b"12 / 4 / 3", 1),
])
def test_precedence_and_lexemes(span, out):
    assert evaluate(span) == out


@pytest.mark.parametrize("span,code", [
    (b"1 / 0", "div_zero"), (b"1 +", "parse"), (b"", "parse"), (b"7 / 2", "non_integer"),
    (b"(1", "parse"), (b"1)", "parse"), (b".", "parse"), (b"1 2", "parse"),
    (b"9" * 33 + b" * " + b"9" * 33, "overflow"),
])
def test_error_codes(span, code):
    with pytest.raises(EvalError) as e:
        evaluate(span)
    assert e.value.code == code


def test_greedy_tokeniser_is_longest_prefix():
    rng = random.Random(13)
    toks = [bytes([b]) for b in range(256)] + [b"<re", b"<result>", b"sult", b"</", b"</result>", b"48", b"482"]
    for _ in range(200):
        text = bytes(rng.choice(b"<>/resultab48 2") for _ in range(rng.randint(0, 30)))
        out = tokenize_greedy(text, toks)
        assert b"".join(toks[t] for t in out) == text
        i = 0
        for t in out:
            longest = max(len(c) for c in toks if text.startswith(c, i))
            assert len(toks[t]) == longest
            i += len(toks[t])


def test_evaluator_aware_generation_end_to_end():
    spec = GRAMMARS["calc_eval"]
    dfa = oracle_dfa("calc_eval")
    toks = [bytes([b]) for b in range(256)] + [b"<result>", b"</result>"]
    run = OracleRun([dfa], [spec], toks, max_tokens=2048)
    row = Row(0, 0)
    target = b"The expression is <calc>17 * 23 + 91</calc>"
    tail = b", ok."
    produced = b""
    step = 0
    script = list(target)
    while step < 200:
        x = np.zeros(len(toks))
        if script:
            x[script[0]] = 10.0
        elif row.queue:
            pass                               # the forced token wins whatever the logits
        else:
            x[tail[len(produced) - len(target) - len(b"<result>482</result>")]] = 10.0
        rec = run.step_row(row, x, 0.0, 1.0, 0, step)
        if rec["forced"] < 0 and script:
            script.pop(0)
        produced += toks[rec["tok"]]
        step += 1
        if rec["flags"] & FLAG_DONE:
            break
    assert produced == target + b"<result>482</result>" + tail
    assert row.state == 0 and row.text == b"" and not row.queue
