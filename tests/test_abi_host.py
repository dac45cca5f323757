"""CPU tests of libcg.so: exported symbols, the grammar compiler against the
oracle's automata, and the host-side evaluator/tokeniser/driver against the
oracle.  No device call is made here."""

import ctypes
import json
import os
import random
import re

import numpy as np
import pytest

from oracle.dfa import build_dfa
from oracle.driver import OracleRun, Row
from oracle.evaluator import format_result, tokenize_greedy
from oracle.grammar import GrammarError, gbnf_to_tree, schema_to_tree, source_to_tree
from oracle.step import FLAG_DONE, FLAG_FORCED_NEXT
from tests.oracle_cache import oracle_dfa, vocab
from tests.test_oracle_grammar import _gbnf, _lang, _rand_tree
from workloads import GRAMMARS, Bounds as WBounds

gcd = pytest.importorskip("grammar_constrained_decoding_gb300")
from grammar_constrained_decoding_gb300 import Bounds, Grammar, Vocab, Driver, eval_arith, eval_strop, _lib  # noqa: E402

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "cg.h")


def _bounds(b):
    return Bounds(b.ws_max, b.max_len_default, b.depth_max, b.max_items_default, b.max_tokens)


def test_library_exports_every_declared_symbol():
    text = open(HEADER).read()
    names = set(re.findall(r"^\s*(?:int|void)\s+(cg_\w+)\s*\(", text, flags=re.M))
    assert len(names) >= 20
    lib = ctypes.CDLL(_lib.LIB_PATH)
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names == set(_lib.SIGNATURES), names ^ set(_lib.SIGNATURES)


@pytest.mark.parametrize("name", sorted(GRAMMARS))
def test_compiler_matches_oracle_tables(name):
    spec = GRAMMARS[name]
    g = Grammar.compile(spec.source, spec.kind, _bounds(spec.bounds))
    nxt, flags = g.export()
    o = oracle_dfa(name)
    assert np.array_equal(nxt, o.next)
    assert np.array_equal((flags & _lib.CG_STATE_ACCEPT) != 0, o.accept)
    assert np.array_equal((flags & _lib.CG_STATE_SINK) != 0, o.sink())
    assert np.array_equal((flags & _lib.CG_STATE_FORCED_ONLY) != 0, o.forced_only())


def test_compiler_matches_oracle_on_random_grammars():
    rng = random.Random(99)
    done = 0
    while done < 150:
        t = _rand_tree(rng, 5)
        src = "root ::= " + _gbnf(t)
        try:
            o = build_dfa(gbnf_to_tree(src, 5))
        except GrammarError:
            with pytest.raises(_lib.CgError) as e:
                Grammar.compile(src, "gbnf")
            assert e.value.code == _lib.CG_E_EMPTY
            continue
        nxt, _ = Grammar.compile(src, "gbnf").export()
        assert np.array_equal(nxt, o.next), src
        done += 1


def _rand_regex(rng, depth):
    atoms = ["a", "b", "\\.", "[a-c]", "[^ab]", "\\d", ".", "x", "[\\-y]"]
    if depth == 0 or rng.random() < 0.35:
        return rng.choice(atoms)
    kind = rng.randrange(4)
    if kind == 0:
        return _rand_regex(rng, depth - 1) + _rand_regex(rng, depth - 1)
    if kind == 1:
        return "(" + _rand_regex(rng, depth - 1) + "|" + _rand_regex(rng, depth - 1) + ")"
    if kind == 2:
        return "(" + _rand_regex(rng, depth - 1) + ")" + rng.choice(["*", "+", "?", "{2}", "{1,3}", "{2,}"])
    return _rand_regex(rng, depth - 1)


def _rand_structtag(rng, depth):
    kind = rng.randrange(6) if depth > 0 else rng.randrange(2)
    if kind == 0:
        return {"type": "literal", "text": rng.choice(["ab", "x", "<t>", ""])}
    if kind == 1:
        return {"type": "regex", "pattern": _rand_regex(rng, 3)}
    if kind == 2:
        return {"type": "sequence", "elements": [_rand_structtag(rng, depth - 1) for _ in range(rng.randint(0, 3))]}
    if kind == 3:
        return {"type": "or", "elements": [_rand_structtag(rng, depth - 1) for _ in range(rng.randint(1, 3))]}
    if kind == 4:
        return {"type": "tag", "begin": "<t>", "content": _rand_structtag(rng, depth - 1), "end": "</t>"}
    return {"type": "evaluated_tag", "begin": "<c>", "content": _rand_structtag(rng, depth - 1), "end": "</c>",
            "evaluator": rng.choice(["arithmetic", "string"]), "result": {"begin": "<result>", "end": "</result>"}}


def test_structural_tags_match_oracle():
    """Random structural tags (nested regexes, sequences, alternatives, tags,
    evaluated tags, a JSON-schema element) compile to the oracle's tables;
    documents the oracle refuses are refused too."""
    rng = random.Random(41)
    wb = WBounds(max_len_default=12)
    b = _bounds(wb)
    docs = [_rand_structtag(rng, 3) for _ in range(120)]
    docs.append({"type": "sequence", "elements": [
        {"type": "literal", "text": "A:"},
        {"type": "json_schema", "json_schema": {"type": "object", "properties": {"n": {"type": "integer"}},
                                                "required": ["n"]}}]})
    docs += [{"type": "regex", "pattern": "^a"}, {"type": "or", "elements": []}, {"type": "literal", "text": 3},
             {"type": "tag", "begin": "<t>", "content": {"type": "literal", "text": "a"}, "end": "</t>", "x": 1}]
    for doc in docs:
        src = json.dumps(doc)
        try:
            o = build_dfa(source_to_tree("structtag", src, wb))
        except GrammarError:
            with pytest.raises(_lib.CgError):
                Grammar.compile(src, "structtag", b)
            continue
        nxt, _ = Grammar.compile(src, "structtag", b).export()
        assert np.array_equal(nxt, o.next), src


def test_compiler_unbounded_and_recursive_rules():
    srcs = ['root ::= ("ab" | "c")* "a" & [abc]{0,7}',
            'root ::= e\ne ::= "x" | "(" e ")"',
            'root ::= "a"+ "b"* & "a"{1,3} [ab]{0,2}',
            'root ::= ( [^ ] | " "{1,3} [^ ] )* " "{0,3} & [a ]{0,9}',
            'root ::= "q" @forced( [0-9]{1,3} ) "!"']
    for src in srcs:
        o = build_dfa(gbnf_to_tree(src, 4))
        nxt, _ = Grammar.compile(src, "gbnf", Bounds(depth_max=4)).export()
        assert np.array_equal(nxt, o.next), src


@pytest.mark.parametrize("schema", [
    {"type": "string", "pattern": "a+"}, {"$ref": "#/x"},
    {"type": "object", "properties": {"a": {"type": "integer"}}},
    {"type": "object", "properties": {"a": {"type": "integer"}}, "required": ["a"], "additionalProperties": True},
    {"type": "integer", "minimum": 3}, {"oneOf": [{"type": "null"}]}, {"enum": [1.5]},
    {"type": "string", "format": "date"}, {"type": "string", "minLength": 5, "maxLength": 2},
    {"enum": ["a", 1], "type": ["string", "integer"]}, {},
])
def test_fail_closed_like_the_oracle(schema):
    b = WBounds()
    with pytest.raises(GrammarError) as oe:
        schema_to_tree(json.dumps(schema), b.ws_max, b.max_len_default, b.max_items_default)
    with pytest.raises(_lib.CgError) as pe:
        Grammar.compile(json.dumps(schema), "json")
    assert oe.value.code == "unsupported" and pe.value.code == _lib.CG_E_UNSUPPORTED


def test_try_input_reports_refusal_offset():
    g = Grammar.compile(GRAMMARS["calc_call"].source, "gbnf")
    ok = b'calculate({"expression":"125*8"})'
    assert g.try_input(ok)[0::2] == (len(ok), True)
    ref, _, acc = g.try_input(b'calculate({"expression":"125x8"})')
    assert (ref, acc) == (len(b'calculate({"expression":"125'), False)
    je = Grammar.compile(GRAMMARS["json_eval"].source, "gbnf")
    text = b'{"expression": "17 * 23 + 91", "answer": 482}'
    inj = np.zeros(len(text), np.uint8)
    inj[text.index(b", "):] = 1
    assert je.try_input(text, inj)[0::2] == (len(text), True)
    assert je.try_input(text)[0] == text.index(b", ")


def test_live_states_match_oracle_rule():
    from oracle.driver import live_states
    for name in ("calc_eval", "booking_200"):
        spec = GRAMMARS[name]
        g = Grammar.compile(spec.source, spec.kind, _bounds(spec.bounds))
        assert np.array_equal(g.live_states(), live_states(oracle_dfa(name)))


def test_evaluator_matches_oracle():
    rng = random.Random(21)
    spans = [b"17 * 23 + 91", b"1 / 0", b"7 / 2", b"", b"(", b"1/0 x", b"(1/0", b".", b"1..2", b"--3",
             b"9" * 33 + b" * " + b"9" * 33, b"1" * 64, b"-" + b"1" * 64, b"1" * 65, b"0.5 * 8", b"1" * 5000]
    alphabet = b"0123456789+-*/(). "
    spans += [bytes(rng.choice(alphabet) for _ in range(rng.randint(1, 30))) for _ in range(3000)]
    for span in spans:
        for fmt in ("calc_tag", "json_answer"):
            out, _ = eval_arith(span, fmt)
            assert out == format_result(span, fmt), span


def test_string_operations_match_oracle():
    """cg_eval_strop against the oracle's string-operation evaluator, on the
    page's example, the error cases and random well- and ill-formed spans."""
    rng = random.Random(23)
    spans = [b'count("strawberry", "r")', b'len("")', b'substr("abc", -2, 99)', b'upper("a<b")', b'reverse("b<")',
             b'count("a", "")', b'lower("a")', b'len(1)', b'len("a"', b' len ( "a\\\"b" ) ', b'substr("a", 1, 2, 3)',
             b'substr("abc", 1234567890, 1)', b'upper("' + b"x" * 70 + b'")', b'len("' + b"y" * 5000 + b'")', b""]
    ops = [b"count", b"len", b"reverse", b"upper", b"substr", b"lower"]
    chars = b'ab rs"\\<,()-0123456789'
    for _ in range(4000):
        args = []
        for _ in range(rng.randint(0, 3)):
            if rng.random() < 0.6:
                body = bytes(rng.choice(b"abcrs .!\\\"") for _ in range(rng.randint(0, 12)))
                args.append(b'"' + body + b'"')
            else:
                args.append(str(rng.randint(-30, 30)).encode())
        span = rng.choice(ops) + b"(" + b", ".join(args) + b")"
        if rng.random() < 0.2:
            k = rng.randrange(len(span) + 1)
            span = span[:k] + bytes([rng.choice(chars)]) + span[k:]
        spans.append(span)
    for span in spans:
        out, ok = eval_strop(span)
        assert out == format_result(span, "strop_tag"), span
        assert ok == out.startswith(b"<result>"), span


def test_joint_mask_classes_are_sound_and_shared():
    """Mask classes computed over several grammars at once: every class's
    member states, from whichever grammar, have the same oracle mask, and
    classes are shared across grammars (fewer than computed one by one)."""
    from grammar_constrained_decoding_gb300 import mask_classes
    from oracle.step import VocabMatrix, token_mask
    names = ("calc_eval", "json_eval", "booking_200", "strop_eval")
    toks = vocab("bpe", 2000)
    max_len = max(len(t) for t in toks)
    gs = [Grammar.compile(GRAMMARS[n].source, GRAMMARS[n].kind, _bounds(GRAMMARS[n].bounds)) for n in names]
    cls, n = mask_classes(gs, max_len)
    n_sep = sum(mask_classes([g], max_len)[1] for g in gs)
    assert n < n_sep
    dfas = [oracle_dfa(x) for x in names]
    off = np.cumsum([0] + [d.n_states for d in dfas])
    vm = VocabMatrix(toks)
    members = {}
    for gi, d in enumerate(dfas):
        for s in range(d.n_states):
            members.setdefault(int(cls[off[gi] + s]), []).append((gi, s))
    shared = 0
    for c, ms in members.items():
        grammars = {gi for gi, _ in ms}
        shared += len(grammars) > 1
        pick = ms[:2] + [m for m in ms if m[0] != ms[0][0]][:2]
        want = token_mask(dfas[pick[0][0]], vm, pick[0][1])
        for gi, s in pick[1:]:
            assert np.array_equal(token_mask(dfas[gi], vm, s), want), (c, pick)
    assert shared > 0


def test_tokenizer_matches_oracle():
    toks = vocab("bpe", 4000)
    v = Vocab(toks)
    rng = random.Random(22)
    for _ in range(300):
        text = b"".join(rng.choice(toks) for _ in range(rng.randint(0, 12)))
        text += bytes(rng.randrange(256) for _ in range(rng.randint(0, 4)))
        assert v.tokenize_greedy(text) == tokenize_greedy(text, toks)


def test_driver_matches_oracle_host_rules():
    """The C++ driver applies the same host rules as the oracle on the same
    stream of (token, flags): a scripted evaluator-aware generation."""
    spec = GRAMMARS["calc_eval"]
    toks = [bytes([b]) for b in range(256)] + [b"<result>", b"</result>", b" + ", b"17"]
    v = Vocab(toks)
    d = Driver(v, 1, None, [(spec.span_open, spec.span_close, _lib.CG_RESULT_CALC_TAG)])
    run = OracleRun([oracle_dfa("calc_eval")], [spec], toks, 2048)
    row = Row(0, 0)
    script = list(b"The expression is <calc>") + [259, 258] + list(b"23 * 2") + list(b"</calc>")
    fnext = np.full(1, -1, np.int32)
    produced = []
    for step in range(80):
        x = np.zeros(len(toks))
        if script and not row.queue:
            x[script[0]] = 9.0
        else:
            x[ord(".")] = 9.0
        rec = run.step_row(row, x, 0.0, 1.0, 0, step)
        if rec["forced"] < 0 and script:
            script.pop(0)
        used = np.array([rec["forced"]], np.int32)
        assert used[0] == fnext[0]
        d.update(np.array([rec["tok"]], np.uint32), np.array([rec["flags"]], np.uint8), used, fnext)
        assert fnext[0] == (row.queue[0] if row.queue else -1)
        produced.append(rec["tok"])
        if rec["flags"] & FLAG_DONE:
            break
    text = b"".join(toks[t] for t in produced)
    assert text == b"The expression is <calc>17 + 23 * 2</calc><result>63</result>."


def test_driver_evaluates_string_operations():
    """The C++ driver evaluates a <strop> span and queues the result tokens the
    oracle's host rules queue (the page's count("strawberry", "r") = 3)."""
    spec = GRAMMARS["strop_eval"]
    toks = [bytes([b]) for b in range(256)] + [b"<result>", b"</result>", b"straw", b"berry"]
    v = Vocab(toks)
    d = Driver(v, 1, None, [(spec.span_open, spec.span_close, _lib.CG_RESULT_STROP_TAG)])
    run = OracleRun([oracle_dfa("strop_eval")], [spec], toks, 2048)
    row = Row(0, 0)
    script = list(b'The answer is <strop>count("') + [258, 259] + list(b'", "r")</strop>')
    fnext = np.full(1, -1, np.int32)
    produced = []
    for step in range(120):
        x = np.zeros(len(toks))
        if script and not row.queue:
            x[script[0]] = 9.0
        else:
            x[ord(".")] = 9.0
        rec = run.step_row(row, x, 0.0, 1.0, 0, step)
        if rec["forced"] < 0 and script:
            script.pop(0)
        used = np.array([rec["forced"]], np.int32)
        assert used[0] == fnext[0]
        d.update(np.array([rec["tok"]], np.uint32), np.array([rec["flags"]], np.uint8), used, fnext)
        assert fnext[0] == (row.queue[0] if row.queue else -1)
        produced.append(rec["tok"])
        if rec["flags"] & FLAG_DONE:
            break
    text = b"".join(toks[t] for t in produced)
    assert text == b'The answer is <strop>count("strawberry", "r")</strop><result>3</result>.'
