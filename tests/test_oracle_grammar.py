"""Pins for the oracle's grammar front-ends and automaton construction.

* worked strings printed on the pages (tests/golden/worked_strings.txt);
* brute force: random small grammars, membership of every string up to length
  6 over {a,b,c} against the language computed by set algebra in this file;
* uniqueness: two sources with one language give bit-identical tables;
* minimality by brute force on small automata;
* JSON soundness: whatever the booking automaton accepts parses as JSON and
  validates against the schema; generated valid documents are accepted;
* canonical integer lexicon vs the json module (>= 1,500 cases);
* bounds: whitespace runs, maxLength, x-maxBytes, nesting depth, acyclicity;
* fail-closed refusals of unsupported schema features.
"""

import ast
import itertools
import json
import os
import random

import numpy as np
import pytest

from oracle.dfa import DEAD, build_dfa, compile_grammar, is_acyclic, walk
from oracle.grammar import GrammarError, gbnf_to_tree, schema_to_tree
from tests.oracle_cache import oracle_dfa, parse_marked
from workloads import CONFIGS, GRAMMARS, Bounds

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_strings.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        if not line.strip() or line.startswith("#"):
            continue
        g, verdict, lit = line.rstrip("\n").split("\t")
        rows.append((g, verdict, ast.literal_eval(lit)))
    return rows


@pytest.mark.parametrize("grammar,verdict,data", _golden())
def test_worked_strings(grammar, verdict, data):
    dfa = oracle_dfa(grammar)
    s = walk(dfa, 0, parse_marked(data))
    if verdict == "accept":
        assert s != DEAD and dfa.accept[s]
    elif verdict == "prefix":
        assert s != DEAD and not dfa.accept[s]
    else:
        assert s == DEAD or not dfa.accept[s]


# ---------------------------------------------------------------- brute force
ALPHA = "abc"
L = 6


def _rand_tree(rng, depth):
    k = rng.random()
    if depth == 0 or k < 0.3:
        if rng.random() < 0.5:
            return ("c", rng.choice(ALPHA))
        return ("set", "".join(sorted(rng.sample(ALPHA, rng.randint(1, 3)))))
    op = rng.choice(["cat", "cat", "alt", "and", "rep", "opt"])
    if op in ("cat", "alt", "and"):
        return (op, _rand_tree(rng, depth - 1), _rand_tree(rng, depth - 1))
    if op == "rep":
        m = rng.randint(0, 2)
        return ("rep", _rand_tree(rng, depth - 1), m, m + rng.randint(0, 2))
    return ("opt", _rand_tree(rng, depth - 1))


def _gbnf(t):
    k = t[0]
    if k == "c":
        return f'"{t[1]}"'
    if k == "set":
        return f"[{t[1]}]"
    if k == "cat":
        return f"({_gbnf(t[1])} {_gbnf(t[2])})"
    if k == "alt":
        return f"({_gbnf(t[1])} | {_gbnf(t[2])})"
    if k == "and":
        return f"({_gbnf(t[1])} & {_gbnf(t[2])})"
    if k == "rep":
        return f"({_gbnf(t[1])}){{{t[2]},{t[3]}}}"
    return f"({_gbnf(t[1])})?"


def _lang(t):
    """All words of the language, as a set (every tree here is finite)."""
    k = t[0]
    if k == "c":
        return {t[1]}
    if k == "set":
        return set(t[1])
    if k == "cat":
        return {x + y for x in _lang(t[1]) for y in _lang(t[2])}
    if k == "alt":
        return _lang(t[1]) | _lang(t[2])
    if k == "and":
        return _lang(t[1]) & _lang(t[2])
    if k == "opt":
        return _lang(t[1]) | {""}
    a = _lang(t[1])
    out, cur = set(), {""}
    for i in range(t[3] + 1):
        if i >= t[2]:
            out |= cur
        cur = {x + y for x in cur for y in a}
    return out


def _words(maxlen):
    for n in range(maxlen + 1):
        for w in itertools.product(ALPHA, repeat=n):
            yield "".join(w)


def test_bruteforce_random_grammars():
    rng = random.Random(1234)
    checked = 0
    while checked < 60:
        t = _rand_tree(rng, 4)
        lang = _lang(t)
        if not lang or max(len(w) for w in lang) > L:
            continue
        src = "root ::= " + _gbnf(t)
        dfa = build_dfa(gbnf_to_tree(src, 5))
        prefixes = {w[:i] for w in lang for i in range(len(w) + 1)}
        for w in _words(L):
            s = walk(dfa, 0, list(w.encode()))
            assert (s != DEAD and bool(dfa.accept[s])) == (w in lang), (src, w)
            assert (s != DEAD) == (w in prefixes), (src, w)
        checked += 1


def test_unbounded_repetition_membership():
    src = 'root ::= ("ab" | "c")* "a" & [abc]{0,5}'
    dfa = build_dfa(gbnf_to_tree(src, 5))
    import re
    for w in _words(L):
        s = walk(dfa, 0, list(w.encode()))
        expect = re.fullmatch(r"(ab|c)*a", w) is not None and len(w) <= 5
        assert (s != DEAD and bool(dfa.accept[s])) == expect


def test_same_language_same_tables():
    pairs = [
        ('root ::= "ab" | "ac"', 'root ::= "a" [bc]'),
        ('root ::= "x"{2,4}', 'root ::= "xx" "x"? "x"?'),
        ('root ::= ([ab] "c")? "d"', 'root ::= "d" | "ac" "d" | "bcd"'),
        ('root ::= [a-c]{1,3} & "b"*', 'root ::= "b" | "bb" | "bbb"'),
    ]
    for a, b in pairs:
        da = build_dfa(gbnf_to_tree(a, 5))
        db = build_dfa(gbnf_to_tree(b, 5))
        assert np.array_equal(da.next, db.next) and np.array_equal(da.accept, db.accept), (a, b)


def test_minimal_by_bruteforce():
    for src in ['root ::= ("a" | "b"){0,3} "c"', 'root ::= [ab]{1,4} & ("a" [ab]*)',
                'root ::= "a"{0,2} ("b" | "c" "c")?']:
        dfa = build_dfa(gbnf_to_tree(src, 5))
        sigs = set()
        for s in range(dfa.n_states):
            suffixes = frozenset(w for w in _words(6)
                                 if (e := walk(dfa, s, list(w.encode()))) != DEAD and dfa.accept[e])
            assert suffixes not in sigs, src
            sigs.add(suffixes)


def test_canonical_numbering_is_breadth_first():
    dfa = oracle_dfa("calc_eval")
    seen = {0}
    order = [0]
    for s in order:
        for a in range(512):
            d = int(dfa.next[s, a])
            if d >= 0 and d not in seen:
                seen.add(d)
                order.append(d)
    assert order == list(range(dfa.n_states))


# -------------------------------------------------------------- JSON soundness
_SCHEMA = json.loads(GRAMMARS["booking"].source)


def _validate_booking(obj):
    props = _SCHEMA["properties"]
    if not isinstance(obj, dict) or list(obj) != list(props):
        return False
    el = obj["eligibility"]
    if not isinstance(el, dict) or list(el) != ["criteria_met", "reason_code"]:
        return False
    if not isinstance(el["criteria_met"], bool):
        return False
    if el["reason_code"] not in props["eligibility"]["properties"]["reason_code"]["enum"]:
        return False
    if obj["action"] not in props["action"]["enum"]:
        return False
    ap = obj["appointment"]
    if ap is not None:
        if not isinstance(ap, dict) or list(ap) != ["date", "time"]:
            return False
        if not (isinstance(ap["date"], str) and len(ap["date"]) <= 20):
            return False
        if not (isinstance(ap["time"], str) and len(ap["time"]) <= 10):
            return False
    return isinstance(obj["response_text"], str) and len(obj["response_text"]) <= 700


def _random_booking(rng):
    ascii_only = rng.random() < 0.5
    # an escaped astral character is two escapes, i.e. two characters of the
    # schema's maxLength, so the generator keeps emoji to raw UTF-8 output
    alphabet = "abc XYZ,.'éλ€\\\"\n/\u00e9" + ("" if ascii_only else "😀")

    def s(n):
        return "".join(rng.choice(alphabet) for _ in range(rng.randint(0, n)))
    obj = {"eligibility": {"criteria_met": rng.random() < 0.5,
                           "reason_code": rng.choice(_SCHEMA["properties"]["eligibility"]["properties"]["reason_code"]["enum"])},
           "action": rng.choice(_SCHEMA["properties"]["action"]["enum"]),
           "appointment": rng.choice([None, {"date": s(20), "time": s(10)}]),
           "response_text": s(60)}
    ws = lambda: rng.choice(["", " ", "  ", "\n", "\t ", "    "])
    sep = (ws() + "," + ws(), ws() + ":" + ws())
    return json.dumps(obj, ensure_ascii=ascii_only, separators=sep).encode()


def test_booking_accepts_generated_documents():
    dfa = oracle_dfa("booking")
    rng = random.Random(5)
    for _ in range(300):
        doc = _random_booking(rng)
        s = walk(dfa, 0, list(doc))
        assert s != DEAD and dfa.accept[s], doc


def test_booking_soundness_under_mutation():
    dfa = oracle_dfa("booking")
    rng = random.Random(6)
    accepted = 0
    for _ in range(3000):
        doc = bytearray(_random_booking(rng))
        for _ in range(rng.randint(1, 3)):
            i = rng.randrange(len(doc))
            op = rng.random()
            if op < 0.4:
                doc[i] = rng.choice(b'{}[]:,"\\ 0aetn\x00\xff\xc3')
            elif op < 0.7:
                del doc[i]
            else:
                doc.insert(i, rng.choice(b'{}[]:," \\ea\xe2'))
        s = walk(dfa, 0, list(doc))
        if s != DEAD and dfa.accept[s]:
            accepted += 1
            obj = json.loads(bytes(doc).decode("utf-8"))
            assert _validate_booking(obj), bytes(doc)
    assert accepted > 50


# ---------------------------------------------------------- integer lexicon
def _is_json_integer(text: str) -> bool:
    if text != text.strip() or not text:
        return False
    try:
        v = json.loads(text)
    except ValueError:
        return False
    return isinstance(v, int) and not isinstance(v, bool) and len(text.lstrip("-")) <= 19


def test_integer_lexicon_property():
    dfa = oracle_dfa("reasoning_answer_1024")
    # the whitespace slots around the value are filled to their cap (4), so any
    # further space belongs to the candidate lexeme itself
    prefix = list(b'{"reasoning":"x","answer":    ')
    base = walk(dfa, 0, prefix)
    rng = random.Random(7)
    alphabet = "0123456789-+.eE tfrua"
    cases = ["+26", "00026", "26.0", "2.6e1", "true", "false", "-0", "0", "-", "", "1" * 19, "1" * 20,
             "-" + "9" * 19, "18000", "-14", "01", " 1", "1 "]
    while len(cases) < 1600:
        n = rng.randint(1, 22)
        cases.append("".join(rng.choice(alphabet) for _ in range(n)))
    for c in cases:
        s = walk(dfa, base, list(c.encode()) + list(b"    }"))
        assert (s != DEAD and bool(dfa.accept[s])) == _is_json_integer(c), c


def test_integer_boundary_keeps_minus_drops_quote():
    # dev.to "I found a runner bug...": where the answer starts, an integer-typed
    # field allows a minus sign but neither a quote nor a space.
    dfa = oracle_dfa("reasoning_answer_1024")
    s = walk(dfa, 0, list(b'{"reasoning":"x","answer":'))
    assert dfa.next[s, ord("-")] >= 0
    assert all(dfa.next[s, ord(d)] >= 0 for d in "0123456789")
    assert dfa.next[s, ord('"')] < 0
    assert dfa.next[s, ord("+")] < 0


# ----------------------------------------------------------------- bounds
def _refused(dfa, data):
    s = walk(dfa, 0, parse_marked(data))
    return s == DEAD or not dfa.accept[s]


def test_string_and_byte_bounds():
    dfa = oracle_dfa("booking")
    head = b'{"eligibility":{"criteria_met":true,"reason_code":"eligible"},"action":"decline","appointment":null,"response_text":"'
    assert not _refused(dfa, head + b"a" * 700 + b'"}')
    assert _refused(dfa, head + b"a" * 701 + b'"}')
    assert not _refused(dfa, head + "é".encode() * 700 + b'"}')        # code points, not bytes
    assert not _refused(dfa, head + b"\\u00e9" * 700 + b'"}')           # an escape is one character
    assert _refused(dfa, head + b"\xc3" + b'"}')                          # truncated UTF-8
    assert _refused(dfa, head + b"\xed\xa0\x80" + b'"}')                  # surrogate
    ra = oracle_dfa("reasoning_answer_1024")
    assert not _refused(ra, b'{"reasoning":"' + b"b" * 1024 + b'","answer":1}')
    assert _refused(ra, b'{"reasoning":"' + b"b" * 1025 + b'","answer":1}')
    assert not _refused(ra, b'{"reasoning":"' + "é".encode() * 512 + b'","answer":1}')
    assert _refused(ra, b'{"reasoning":"' + "é".encode() * 513 + b'","answer":1}')


def test_whitespace_runs():
    dfa = oracle_dfa("reasoning_answer_1024")
    for n in range(0, 5):
        assert not _refused(dfa, b'{' + b" " * n + b'"reasoning":"x","answer":1}')
    assert _refused(dfa, b'{' + b" " * 5 + b'"reasoning":"x","answer":1}')
    assert _refused(dfa, b'{"reasoning":"x","answer":1} ')


def test_nesting_depth_bound():
    dfa = oracle_dfa("calc_eval")
    pre = b"The expression is <calc>"
    post = b"</calc>"
    ok = b"(" * 4 + b"1" + b")" * 4
    bad = b"(" * 5 + b"1" + b")" * 5
    s = walk(dfa, 0, list(pre + ok + post))
    assert s != DEAD and dfa.forced_only()[s]
    assert walk(dfa, 0, list(pre + bad + post)) == DEAD


@pytest.mark.parametrize("name", sorted(GRAMMARS))
def test_workload_automata_invariants(name):
    dfa = oracle_dfa(name)
    assert is_acyclic(dfa)                                   # every bound is finite
    sink, fo = dfa.sink(), dfa.forced_only()
    model_moves = (dfa.next[:, :256] >= 0).any(axis=1)
    # a live state that is neither finished nor waiting for injected bytes
    # always offers the model a byte (all single bytes are tokens: mask non-empty)
    assert np.all(sink | fo | model_moves)
    assert int(dfa.accept.sum()) == int(sink.sum())           # accepting states are final
    if any(name in c.grammars for c in CONFIGS.values()):
        assert 500 <= dfa.n_states <= 30000                   # the workloads' automaton sizes


def test_fail_closed():
    b = Bounds()
    for schema in [{"type": "string", "pattern": "a+"}, {"$ref": "#/x"},
                   {"type": "object", "properties": {"a": {"type": "integer"}}},
                   {"type": "object", "properties": {"a": {"type": "integer"}}, "required": ["a"],
                    "additionalProperties": True},
                   {"type": "integer", "minimum": 3}, {"oneOf": [{"type": "null"}]},
                   {"enum": [1.5]}, {"type": "string", "format": "date"}]:
        with pytest.raises(GrammarError) as e:
            schema_to_tree(json.dumps(schema), b.ws_max, b.max_len_default, b.max_items_default)
        assert e.value.code == "unsupported"
    with pytest.raises(GrammarError):
        gbnf_to_tree('root ::= "a" missing', 5)
    with pytest.raises(GrammarError):
        compile_grammar("gbnf", 'root ::= "a" & "b"', b)
