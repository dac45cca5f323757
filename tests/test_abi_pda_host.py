"""The pushdown compiler of the C library against the oracle, on the host.

cg_pda_try_input walks bytes through the compiled pushdown automaton (its
actions, call chains, pops and headroom checks) from a fresh row; the oracle
walks the same bytes through the DFA of the same grammar flattened under the
same stack bound (oracle/pda.py).  For every string both must refuse the same
byte (or none) and agree on whether the text may end.  Strings: random walks
of the oracle automaton (long viable prefixes, deep nesting), then random
edits of them.  Plus the grammar class the compiler refuses (left recursion,
recursive rules matching the empty string, two actions for one byte, a rule
that may both end and continue on a byte, recursion inside @forced or '&').
"""

import ctypes as C
import random

import numpy as np
import pytest

from grammar_constrained_decoding_gb300 import CgError, PdaGrammar
from grammar_constrained_decoding_gb300 import _lib as L
from oracle.dfa import DEAD
from oracle.grammar import GrammarError
from oracle.pda import compile_pda
from workloads.grammars import JSON_NESTED

DYCK = r'''
root ::= pair*
pair ::= "(" pair* ")"
'''
TREE = r'''
root ::= node "."
node ::= "(" node "," node ")" | [a-c]+
'''
ROOTED = r'''
root ::= "[" ( root ( ";" root )* )? "]" | "x"
'''
MIXED = r'''
root ::= "call " args @forced( "=" [0-9]{1,3} ) " ok"
args ::= "(" item ( "," item )* ")"
item ::= [0-9]+ | args
'''


def _oracle_walk(dfa, syms):
    """(index of the first refused symbol or len, accepted)."""
    s = 0
    for i, a in enumerate(syms):
        s = int(dfa.next[s, a])
        if s == DEAD:
            return i, False
    return len(syms), bool(dfa.accept[s])


def _random_walk(dfa, rng, n_max, inj_ok=True):
    """Bytes and injected flags of a random walk from the start state."""
    s, out, inj = 0, [], []
    for _ in range(rng.randrange(0, n_max)):
        live = np.flatnonzero(dfa.next[s] >= 0)
        if not inj_ok:
            live = live[live < 256]
        if live.size == 0:
            break
        a = int(live[rng.randrange(live.size)])
        out.append(a & 255)
        inj.append(a >= 256)
        s = int(dfa.next[s, a])
    return out, inj


def _edit(data, inj, rng, alphabet):
    data, inj = list(data), list(inj)
    for _ in range(rng.randrange(1, 3)):
        op = rng.randrange(3) if data else 1
        if op == 1:
            i = rng.randrange(len(data) + 1)
            data.insert(i, rng.choice(alphabet))
            inj.insert(i, inj[i - 1] if 0 < i <= len(inj) else False)
        elif op == 0:
            data[rng.randrange(len(data))] = rng.choice(alphabet)
        else:
            i = rng.randrange(len(data))
            del data[i]
            del inj[i]
    return data, inj


def _check(source, D, n, alphabet, seed, n_max=60):
    dfa = compile_pda(source, D)
    g = PdaGrammar(source, D)
    rng = random.Random(seed)
    seen_acc = seen_cut = 0
    for k in range(n):
        data, inj = _random_walk(dfa, rng, n_max)
        if k % 2:
            data, inj = _edit(data, inj, rng, alphabet)
        syms = [b + (256 if f else 0) for b, f in zip(data, inj)]
        want = _oracle_walk(dfa, syms)
        got = g.try_input(bytes(data), np.array(inj, dtype=np.uint8) if any(inj) else None)
        assert (got[0], got[1]) == want, (bytes(data), inj, got, want)
        seen_acc += want[1]
        seen_cut += want[0] < len(syms)
    assert seen_acc > n // 20 and seen_cut > n // 20


@pytest.mark.parametrize("D", [1, 2, 3, 5, 8])
def test_json_nested_matches_the_oracle(D):
    _check(JSON_NESTED, D, 600, list(b'{}[]",:-019atrue '), 100 + D)


@pytest.mark.parametrize("D", [1, 2, 4, 6])
def test_dyck_matches_the_oracle(D):
    _check(DYCK, D, 400, list(b"()x"), 200 + D)


@pytest.mark.parametrize("D", [1, 2, 3, 5])
def test_tree_with_completion_heights_matches_the_oracle(D):
    # a node needs two children once opened, so the headroom a prefix needs
    # grows with every open "(" and every pending second child
    _check(TREE, D, 500, list(b"(),abc."), 300 + D)


@pytest.mark.parametrize("D", [0, 1, 3, 4])
def test_recursive_start_rule_matches_the_oracle(D):
    _check(ROOTED, D, 400, list(b"[];x"), 400 + D)


@pytest.mark.parametrize("D", [2, 3, 5])
def test_forced_region_after_recursion_matches_the_oracle(D):
    # args and item call each other: an argument list needs two frames
    _check(MIXED, D, 400, list(b"call (),0123= ok"), 500 + D)


def test_sizes_stay_small_where_the_flattened_automaton_grows():
    g8 = PdaGrammar(JSON_NESTED, 8).info()
    g64 = PdaGrammar(JSON_NESTED, 64).info()
    assert g8["n_states"] == g64["n_states"] and g64["depth"] == 64
    assert g8["n_rules"] == 5
    assert compile_pda(JSON_NESTED, 12).n_states > 10 * g8["n_states"]


@pytest.mark.parametrize("src,why", [
    (r'''root ::= e
e ::= e "+" "x" | "x"''', "left recursion"),
    (r'''root ::= e "."
e ::= "(" e ")" | ""''', "recursive rule matching the empty string"),
    (r'''root ::= a | b
a ::= "x" a | "y"
b ::= "x" b | "z"''', "two rules start with the same byte"),
    (r'''root ::= a "b"
a ::= "(" a ")" "b"? | "x"''', "a rule may end or continue on 'b'"),
    (r'''root ::= "<" @forced( e ) ">"
e ::= "(" e ")" | "x"''', "recursion inside @forced"),
    (r'''root ::= e & "(x)"
e ::= "(" e ")" | "x"''', "recursion under '&'"),
])
def test_refused_grammar_class(src, why):
    with pytest.raises(CgError) as ei:
        PdaGrammar(src, 4)
    assert ei.value.code == L.CG_E_UNSUPPORTED, why


def test_argument_and_emptiness_errors():
    with pytest.raises(CgError) as ei:
        PdaGrammar(DYCK, L.CG_PDA_MAX_DEPTH + 1)
    assert ei.value.code == L.CG_E_ARG
    with pytest.raises(CgError) as ei:
        PdaGrammar(r'''root ::= e
e ::= "(" e ")"''', 4)
    assert ei.value.code == L.CG_E_EMPTY
    with pytest.raises(CgError) as ei:
        PdaGrammar(r'''root ::= e''', 4)
    assert ei.value.code == L.CG_E_UNDEFINED_RULE
    # a JSON text needs the value frame: with no frame the language is empty
    with pytest.raises(CgError) as ei:
        PdaGrammar(JSON_NESTED, 0)
    assert ei.value.code == L.CG_E_EMPTY
    with pytest.raises(GrammarError):
        compile_pda(JSON_NESTED, 0)


def test_device_entry_points_refuse_missing_handles_without_a_gpu():
    """The pushdown device calls check their arguments on the host before any
    CUDA call: a NULL object or a NULL required buffer is CG_E_ARG."""
    lib = L.lib()
    dummy = 16  # a non-null address the calls must not reach
    assert lib.cg_pda_fill_bitmask(None, dummy, 4, None, dummy) == L.CG_E_ARG
    assert lib.cg_pda_accept(None, dummy, 4, dummy, None, None, 0, dummy) == L.CG_E_ARG
    assert lib.cg_pda_accept_fill(None, dummy, 4, dummy, None, None, 0, dummy, None, dummy) == L.CG_E_ARG
    assert lib.cg_pda_accept_many(None, dummy, 4, dummy, dummy, None, 8, None, 0, dummy, dummy) == L.CG_E_ARG
    assert lib.cg_pda_step(None, dummy, 4, dummy, L.CG_BF16, 4096, 0.7, 0.9, 1, 0, None, None, 0, None, dummy,
                           dummy) == L.CG_E_ARG
    assert lib.cg_pda_create(None, None, None, None) == L.CG_E_ARG
    assert lib.cg_pda_info(None, None, None, None, None) == L.CG_E_ARG
    assert lib.cg_pda_grammar_info(None, None, None, None, None) == L.CG_E_ARG
    n, acc = C.c_size_t(), C.c_int()
    assert lib.cg_pda_try_input(None, b"x", 1, None, C.byref(n), C.byref(acc), None) == L.CG_E_ARG
    lib.cg_pda_destroy(None)
    lib.cg_pda_grammar_destroy(None)
