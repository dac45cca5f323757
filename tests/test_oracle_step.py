"""Pins for the oracle's mask, sampler and accept.

* mask: the all-tokens walk equals the scalar definition; on the calc-call
  grammar it equals a direct prefix-viability matcher written here from the
  tool-call shape (usetacet.com/docs/grammar);
* bit layout of the packed mask on a hand example;
* softmax probabilities against scipy.special.softmax;
* top-p nucleus against a per-token sort (no grouping of ties);
* greedy special cases and the T -> 0 limit of the Gumbel sampler;
* Gumbel-max frequencies against the renormalised nucleus probabilities (chi^2);
* accept flags on worked strings.
"""

import random

import numpy as np
import pytest
from scipy import special, stats

from oracle.dfa import DEAD, walk
from oracle.step import (FLAG_DONE, FLAG_FORCED_NEXT, FLAG_NO_TOKEN, FLAG_REJECTED, NO_TOKEN,
                         VocabMatrix, accept, pack_bitmask, sample_row, token_allowed,
                         token_mask, unpack_bitmask)
from tests.oracle_cache import oracle_dfa, vocab

PRE = b'calculate({"expression":"'
POST = b'"})'
BODY = set(b"0123456789+*/() -")


def _calc_call_viable(p: bytes) -> bool:
    """Is p a prefix of some calc call?  Written from the shape alone."""
    if len(p) <= len(PRE):
        return PRE.startswith(p)
    if not p.startswith(PRE):
        return False
    rest = p[len(PRE):]
    body = rest
    tail = b""
    k = rest.find(b'"')
    if k >= 0:
        body, tail = rest[:k], rest[k:]
        if not POST.startswith(tail) or not body:
            return False
    if len(body) > 64 or any(c not in BODY for c in body):
        return False
    run = 0
    for c in body:
        run = run + 1 if c == 0x20 else 0
        if run > 8:
            return False
    return True


def test_mask_matches_scalar_definition_and_direct_matcher():
    dfa = oracle_dfa("calc_call")
    toks = vocab("tiny", 512)
    vm = VocabMatrix(toks)
    rng = random.Random(3)
    for _ in range(40):
        n = rng.randint(0, 40)
        body = bytes(rng.choice(b"0123456789+*() ") for _ in range(n))
        prefix = (PRE + body)[:rng.randint(0, len(PRE) + n)]
        s = walk(dfa, 0, list(prefix))
        if s == DEAD:
            continue
        m = token_mask(dfa, vm, s)
        for t in range(len(toks)):
            assert m[t] == token_allowed(dfa, s, toks[t])
            assert m[t] == _calc_call_viable(prefix + toks[t]), (prefix, toks[t])


def test_mask_vectorised_on_bpe_vocab():
    dfa = oracle_dfa("booking_200")
    toks = vocab("bpe", 3000)
    vm = VocabMatrix(toks)
    rng = np.random.default_rng(4)
    for s in rng.integers(0, dfa.n_states, 12):
        m = token_mask(dfa, vm, int(s))
        for t in rng.integers(0, len(toks), 400):
            assert m[t] == token_allowed(dfa, int(s), toks[t])


def test_bit_layout():
    mask = np.zeros(40, dtype=bool)
    mask[[0, 31, 32, 39]] = True
    words = pack_bitmask(mask)
    assert words.tolist() == [0x80000001, 0x81]
    assert np.array_equal(unpack_bitmask(words, 40), mask)


def _row(V, seed, distinct=None):
    rng = np.random.default_rng(seed)
    x = rng.normal(0, 2, V).astype(np.float32)
    if distinct:
        x = np.round(x * distinct) / distinct
    allowed = rng.random(V) < 0.7
    return x.astype(np.float64), allowed


def test_softmax_against_scipy():
    x, allowed = _row(300, 1)
    r = sample_row(x, allowed, 0.7, 1.0, 9, 0, 0)
    T = float(np.float32(0.7))
    ref = special.softmax(x[allowed] / T)
    assert np.allclose(r.probs[allowed], ref, rtol=0, atol=1e-15)
    assert np.all(r.probs[~allowed] == 0)


@pytest.mark.parametrize("seed,distinct", [(2, None), (3, 2), (4, 1), (5, 8)])
def test_top_p_against_per_token_sort(seed, distinct):
    x, allowed = _row(400, seed, distinct)
    for top_p in (0.1, 0.5, 0.9, 0.95):
        r = sample_row(x, allowed, 0.7, top_p, 1, 0, 0)
        idx = np.flatnonzero(allowed)
        T = float(np.float32(0.7))
        z = x[idx] / T
        p = special.softmax(z)
        order = sorted(range(len(idx)), key=lambda i: (-z[i], idx[i]))
        c = 0.0
        for k, i in enumerate(order):
            c += p[i]
            if c >= float(np.float32(top_p)):
                tau = z[i]
                break
        nucleus = set(idx[z >= tau].tolist())
        assert r.nucleus_size == len(nucleus)
        assert r.tok in nucleus


def test_greedy_cases():
    x = np.array([1.0, 5.0, 5.0, 9.0, 2.0])
    allowed = np.array([True, True, True, False, True])
    assert sample_row(x, allowed, 0.0, 1.0, 0, 0, 0).tok == 1          # tie -> lowest id, masked max ignored
    one = np.zeros(5, dtype=bool)
    one[4] = True
    assert sample_row(x, one, 0.0, 1.0, 0, 0, 0).tok == 4
    assert sample_row(x, one, 0.7, 0.9, 0, 0, 0).tok == 4               # one-hot mask fixes the sample
    assert sample_row(x, np.zeros(5, dtype=bool), 0.7, 0.9, 0, 0, 0).tok == NO_TOKEN


def test_low_temperature_limit_is_greedy():
    rng = np.random.default_rng(8)
    for trial in range(30):
        x = rng.permutation(200).astype(np.float64) * 0.01   # distinct, gaps >= 0.01
        allowed = rng.random(200) < 0.5
        g = sample_row(x, allowed, 0.0, 1.0, 0, trial, 0).tok
        for top_p in (1.0, 0.5):
            assert sample_row(x, allowed, 1e-4, top_p, 77, trial, 3).tok == g


@pytest.mark.parametrize("top_p", [1.0, 0.8])
def test_gumbel_frequencies(top_p):
    x = np.array([0.3, -1.0, 1.2, 0.0, 0.9, 2.0, -0.4, 0.6])
    allowed = np.array([True, True, True, False, True, True, True, True])
    T = float(np.float32(0.7))
    r0 = sample_row(x, allowed, 0.7, top_p, 5, 0, 0)
    p = r0.probs.copy()
    if top_p < 1.0:
        z = np.where(allowed, x / T, -np.inf)
        order = np.argsort(-z)
        cum = np.cumsum(p[order])
        k = int(np.flatnonzero(cum >= float(np.float32(top_p)))[0])
        keep = z >= z[order[k]]
        p = np.where(keep, p, 0.0)
    p = p / p.sum()
    n = 20000
    counts = np.zeros(8)
    for step in range(n):
        counts[sample_row(x, allowed, 0.7, top_p, 5, 1, step).tok] += 1
    support = p > 0
    assert np.all(counts[~support] == 0)
    assert stats.chisquare(counts[support], n * p[support]).pvalue > 1e-4


def test_accept_flags():
    dfa = oracle_dfa("json_eval")
    toks = [bytes([b]) for b in range(256)] + [b'{"expression": "', b', "answer": ', b'"']
    s, f = accept(dfa, 0, 256, toks, False)
    assert f == 0 and s != DEAD
    for c in b"17 * 23 + 91":
        s, f = accept(dfa, s, c, toks, False)
        assert f == 0
    s, f = accept(dfa, s, ord('"'), toks, False)
    assert f == FLAG_FORCED_NEXT
    s_bad, f_bad = accept(dfa, s, ord(','), toks, False)             # the model may not answer
    assert s_bad == DEAD and f_bad == FLAG_REJECTED
    s, f = accept(dfa, s, 257, toks, True)
    assert f == FLAG_FORCED_NEXT
    for c in b"482":
        s, f = accept(dfa, s, c, toks, True)
    s, f = accept(dfa, s, ord("}"), toks, True)
    assert f == FLAG_DONE
    assert accept(dfa, s, NO_TOKEN, toks, False) == (s, FLAG_NO_TOKEN)
