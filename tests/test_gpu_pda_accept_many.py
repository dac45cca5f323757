"""Speculative verification of pushdown rows (cg_pda_accept_many) against the
oracle's accept_many on the DFA of the same grammar under the same stack bound
(oracle/step.py, oracle/pda.py).

Rows are first advanced by a random number of allowed tokens (through
cg_pda_accept and the oracle side by side), so that they start from varied
configurations.  Drafts are walks of the oracle automaton: allowed tokens one
after another, a refused token planted in some rows, random lengths (empty
drafts included).  Tokens accepted, flags and counts must equal the oracle's,
and the rows' next masks (cg_pda_fill_bitmask) must equal the oracle's masks
of the state after the accepted prefix.  On the grammar with a forced region,
positions whose state continues only with injected bytes are pinned to a
single-byte token, as the host driver pins an evaluator's result.
"""

import numpy as np
import pytest

from oracle.dfa import DEAD
from oracle.pda import compile_pda
from oracle.step import NO_TOKEN, VocabMatrix, accept, accept_many, pack_bitmask, token_mask
from tests.gpu_helpers import empty, host, make_ctx, product_vocab, u32
from tests.oracle_cache import vocab
from workloads.grammars import JSON_NESTED

pytestmark = pytest.mark.gpu

MIXED = r'''
root ::= "call " args @forced( "=" [0-9]{1,3} ) " ok"
args ::= "(" item ( "," item )* ")"
item ::= [0-9]+ | args
'''


class Masks:
    def __init__(self, dfa, toks):
        self.dfa, self.vm, self.V = dfa, VocabMatrix(toks), len(toks)
        self.cache = {}

    def ids(self, s):
        if s not in self.cache:
            self.cache[s] = np.flatnonzero(token_mask(self.dfa, self.vm, s)) if s != DEAD else np.zeros(0, np.int64)
        return self.cache[s]

    def packed(self, s):
        m = np.zeros(self.V, bool)
        m[self.ids(s)] = True
        return pack_bitmask(m)


def _forced_only(dfa, s):
    return s != DEAD and (dfa.next[s, :256] < 0).all() and (dfa.next[s, 256:] >= 0).any()


def _run(source, D, V, B, K, seed, max_tokens, pins):
    import torch
    from grammar_constrained_decoding_gb300 import Pda, PdaGrammar
    toks = vocab("bpe", V)
    dfa = compile_pda(source, D)
    mk = Masks(dfa, toks)
    single = {t[0]: i for i, t in enumerate(toks) if len(t) == 1}
    ctx = make_ctx(("calc_call",), "bpe", V)
    pda = Pda(ctx, product_vocab("bpe", V), PdaGrammar(source, D))
    rng = np.random.default_rng(seed)
    cfg = torch.zeros((B, D + 2), dtype=torch.int32, device="cuda").view(torch.uint32)
    flags = empty((B,), torch.uint8)
    st = [0] * B

    def pick(s):
        """An allowed next token and its pin (-1 for none) from oracle state s."""
        if pins and _forced_only(dfa, s):
            live = np.flatnonzero(dfa.next[s, 256:] >= 0)
            t = single[int(live[rng.integers(live.size)])]
            return t, t
        ids = mk.ids(s)
        return (int(ids[rng.integers(ids.size)]) if ids.size else NO_TOKEN), -1

    # a random prefix per row, accepted one token per call on both sides
    for _ in range(int(rng.integers(3, 9))):
        tk = np.empty(B, np.uint32)
        fc = np.full(B, -1, np.int32)
        for b in range(B):
            t, f = pick(st[b]) if rng.random() < 0.8 else (NO_TOKEN, -1)
            tk[b], fc[b] = t, f
        pda.accept(cfg, u32(tk), flags, forced=u32(fc.view(np.uint32)).view(torch.int32))
        g_fl = host(flags)
        for b in range(B):
            if tk[b] == NO_TOKEN:
                continue
            s, f = accept(dfa, st[b], int(tk[b]), toks, fc[b] >= 0)
            assert g_fl[b] == f, b
            if f & 1:  # a finished row starts again
                cfg.view(torch.int32)[b] = 0
                s = 0
            st[b] = s
    assert ctx.status() == 0
    # drafts
    draft = np.zeros((B, K), np.uint32)
    forced = np.full((B, K), -1, np.int32)
    dlen = rng.integers(0, K + 1, B).astype(np.uint32)
    for b in range(B):
        s = st[b]
        cut_at = int(rng.integers(0, K)) if rng.random() < 0.35 else K
        for j in range(int(dlen[b])):
            if j == cut_at and s != DEAD:
                ids = mk.ids(s)
                refused = np.setdiff1d(np.arange(V), ids)
                draft[b, j] = int(refused[rng.integers(refused.size)])
                s = DEAD
                continue
            if s == DEAD:
                draft[b, j] = int(rng.integers(V))
                continue
            t, f = pick(s)
            if t == NO_TOKEN:
                draft[b, j] = int(rng.integers(V))
                s = DEAD
                continue
            draft[b, j], forced[b, j] = t, f
            s = accept(dfa, s, t, toks, f >= 0)[0]
    counts0 = rng.integers(0, max_tokens, B).astype(np.uint32)
    counts = u32(counts0)
    out_n = empty((B,), torch.int32).view(torch.uint32)
    pda.accept_many(cfg, u32(draft), u32(dlen), out_n, flags,
                    forced=u32(forced.view(np.uint32)).view(torch.int32) if pins else None,
                    counts=counts, max_tokens=max_tokens)
    assert ctx.status() == 0
    g_n, g_fl, g_cnt = host(out_n).view(np.uint32), host(flags), host(counts).view(np.uint32)
    W = (V + 31) // 32
    bm = empty((B, W), torch.int32)
    pda.fill_bitmask(cfg, bm)
    g_bm = host(bm).view(np.uint32)
    n_cut = n_long = 0
    for b in range(B):
        res = accept_many(dfa, st[b], [int(x) for x in draft[b, :dlen[b]]], toks,
                          [int(x) for x in forced[b, :dlen[b]]] if pins else None, int(counts0[b]), max_tokens)
        assert (g_n[b], g_fl[b], g_cnt[b]) == (res.n, res.flags, res.count), (b, g_n[b], g_fl[b], res)
        assert np.array_equal(g_bm[b], mk.packed(res.state)), b
        n_cut += bool(res.flags & 32)
        n_long += res.n >= 3
    assert n_cut > B // 10 and n_long > B // 10


def test_json_drafts_match_the_oracle():
    _run(JSON_NESTED, 8, 32000, 128, 8, 3, 14, pins=False)


def test_pinned_drafts_on_a_forced_region_match_the_oracle():
    _run(MIXED, 4, 4096, 96, 10, 4, 40, pins=True)
