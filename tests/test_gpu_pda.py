"""Pushdown rows on the GPU (cg_pda_fill_bitmask / cg_pda_accept) against the
oracle of the same grammar flattened under the same stack bound.

* random walks: every row starts fresh; at each step the device mask of every
  row must equal the oracle's mask of the DFA state the same tokens reached,
  bit for bit; the row then takes a random allowed token (biased towards
  tokens that open brackets, so that rows nest deeply and pop through the
  per-row token lists), some rows a refused one, and the device flags must
  equal the oracle's (REJECTED, DONE, and the restart of finished rows when
  counts are kept) -- json_nested at a stack bound of 8 with the 128256-token
  vocabulary and 256 rows, and at 16 with 32000 tokens;
* the three-call path with sampling (cg_mask_and_sample between the two):
  ids identical to the oracle's sampler except where its rounding tolerance
  allows, flags identical;
* a forced region after recursion: one-hot masks, injected walks and
  FORCED_NEXT as the oracle has them;
* a stack bound of 32 (the flattened automaton grows about 1.3 times per
  frame: 1896 states at 16): rows nest to the bound, where the device refuses
  a further "[", and every finished text parses as JSON within the bound;
* edge cases: an empty batch, malformed configurations, refused and
  out-of-range tokens, a forced token that differs from the sampled one;
* cg_pda_accept_fill equals cg_pda_accept followed by cg_pda_fill_bitmask;
* cg_pda_step (the fused pushdown step) equals the three calls, with and
  without forced rows;
* random walks on two more grammar shapes: one whose open nodes need headroom
  to complete, one whose start rule is itself recursive.
"""

import json

import numpy as np
import pytest

from oracle.dfa import DEAD
from oracle.pda import compile_pda
from oracle.step import FLAG_DONE, NO_TOKEN, VocabMatrix, accept, pack_bitmask, sample_row, token_mask
from tests.gpu_helpers import empty, host, logits_rows, make_ctx, product_vocab, same_token, u32
from tests.oracle_cache import vocab
from workloads.grammars import JSON_NESTED

pytestmark = pytest.mark.gpu

MIXED = r'''
root ::= "call " args @forced( "=" [0-9]{1,3} ) " ok"
args ::= "(" item ( "," item )* ")"
item ::= [0-9]+ | args
'''


class OracleRows:
    """Oracle DFA states of B rows, with a cache of packed masks per state."""

    def __init__(self, source, D, toks):
        self.dfa = compile_pda(source, D)
        self.vm = VocabMatrix(toks)
        self.toks = toks
        self.masks = {}

    def mask(self, s):
        if s not in self.masks:
            self.masks[s] = (pack_bitmask(token_mask(self.dfa, self.vm, s)) if s != DEAD
                             else np.zeros((self.vm.V + 31) // 32, np.uint32))
        return self.masks[s]


def _pda(source, D, V):
    from grammar_constrained_decoding_gb300 import Pda, PdaGrammar
    ctx = make_ctx(("calc_call",), "bpe", V)  # the context's own grammar is not used here
    g = PdaGrammar(source, D)
    return ctx, Pda(ctx, product_vocab("bpe", V), g)


def _fresh(B, D):
    import torch
    cfg = torch.zeros((B, D + 2), dtype=torch.int32, device="cuda")
    return cfg.view(torch.uint32)


def _pick(rng, allowed_words, V, opens, bias):
    ids = np.flatnonzero(np.unpackbits(allowed_words.view(np.uint8), bitorder="little")[:V])
    if ids.size == 0:
        return NO_TOKEN
    deep = ids[opens[ids] > 0]
    if deep.size and rng.random() < bias:
        return int(deep[rng.integers(deep.size)])
    return int(ids[rng.integers(ids.size)])


@pytest.mark.parametrize("D,V,B,steps", [(8, 128256, 256, 24), (16, 32000, 128, 40)])
def test_random_walk_masks_and_flags_match_the_oracle(D, V, B, steps):
    import torch
    toks = vocab("bpe", V)
    orc = OracleRows(JSON_NESTED, D, toks)
    ctx, pda = _pda(JSON_NESTED, D, V)
    opens = np.array([t.count(b"[") + t.count(b"{") for t in toks])
    rng = np.random.default_rng(D)
    W = (V + 31) // 32
    cfg = _fresh(B, D)
    bm = empty((B, W), torch.int32)
    flags = empty((B,), torch.uint8)
    counts = torch.zeros((B,), dtype=torch.int32, device="cuda").view(torch.uint32)
    max_tokens = 30
    st = [0] * B
    cnt = [0] * B
    max_level = n_done = n_rej = 0
    for step in range(steps):
        pda.fill_bitmask(cfg, bm)
        assert ctx.status() == 0
        g_bm = host(bm).view(np.uint32)
        pick = np.empty(B, np.uint32)
        for b in range(B):
            want = orc.mask(st[b])
            assert np.array_equal(g_bm[b], want), (step, b)
            if st[b] != DEAD and rng.random() < 0.03:
                refused = np.flatnonzero(~np.unpackbits(want.view(np.uint8), bitorder="little")[:V].astype(bool))
                pick[b] = int(refused[rng.integers(refused.size)])
            else:
                pick[b] = _pick(rng, want, V, opens, 0.3)
        pda.accept(cfg, u32(pick), flags, counts=counts, max_tokens=max_tokens)
        code = ctx.status()
        g_fl = host(flags)
        g_cfg = host(cfg).view(np.uint32)
        for b in range(B):
            t = int(pick[b])
            if t == NO_TOKEN:
                s, f = st[b], 8
            else:
                s, f = accept(orc.dfa, st[b], t, toks, False)
            n = cnt[b] + (t != NO_TOKEN)
            if f & FLAG_DONE or n >= max_tokens:
                f |= 0 if f & FLAG_DONE else 16
                s, n = 0, 0
            assert g_fl[b] == f, (step, b, t, g_fl[b], f)
            assert (g_cfg[b, 0] == 0xFFFFFFFF) == (s == DEAD), (step, b)
            n_done += bool(f & FLAG_DONE)
            n_rej += bool(f & 4)
            st[b], cnt[b] = s, n
            max_level = max(max_level, int(g_cfg[b, 1]))
        assert code in (0, 7)  # CG_DEV_REJECTED from the refused picks
        # failed rows start again, with their token counts
        dead = [b for b in range(B) if st[b] == DEAD]
        if dead:
            cfg.view(torch.int32)[dead] = 0
            counts.view(torch.int32)[dead] = 0
            for b in dead:
                st[b], cnt[b] = 0, 0
    assert n_rej > 0 and max_level >= min(D, 6)


def test_sampled_three_call_path_matches_the_oracle():
    import torch
    D, V, B, steps = 8, 32000, 64, 16
    temp, top_p, seed = 0.7, 0.9, 11
    toks = vocab("bpe", V)
    orc = OracleRows(JSON_NESTED, D, toks)
    ctx, pda = _pda(JSON_NESTED, D, V)
    W = (V + 31) // 32
    cfg = _fresh(B, D)
    bm = empty((B, W), torch.int32)
    tok = empty((B,), torch.int32)
    flags = empty((B,), torch.uint8)
    st = [0] * B
    for step in range(steps):
        vals, x = logits_rows(V, range(B), step, 3, 2.0, 4.0, 0.05, "bf16")
        pda.fill_bitmask(cfg, bm)
        ctx.mask_and_sample(x, bm, temp, top_p, seed, step, tok)
        g_tok = host(tok).view(np.uint32).copy()
        pda.accept(cfg, tok.view(torch.uint32), flags)
        assert ctx.status() == 0
        g_bm, g_fl = host(bm).view(np.uint32), host(flags)
        for b in range(B):
            want = orc.mask(st[b])
            assert np.array_equal(g_bm[b], want), (step, b)
            allowed = np.unpackbits(want.view(np.uint8), bitorder="little")[:V].astype(bool)
            res = sample_row(vals[b], allowed, temp, top_p, seed, b, step)
            assert same_token(int(g_tok[b]), res), (step, b)
            s, f = accept(orc.dfa, st[b], int(g_tok[b]), toks, False) if g_tok[b] != NO_TOKEN else (st[b], 8)
            assert g_fl[b] == f, (step, b)
            st[b] = s
        done = [b for b in range(B) if g_fl[b] & FLAG_DONE]
        if done:  # finished rows start again
            cfg.view(torch.int32)[done] = 0
            for b in done:
                st[b] = 0


def test_forced_region_after_recursion_matches_the_oracle():
    import torch
    D, V, B = 4, 4096, 32
    toks = vocab("bpe", V)
    orc = OracleRows(MIXED, D, toks)
    ctx, pda = _pda(MIXED, D, V)
    W = (V + 31) // 32
    rng = np.random.default_rng(5)
    single = {t[0]: i for i, t in enumerate(toks) if len(t) == 1}
    cfg = _fresh(B, D)
    bm = empty((B, W), torch.int32)
    flags = empty((B,), torch.uint8)
    st = [0] * B
    n_forced = 0
    for step in range(40):
        forced = np.full(B, -1, np.int32)
        for b in range(B):
            s = st[b]
            if s != DEAD and (orc.dfa.next[s, :256] < 0).all() and (orc.dfa.next[s, 256:] >= 0).any():
                live = np.flatnonzero(orc.dfa.next[s, 256:] >= 0)
                forced[b] = single[int(live[rng.integers(live.size)])]
        pda.fill_bitmask(cfg, bm, forced=u32(forced.view(np.uint32)).view(torch.int32))
        g_bm = host(bm).view(np.uint32)
        pick = np.empty(B, np.uint32)
        for b in range(B):
            if forced[b] >= 0:
                want = np.zeros(W, np.uint32)
                want[forced[b] >> 5] = np.uint32(1 << (forced[b] & 31))
                pick[b] = forced[b]
                n_forced += 1
            else:
                want = orc.mask(st[b])
                ids = np.flatnonzero(np.unpackbits(want.view(np.uint8), bitorder="little")[:V])
                pick[b] = int(ids[rng.integers(ids.size)]) if ids.size else NO_TOKEN
            assert np.array_equal(g_bm[b], want), (step, b)
        pda.accept(cfg, u32(pick), flags, forced=u32(forced.view(np.uint32)).view(torch.int32))
        assert ctx.status() == 0
        g_fl = host(flags)
        for b in range(B):
            t = int(pick[b])
            s, f = (st[b], 8) if t == NO_TOKEN else accept(orc.dfa, st[b], t, toks, forced[b] >= 0)
            assert g_fl[b] == f, (step, b, t)
            st[b] = s
        done = [b for b in range(B) if g_fl[b] & FLAG_DONE]
        if done:
            cfg.view(torch.int32)[done] = 0
            for b in done:
                st[b] = 0
    assert n_forced > 20


def _frames(v):
    if isinstance(v, list):
        return 2 + max((_frames(x) for x in v), default=0)
    if isinstance(v, dict):
        return 2 + max((1 + _frames(x) for x in v.values()), default=0)
    return 1


@pytest.mark.parametrize("D,steps", [(32, 120), (64, 220)])
def test_deep_stack_texts_are_json_within_the_bound(D, steps):
    """Rows open arrays while they may, then close: the stack reaches its
    bound (up to the largest, CG_PDA_MAX_DEPTH = 64), where the device refuses
    "[" outside strings, and every finished text is JSON whose frame count fits
    the bound."""
    import torch
    V, B = 32000, 64
    toks = vocab("bpe", V)
    ctx, pda = _pda(JSON_NESTED, D, V)
    W = (V + 31) // 32
    rng = np.random.default_rng(32)
    opening = [i for i, t in enumerate(toks) if t and set(t) <= set(b"[")]
    closing = [toks.index(c) for c in (b"]", b"}", b'"')]
    cfg = _fresh(B, D)
    bm = empty((B, W), torch.int32)
    flags = empty((B,), torch.uint8)
    text = [b""] * B
    n_done = max_level = n_full = 0
    phase = [0] * B  # 0 opening, 1 closing
    for step in range(steps):
        pda.fill_bitmask(cfg, bm)
        g_bm, g_cfg = host(bm).view(np.uint32), host(cfg).view(np.uint32)
        pick = np.empty(B, np.uint32)
        for b in range(B):
            ok = np.unpackbits(g_bm[b].view(np.uint8), bitorder="little")[:V].astype(bool)
            assert ok.any(), (step, b)
            if g_cfg[b, 1] >= D - 1:
                if text[b].count(b'"') % 2 == 0:
                    # outside a string "[" opens a value and an array: two more frames
                    assert not ok[toks.index(b"[")], (step, b)
                    n_full += 1
                phase[b] = 1
            pref = [t for t in (opening if phase[b] == 0 else closing) if ok[t]]
            if pref and rng.random() < 0.9:
                pick[b] = pref[rng.integers(len(pref))]
            else:
                ids = np.flatnonzero(ok)
                pick[b] = int(ids[rng.integers(ids.size)])
        pda.accept(cfg, u32(pick), flags)
        assert ctx.status() == 0
        g_fl, g_cfg = host(flags), host(cfg).view(np.uint32)
        for b in range(B):
            assert g_cfg[b, 1] <= D
            text[b] += toks[int(pick[b])]
            max_level = max(max_level, int(g_cfg[b, 1]))
            if g_fl[b] & FLAG_DONE:
                v = json.loads(text[b])
                assert _frames(v) <= D
                n_done += 1
                text[b], phase[b] = b"", 0
        done = [b for b in range(B) if g_fl[b] & FLAG_DONE]
        if done:
            cfg.view(torch.int32)[done] = 0
    assert max_level >= D - 1 and n_full > 0 and n_done > 0


def test_edge_cases():
    import torch
    D, V = 6, 4096
    ctx, pda = _pda(JSON_NESTED, D, V)
    W = (V + 31) // 32
    z = torch.empty((0, D + 2), dtype=torch.int32, device="cuda").view(torch.uint32)
    pda.fill_bitmask(z, torch.empty((0, W), dtype=torch.int32, device="cuda"))
    pda.accept(z, torch.empty((0,), dtype=torch.int32, device="cuda").view(torch.uint32),
               torch.empty((0,), dtype=torch.uint8, device="cuda"))
    assert ctx.status() == 0
    n_states = pda.info()
    assert n_states["n_masks"] >= 1
    # malformed rows: a state past the automaton, a level past the bound
    cfg = u32(np.array([[10**6, 0] + [0] * D, [0, D + 1] + [0] * D, [0xFFFFFFFF, 0] + [0] * D],
                       np.uint32))
    bm = empty((3, W), torch.int32)
    pda.fill_bitmask(cfg, bm)
    assert (host(bm) == 0).all()
    assert ctx.status() == 1  # CG_DEV_BAD_STATE
    # a refused token, a token id past V, a forced token that differs
    toks = vocab("bpe", V)
    close = toks.index(b"]")
    cfg = _fresh(3, D)
    flags = empty((3,), torch.uint8)
    pda.accept(cfg, u32([close, V + 5, ord("[")]), flags,
               forced=u32(np.array([-1, -1, ord("{")], np.int32).view(np.uint32)).view(torch.int32))
    g_fl, g_cfg = host(flags), host(cfg).view(np.uint32)
    assert list(g_fl) == [4, 4, 4] and (g_cfg[:, 0] == 0xFFFFFFFF).all()
    assert ctx.status() in (2, 4, 7)


def test_accept_fill_equals_the_two_calls():
    """cg_pda_accept_fill (accept of one step and fill of the next in one
    launch) gives the configurations, flags, counts and masks of cg_pda_accept
    followed by cg_pda_fill_bitmask, and the masks are the oracle's."""
    import torch
    D, V, B, steps = 8, 32000, 96, 30
    toks = vocab("bpe", V)
    orc = OracleRows(JSON_NESTED, D, toks)
    ctx, pda = _pda(JSON_NESTED, D, V)
    opens = np.array([t.count(b"[") + t.count(b"{") for t in toks])
    rng = np.random.default_rng(77)
    W = (V + 31) // 32
    cfg_a, cfg_b = _fresh(B, D), _fresh(B, D)
    bm_a, bm_b = empty((B, W), torch.int32), empty((B, W), torch.int32)
    fl_a, fl_b = empty((B,), torch.uint8), empty((B,), torch.uint8)
    cnt_a = torch.zeros((B,), dtype=torch.int32, device="cuda").view(torch.uint32)
    cnt_b = torch.zeros((B,), dtype=torch.int32, device="cuda").view(torch.uint32)
    st = [0] * B
    pda.fill_bitmask(cfg_b, bm_b)
    for step in range(steps):
        pda.fill_bitmask(cfg_a, bm_a)
        g_a = host(bm_a).view(np.uint32)
        assert np.array_equal(g_a, host(bm_b).view(np.uint32)), step
        pick = np.empty(B, np.uint32)
        for b in range(B):
            want = orc.mask(st[b])
            assert np.array_equal(g_a[b], want), (step, b)
            pick[b] = _pick(rng, want, V, opens, 0.3)
        toks_d = u32(pick)
        pda.accept(cfg_a, toks_d, fl_a, counts=cnt_a, max_tokens=12)
        pda.accept_fill(cfg_b, toks_d, fl_b, bm_b, counts=cnt_b, max_tokens=12)
        assert ctx.status() == 0
        assert np.array_equal(host(fl_a), host(fl_b)), step
        assert np.array_equal(host(cfg_a), host(cfg_b)), step
        assert np.array_equal(host(cnt_a), host(cnt_b)), step
        g_fl = host(fl_a)
        for b in range(B):
            t = int(pick[b])
            s, f = (st[b], 8) if t == NO_TOKEN else accept(orc.dfa, st[b], t, toks, False)
            st[b] = 0 if g_fl[b] & (FLAG_DONE | 16) else s


@pytest.mark.parametrize("dtype,V,B,D", [("bf16", 128256, 256, 32), ("f32", 32000, 64, 8), ("bf16", 4013, 32, 8)])
def test_pda_step_equals_the_three_calls(dtype, V, B, D):
    """cg_pda_step (one fused kernel per row on the bf16 top-p path, else the
    three calls inside the library) gives the ids, flags, configurations,
    counts and masks of cg_pda_fill_bitmask, cg_mask_and_sample and
    cg_pda_accept, step after step; the masks are the oracle's at D = 8."""
    import torch
    temp, top_p, seed, steps = 0.7, 0.9, 5, 12
    toks = vocab("bpe", V)
    ctx, pda = _pda(JSON_NESTED, D, V)
    orc = OracleRows(JSON_NESTED, D, toks) if D <= 8 else None
    W = (V + 31) // 32
    cfg_a, cfg_b = _fresh(B, D), _fresh(B, D)
    bm_a, bm_b = empty((B, W), torch.int32), empty((B, W), torch.int32)
    tok_a, tok_b = empty((B,), torch.int32), empty((B,), torch.int32)
    fl_a, fl_b = empty((B,), torch.uint8), empty((B,), torch.uint8)
    cnt_a = torch.zeros((B,), dtype=torch.int32, device="cuda").view(torch.uint32)
    cnt_b = torch.zeros((B,), dtype=torch.int32, device="cuda").view(torch.uint32)
    st = [0] * B
    for step in range(steps):
        vals, x = logits_rows(V, range(B), step, 4, 2.0, 4.0, 0.05, dtype)
        pda.fill_bitmask(cfg_a, bm_a)
        ctx.mask_and_sample(x, bm_a, temp, top_p, seed, step, tok_a)
        pda.accept(cfg_a, tok_a.view(torch.uint32), fl_a, counts=cnt_a, max_tokens=20)
        pda.step(cfg_b, x, temp, top_p, seed, step, tok_b.view(torch.uint32), fl_b, counts=cnt_b, max_tokens=20,
                 bitmask=bm_b)
        assert ctx.status() == 0
        g_bm = host(bm_a).view(np.uint32)
        assert np.array_equal(g_bm, host(bm_b).view(np.uint32)), step
        assert np.array_equal(host(tok_a), host(tok_b)), step
        assert np.array_equal(host(fl_a), host(fl_b)), step
        assert np.array_equal(host(cfg_a), host(cfg_b)), step
        assert np.array_equal(host(cnt_a), host(cnt_b)), step
        if orc is not None:
            g_tok, g_fl = host(tok_a).view(np.uint32), host(fl_a)
            for b in range(B):
                assert np.array_equal(g_bm[b], orc.mask(st[b])), (step, b)
                t = int(g_tok[b])
                s, f = (st[b], 8) if t == NO_TOKEN else accept(orc.dfa, st[b], t, toks, False)
                st[b] = 0 if g_fl[b] & (FLAG_DONE | 16) else s


def test_pda_step_with_forced_rows_equals_the_three_calls():
    """The fused step's forced rows: where the oracle's state continues only
    with injected bytes the row gets a forced single-byte token; cg_pda_step
    and the three calls give the same ids, flags, configurations and masks,
    and the flags are the oracle's."""
    import torch
    D, V, B, steps = 4, 4096, 64, 40
    temp, top_p, seed = 0.7, 0.9, 9
    toks = vocab("bpe", V)
    orc = OracleRows(MIXED, D, toks)
    ctx, pda = _pda(MIXED, D, V)
    single = {t[0]: i for i, t in enumerate(toks) if len(t) == 1}
    rng = np.random.default_rng(21)
    W = (V + 31) // 32
    cfg_a, cfg_b = _fresh(B, D), _fresh(B, D)
    bm_a, bm_b = empty((B, W), torch.int32), empty((B, W), torch.int32)
    tok_a, tok_b = empty((B,), torch.int32), empty((B,), torch.int32)
    fl_a, fl_b = empty((B,), torch.uint8), empty((B,), torch.uint8)
    st = [0] * B
    n_forced = 0
    for step in range(steps):
        forced = np.full(B, -1, np.int32)
        for b in range(B):
            s = st[b]
            if s != DEAD and (orc.dfa.next[s, :256] < 0).all() and (orc.dfa.next[s, 256:] >= 0).any():
                live = np.flatnonzero(orc.dfa.next[s, 256:] >= 0)
                forced[b] = single[int(live[rng.integers(live.size)])]
        n_forced += int((forced >= 0).sum())
        f_d = u32(forced.view(np.uint32)).view(torch.int32)
        vals, x = logits_rows(V, range(B), step, 6, 2.0, 4.0, 0.05, "bf16")
        pda.fill_bitmask(cfg_a, bm_a, forced=f_d)
        ctx.mask_and_sample(x, bm_a, temp, top_p, seed, step, tok_a)
        pda.accept(cfg_a, tok_a.view(torch.uint32), fl_a, forced=f_d)
        pda.step(cfg_b, x, temp, top_p, seed, step, tok_b.view(torch.uint32), fl_b, forced=f_d, bitmask=bm_b)
        assert ctx.status() == 0
        assert np.array_equal(host(bm_a), host(bm_b)), step
        assert np.array_equal(host(tok_a), host(tok_b)), step
        assert np.array_equal(host(fl_a), host(fl_b)), step
        assert np.array_equal(host(cfg_a), host(cfg_b)), step
        g_tok, g_fl = host(tok_a).view(np.uint32), host(fl_a)
        for b in range(B):
            t = int(g_tok[b])
            s, f = (st[b], 8) if t == NO_TOKEN else accept(orc.dfa, st[b], t, toks, forced[b] >= 0)
            assert g_fl[b] == f, (step, b, t)
            st[b] = s
        done = [b for b in range(B) if g_fl[b] & FLAG_DONE]
        if done:
            cfg_a.view(torch.int32)[done] = 0
            cfg_b.view(torch.int32)[done] = 0
            for b in done:
                st[b] = 0
    assert n_forced > 20


TREE = r'''
root ::= node "."
node ::= "(" node "," node ")" | [a-c]+
'''
ROOTED = r'''
root ::= "[" ( root ( ";" root )* )? "]" | "x"
'''


@pytest.mark.parametrize("source,D", [(TREE, 3), (TREE, 6), (ROOTED, 3), (ROOTED, 5)])
def test_other_grammar_shapes_match_the_oracle(source, D):
    """Random walks on a grammar whose open nodes need headroom to complete
    (a node opened deep must still fit its second child) and on one whose
    start rule is itself recursive (the base frame and called frames share the
    rule): masks and flags bit for bit against the oracle."""
    import torch
    V, B, steps = 4096, 96, 30
    toks = vocab("bpe", V)
    orc = OracleRows(source, D, toks)
    ctx, pda = _pda(source, D, V)
    rng = np.random.default_rng(D + len(source))
    W = (V + 31) // 32
    cfg = _fresh(B, D)
    bm = empty((B, W), torch.int32)
    flags = empty((B,), torch.uint8)
    opens = np.array([t.count(b"(") + t.count(b"[") for t in toks])
    st = [0] * B
    max_level = 0
    for step in range(steps):
        pda.fill_bitmask(cfg, bm)
        g_bm = host(bm).view(np.uint32)
        pick = np.empty(B, np.uint32)
        for b in range(B):
            want = orc.mask(st[b])
            assert np.array_equal(g_bm[b], want), (step, b)
            pick[b] = _pick(rng, want, V, opens, 0.4)
        pda.accept(cfg, u32(pick), flags)
        assert ctx.status() == 0
        g_fl, g_cfg = host(flags), host(cfg).view(np.uint32)
        for b in range(B):
            t = int(pick[b])
            s, f = (st[b], 8) if t == NO_TOKEN else accept(orc.dfa, st[b], t, toks, False)
            assert g_fl[b] == f, (step, b, t)
            st[b] = s
            max_level = max(max_level, int(g_cfg[b, 1]))
        done = [b for b in range(B) if g_fl[b] & (FLAG_DONE | 8)]
        if done:
            cfg.view(torch.int32)[done] = 0
            for b in done:
                st[b] = 0
    assert max_level >= min(D, 3)


def test_fused_pda_step_matches_the_oracle():
    """cg_pda_step (mask, sample and accept in one fused kernel per row)
    checked against the oracle directly, row by row and step by step: the
    bitmask it writes, the sampled id and the accept flags."""
    import torch
    D, V, B, steps = 8, 32000, 64, 16
    temp, top_p, seed = 0.7, 0.9, 13
    toks = vocab("bpe", V)
    orc = OracleRows(JSON_NESTED, D, toks)
    ctx, pda = _pda(JSON_NESTED, D, V)
    W = (V + 31) // 32
    cfg = _fresh(B, D)
    bm = empty((B, W), torch.int32)
    tok = empty((B,), torch.int32)
    flags = empty((B,), torch.uint8)
    st = [0] * B
    for step in range(steps):
        vals, x = logits_rows(V, range(B), step, 5, 2.0, 4.0, 0.05, "bf16")
        pda.step(cfg, x, temp, top_p, seed, step, tok, flags, bitmask=bm)
        assert ctx.status() == 0
        g_tok, g_bm, g_fl = host(tok).view(np.uint32), host(bm).view(np.uint32), host(flags)
        for b in range(B):
            want = orc.mask(st[b])
            assert np.array_equal(g_bm[b], want), (step, b)
            allowed = np.unpackbits(want.view(np.uint8), bitorder="little")[:V].astype(bool)
            res = sample_row(vals[b], allowed, temp, top_p, seed, b, step)
            assert same_token(int(g_tok[b]), res), (step, b)
            s, f = accept(orc.dfa, st[b], int(g_tok[b]), toks, False) if g_tok[b] != NO_TOKEN else (st[b], 8)
            assert g_fl[b] == f, (step, b)
            st[b] = s
        done = [b for b in range(B) if g_fl[b] & FLAG_DONE]
        if done:  # finished rows start again
            cfg.view(torch.int32)[done] = 0
            for b in done:
                st[b] = 0
