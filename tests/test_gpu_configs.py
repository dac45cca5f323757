"""Every workload configuration at its full batch and vocabulary size, through
cg_step (the call bench.py times), checked against the oracle.

Per step, on every row: the sampled id is allowed by the row's bitmask (a
forced row carries exactly its forced id; an empty mask gives no token), and
the next state and flags are the oracle's walk of that id
(usetacet.com/docs/grammar, "Constrained decoding": a token is allowed when
each of its bytes has a transition; labs.miniml.ai "Evaluator aware decoding":
the state advances over injected tokens too).  On 8 sampled rows per step: the
bitmask bit for bit against the oracle's scalar mask, and the id against the
oracle's sampler on the same logits (ids may differ only where the oracle
reports its top-two Gumbel scores, or the top-p threshold, within 1e-5).
Rows start in seeded random live states (half of them in the start state when
the configuration does not draw start states), so forced-only states and
their forced ids occur at every size.
"""

import zlib

import numpy as np
import pytest

from oracle.dfa import DEAD
from oracle.step import NO_TOKEN, VocabMatrix, accept, onehot_mask, sample_row, token_mask
from tests.gpu_helpers import empty, host, product_grammar, same_token, u16, u32
from tests.oracle_cache import oracle_dfa, vocab
from workloads import CONFIGS, make_logits

pytestmark = pytest.mark.gpu

STEPS = 3
SAMPLED = 8


def _start(cfg, dfas, rng):
    n_g = len(cfg.grammars)
    live = [np.flatnonzero(d.next.max(axis=1) >= 0) for d in dfas]
    states = np.zeros(cfg.B, np.uint32)
    for b in range(cfg.B):
        if cfg.random_start or b % 2:
            states[b] = live[b % n_g][rng.integers(len(live[b % n_g]))]
    return states


def _forced(cfg, dfas, states):
    """A legal injected byte for rows in forced-only states (single-byte token
    ids equal the byte), -1 elsewhere."""
    n_g = len(cfg.grammars)
    forced = np.full(cfg.B, -1, np.int32)
    for b in range(cfg.B):
        d = dfas[b % n_g]
        s = int(states[b])
        if s != 0xFFFFFFFF and s < d.n_states and d.forced_only()[s]:
            syms = np.flatnonzero(d.next[s, 256:] >= 0)
            if syms.size:
                forced[b] = int(syms[0])
    return forced


@pytest.mark.parametrize("name", list(CONFIGS))
def test_config_full_size(name):
    import torch
    from grammar_constrained_decoding_gb300 import Ctx, Vocab
    cfg = CONFIGS[name]
    V, B, n_g = cfg.V, cfg.B, len(cfg.grammars)
    W = (V + 31) // 32
    toks = vocab(cfg.vocab_kind, V, cfg.vocab_seed)
    vm = VocabMatrix(toks)
    dfas = [oracle_dfa(n) for n in cfg.grammars]
    ctx = Ctx([product_grammar(n) for n in cfg.grammars], Vocab(toks))
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    gid_np = (np.arange(B) % n_g).astype(np.uint16)
    gid = u16(gid_np) if n_g > 1 else None
    states = _start(cfg, dfas, rng)
    sampled = np.unique(np.linspace(0, B - 1, SAMPLED).astype(int))
    forced_rows = 0
    for step in range(STEPS):
        vals, raw = make_logits(V, range(B), step, cfg.logit_seed, cfg.sigma, cfg.boost, cfg.boost_frac, cfg.dtype)
        if cfg.dtype == "bf16":
            x = torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
        else:
            x = torch.from_numpy(raw).cuda()
        forced = _forced(cfg, dfas, states)
        forced_rows += int((forced >= 0).sum())
        bm = empty((B, W), torch.int32)
        tok = empty((B,), torch.int32)
        ns, fl = empty((B,), torch.int32).view(torch.uint32), empty((B,), torch.uint8)
        ctx.step(u32(states), x, cfg.temp, cfg.top_p, cfg.sample_seed, step, tok, ns, fl, gid=gid,
                 forced=torch.from_numpy(forced).cuda(), bitmask=bm)
        assert ctx.status() == 0, step
        g_bm = host(bm).view(np.uint32)
        g_tok = host(tok).view(np.uint32)
        g_ns, g_fl = host(ns).view(np.uint32), host(fl)
        for b in range(B):
            d, s, t = dfas[b % n_g], int(states[b]), int(g_tok[b])
            if forced[b] >= 0:
                assert t == forced[b], (step, b, t, forced[b])
            if t == NO_TOKEN:
                assert not g_bm[b].any(), (step, b)
            else:
                assert (g_bm[b, t >> 5] >> (t & 31)) & 1, (step, b, t)
            want_s, want_f = accept(d, -1 if s == 0xFFFFFFFF else s, t, toks, forced[b] >= 0)
            assert g_ns[b] == (0xFFFFFFFF if want_s == DEAD else want_s) and g_fl[b] == want_f, (step, b, s, t)
        for b in sampled:
            d, s = dfas[b % n_g], int(states[b])
            if forced[b] >= 0:
                allowed = onehot_mask(V, int(forced[b]))
            elif s == 0xFFFFFFFF:
                allowed = np.zeros(V, bool)
            else:
                allowed = token_mask(d, vm, s)
            bits = np.zeros(W * 32, bool)
            bits[:V] = allowed
            want_bm = (bits.reshape(W, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(1)
            assert np.array_equal(g_bm[b], want_bm.astype(np.uint32)), (step, b, s)
            res = sample_row(vals[b].astype(np.float64), allowed, cfg.temp, cfg.top_p, cfg.sample_seed, int(b),
                             step)
            assert same_token(int(g_tok[b]), res), (step, b, int(g_tok[b]), res.tok, res.gap, res.margin)
        states = g_ns.copy()
    if name == "mixed_eval_152k":
        assert forced_rows > 0, "no forced-only state was drawn"


@pytest.mark.parametrize("name", ["booking_128k", "reasoning_152k"])
def test_config_every_row(name):
    """One cg_step at full size with every row checked against the oracle:
    its bitmask bit for bit (the oracle's scalar mask, computed once per
    distinct state), its id against the oracle's sampler on the same logits,
    and its next state and flags against the oracle's accept."""
    import torch
    from grammar_constrained_decoding_gb300 import Ctx, Vocab
    cfg = CONFIGS[name]
    V, B, n_g = cfg.V, cfg.B, len(cfg.grammars)
    W = (V + 31) // 32
    toks = vocab(cfg.vocab_kind, V, cfg.vocab_seed)
    vm = VocabMatrix(toks)
    dfas = [oracle_dfa(n) for n in cfg.grammars]
    ctx = Ctx([product_grammar(n) for n in cfg.grammars], Vocab(toks))
    rng = np.random.default_rng(zlib.crc32(name.encode()) ^ 0x5A5A)
    states = _start(cfg, dfas, rng)
    step = 1
    vals, raw = make_logits(V, range(B), step, cfg.logit_seed, cfg.sigma, cfg.boost, cfg.boost_frac, cfg.dtype)
    x = torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
    forced = _forced(cfg, dfas, states)
    bm = empty((B, W), torch.int32)
    tok = empty((B,), torch.int32)
    ns, fl = empty((B,), torch.int32).view(torch.uint32), empty((B,), torch.uint8)
    ctx.step(u32(states), x, cfg.temp, cfg.top_p, cfg.sample_seed, step, tok, ns, fl,
             forced=torch.from_numpy(forced).cuda(), bitmask=bm)
    assert ctx.status() == 0
    g_bm, g_tok = host(bm).view(np.uint32), host(tok).view(np.uint32)
    g_ns, g_fl = host(ns).view(np.uint32), host(fl)
    masks = {}
    for b in range(B):
        d, s, t = dfas[b % n_g], int(states[b]), int(g_tok[b])
        if forced[b] >= 0:
            allowed = onehot_mask(V, int(forced[b]))
        elif s == 0xFFFFFFFF:
            allowed = np.zeros(V, bool)
        else:
            if (b % n_g, s) not in masks:
                masks[(b % n_g, s)] = token_mask(d, vm, s)
            allowed = masks[(b % n_g, s)]
        bits = np.zeros(W * 32, bool)
        bits[:V] = allowed
        want_bm = (bits.reshape(W, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(1)
        assert np.array_equal(g_bm[b], want_bm.astype(np.uint32)), (b, s)
        res = sample_row(vals[b].astype(np.float64), allowed, cfg.temp, cfg.top_p, cfg.sample_seed, b, step)
        assert same_token(t, res), (b, t, res.tok, res.gap, res.margin)
        want_s, want_f = accept(d, -1 if s == 0xFFFFFFFF else s, t, toks, forced[b] >= 0)
        assert g_ns[b] == (0xFFFFFFFF if want_s == DEAD else want_s) and g_fl[b] == want_f, (b, s, t)
