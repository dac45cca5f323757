"""Tokens of 31, 32 and more bytes through both accept paths.

The accept reads a token's bytes from a 32-byte record (length byte plus up to
31 bytes) and falls back to the offset table for longer tokens; the fused step
also reads transitions from a window of the table in shared memory.  The
seeded vocabularies have no token that long, so this test splices long tokens
into one and checks next states and flags against the oracle's walk
(usetacet.com/docs/grammar, "Constrained decoding": a token is accepted when
every one of its bytes has a transition).
"""

import numpy as np
import pytest

from oracle.dfa import DEAD
from oracle.step import accept, token_allowed
from tests.gpu_helpers import empty, host, product_grammar, u32
from tests.oracle_cache import oracle_dfa, vocab

pytestmark = pytest.mark.gpu

V = 3000
LONG = [b"a" * 30, b"a" * 31, b"a" * 32, b"a" * 33, b"b" * 47, b" " * 40, b"Zurich" * 6,
        b"1234567890" * 4, b"x" * 31 + b'"', b"q" * 64]


def _vocab():
    toks = list(vocab("bpe", V))
    have = set(toks)
    base = V - len(LONG)
    for i, t in enumerate(LONG):
        assert t not in have
        toks[base + i] = t
    return toks, list(range(base, V))


def _cases(dfa, toks, long_ids, rng, n):
    """(state, token) pairs: each long token from states that accept it and
    from states that reject it."""
    live = np.flatnonzero([dfa.next[s].max() >= 0 for s in range(dfa.n_states)])
    order = rng.permutation(live)
    pairs = []
    for tid in long_ids:
        ok = [int(s) for s in order[:4000] if token_allowed(dfa, int(s), toks[tid])][: n // 2]
        bad = [int(s) for s in order[:64] if not token_allowed(dfa, int(s), toks[tid])][:2]
        pairs += [(s, tid) for s in ok + bad]
    return pairs


def test_accept_long_tokens():
    import torch
    from grammar_constrained_decoding_gb300 import Ctx, Vocab
    toks, long_ids = _vocab()
    dfa = oracle_dfa("booking")
    rng = np.random.default_rng(21)
    pairs = _cases(dfa, toks, long_ids, rng, 8)
    assert sum(token_allowed(dfa, s, toks[t]) for s, t in pairs) >= 10, "no accepting state for the long tokens"
    ctx = Ctx([product_grammar("booking")], Vocab(toks))
    B = len(pairs)
    states = np.array([p[0] for p in pairs], np.uint32)
    tok = np.array([p[1] for p in pairs], np.uint32)
    out_s, out_f = empty((B,), torch.int32), empty((B,), torch.uint8)
    ctx.accept(u32(states), u32(tok), out_s, out_f)
    ctx.status()
    gs, gf = host(out_s).view(np.uint32), host(out_f)
    for b, (s, t) in enumerate(pairs):
        ns, fl = accept(dfa, s, t, toks, False)
        assert gs[b] == (0xFFFFFFFF if ns == DEAD else ns) and gf[b] == fl, (len(toks[t]), s, gs[b], ns)


def test_fused_step_long_tokens():
    """The fused step samples a long token (its logit far above the rest, a
    small nucleus) and must land where the oracle's walk does."""
    import torch
    from grammar_constrained_decoding_gb300 import Ctx, Vocab
    toks, long_ids = _vocab()
    dfa = oracle_dfa("booking")
    rng = np.random.default_rng(22)
    pairs = [(s, t) for s, t in _cases(dfa, toks, long_ids, rng, 6) if token_allowed(dfa, s, toks[t])]
    assert len(pairs) >= 10
    ctx = Ctx([product_grammar("booking")], Vocab(toks))
    B = len(pairs)
    x = rng.normal(0.0, 1.0, (B, V)).astype(np.float32)
    for b, (_, t) in enumerate(pairs):
        x[b, t] = 60.0
    xt = torch.from_numpy(x).to(torch.bfloat16).cuda()
    states = u32(np.array([p[0] for p in pairs], np.uint32))
    tok = empty((B,), torch.int32)
    ns_t, fl_t = empty((B,), torch.int32).view(torch.uint32), empty((B,), torch.uint8)
    ctx.step(states, xt, 0.7, 0.5, 1, 0, tok, ns_t, fl_t)
    assert ctx.status() == 0
    got_tok, got_s, got_f = host(tok).view(np.uint32), host(ns_t).view(np.uint32), host(fl_t)
    for b, (s, t) in enumerate(pairs):
        assert got_tok[b] == t, (b, got_tok[b], t)
        ns, fl = accept(dfa, s, t, toks, False)
        assert got_s[b] == ns and got_f[b] == fl, (len(toks[t]), s, got_s[b], ns)
