"""cg_accept_many against the oracle's accept_many, row by row.

Drafts of up to K tokens are drawn from seeded random live states: mostly
tokens the grammar allows at that point, sometimes a random token (which may
be refused), and, where a position's state continues only with injected bytes,
a host pin (right or, sometimes, wrong).  Accepted counts, final states, flags,
token counts and the per-position state path must be bit-exact
(labs.miniml.ai "Evaluator aware decoding", "Where XGrammar-2 could take this").
"""

import numpy as np
import pytest

from oracle.dfa import DEAD
from oracle.step import VocabMatrix, accept, accept_many, token_allowed, token_mask
from tests.gpu_helpers import empty, host, make_ctx, u16, u32
from tests.oracle_cache import oracle_dfa, vocab

pytestmark = pytest.mark.gpu


def _drafts(dfas, toks, B, K, rng, gid):
    V = len(toks)
    vm = VocabMatrix(toks)
    states = np.zeros(B, np.int64)
    draft = np.zeros((B, K), np.uint32)
    dlen = np.zeros(B, np.uint32)
    forced = np.full((B, K), -1, np.int32)
    for b in range(B):
        d = dfas[gid[b]]
        live = np.flatnonzero(d.next.max(axis=1) >= 0)
        s = int(live[rng.integers(len(live))])
        states[b] = s
        n = int(rng.integers(0, K + 1))
        st = s
        for j in range(n):
            if st >= 0 and d.forced_only()[st]:
                syms = np.flatnonzero(d.next[st, 256:] >= 0)
                forced[b, j] = int(syms[rng.integers(len(syms))])
                t = forced[b, j] if rng.random() < 0.9 else int(rng.integers(V))
            else:
                t = int(rng.integers(V))
                if st >= 0 and rng.random() < 0.9:
                    for _ in range(20):
                        c = int(rng.integers(V))
                        if token_allowed(d, st, toks[c]):
                            t = c
                            break
                    else:
                        allowed = np.flatnonzero(token_mask(d, vm, st))
                        if allowed.size:
                            t = int(allowed[rng.integers(allowed.size)])
            draft[b, j] = t
            if st >= 0:
                st, _ = accept(d, st, int(t), toks, forced[b, j] >= 0)
        dlen[b] = n
    return states, draft, dlen, forced


@pytest.mark.parametrize("names,V,B,K,use_counts", [
    (("calc_eval", "json_eval", "booking_200"), 2999, 300, 6, False),
    (("calc_eval", "json_eval", "booking_200"), 2999, 300, 6, True),
    (("booking",), 128256, 256, 8, True),
])
def test_accept_many_matches_oracle(names, V, B, K, use_counts):
    import torch
    ctx = make_ctx(names, "bpe", V)
    toks = vocab("bpe", V)
    dfas = [oracle_dfa(n) for n in names]
    rng = np.random.default_rng(V + B + K + use_counts)
    gid = (np.arange(B) % len(names)).astype(np.uint16)
    states, draft, dlen, forced = _drafts(dfas, toks, B, K, rng, gid)
    states[5] = -1                                     # a dead row
    dlen[6] = 0                                        # an empty draft
    counts = rng.integers(0, 9, B).astype(np.uint32)
    cap = 10
    out_s = empty((B,), torch.int32).view(torch.uint32)
    out_n = empty((B,), torch.int32).view(torch.uint32)
    out_f = empty((B,), torch.uint8)
    path = empty((B, K + 1), torch.int32).view(torch.uint32)
    cnt = u32(counts) if use_counts else None
    ctx.accept_many(u32(np.where(states < 0, 0xFFFFFFFF, states)), u32(draft), u32(dlen), out_s, out_n, out_f,
                    gid=u16(gid) if len(names) > 1 else None, forced=torch.from_numpy(forced).cuda(),
                    counts=cnt, max_tokens=cap, path=path)
    assert ctx.status() == 0
    g_s, g_n, g_f, g_p = host(out_s), host(out_n), host(out_f), host(path)
    g_c = host(cnt) if use_counts else None
    cut = 0
    for b in range(B):
        n = int(dlen[b])
        r = accept_many(dfas[gid[b]], int(states[b]), [int(t) for t in draft[b, :n]], toks,
                        [int(f) for f in forced[b, :n]], int(counts[b]) if use_counts else None, cap)
        want_s = 0xFFFFFFFF if r.state == DEAD else r.state
        assert (g_n[b], g_s[b], g_f[b]) == (r.n, want_s, r.flags), (b, r)
        want_p = [0xFFFFFFFF if p == DEAD else p for p in r.path] + [0xFFFFFFFF] * (K - r.n)
        assert list(g_p[b]) == want_p, b
        if use_counts:
            assert g_c[b] == r.count, b
        cut += bool(r.flags & 32)
    assert 0 < cut < B    # both outcomes occur
