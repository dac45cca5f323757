"""cg_step (fill_bitmask + mask_and_sample + accept in one call) gives the
results of the three calls bit for bit: tokens, next states, flags, counts,
the bitmask it can write out, and the device status.  The fused one-kernel
path (bf16, temp > 0, top_p < 1) and the unfused fallback are both covered,
over multi-step trajectories with random live start states, token caps and
forced tokens (valid ones in forced-only states, and invalid ones).
"""

import zlib

import numpy as np
import pytest

from tests.gpu_helpers import empty, host, make_ctx, product_grammar, u16, u32
from workloads import make_logits

pytestmark = pytest.mark.gpu

CG_STATE_FORCED_ONLY = 4
_EXPORTS = {}


def _export(name):
    if name not in _EXPORTS:
        _EXPORTS[name] = product_grammar(name).export()
    return _EXPORTS[name]


def _start_states(names, B, rng):
    states = []
    for b in range(B):
        live = product_grammar(names[b % len(names)]).live_states()
        states.append(int(live[rng.integers(len(live))]))
    return np.array(states, dtype=np.uint32)


def _forced_for(names, states, rng, share):
    """Forced ids: for rows in a forced-only state a token the state accepts as
    injected (single-byte ids are the bytes); for a share of other rows an
    arbitrary id (rejected by both paths alike)."""
    forced = np.full(len(states), -1, dtype=np.int32)
    for b, s in enumerate(states):
        nxt, flags = _export(names[b % len(names)])
        if s < len(flags) and flags[s] & CG_STATE_FORCED_ONLY:
            ok = [c for c in range(256) if nxt[s, 256 + c] >= 0]
            if ok:
                forced[b] = ok[rng.integers(len(ok))]
        elif rng.random() < share:
            forced[b] = int(rng.integers(0, 4000))
    return forced


def _logits(V, B, step, dtype):
    import torch
    vals, raw = make_logits(V, list(range(B)), step, 1234, 2.0, 4.0, 0.05, dtype)
    if dtype == "bf16":
        return torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(raw).cuda()


@pytest.mark.parametrize("names,temp,top_p,dtype", [
    (("booking",), 0.7, 0.9, "bf16"),                       # fused
    (("calc_eval", "json_eval", "booking"), 0.7, 0.9, "bf16"),  # fused, several grammars, forced steps
    (("booking",), 0.7, 1.0, "bf16"),                       # unfused: full softmax
    (("calc_eval", "booking"), 0.0, 1.0, "bf16"),           # unfused: greedy
    (("calc_call",), 0.7, 0.9, "f32"),                      # unfused: f32 logits
])
def test_step_matches_three_calls(names, temp, top_p, dtype):
    import torch
    V, B, steps, cap = 128256, 24, 10, 6
    rng = np.random.default_rng(zlib.crc32(repr((names, temp, top_p, dtype)).encode()))
    ctx_a = make_ctx(names, "bpe", V)
    ctx_b = make_ctx(names, "bpe", V)
    W = (V + 31) // 32
    gid = u16(np.arange(B) % len(names)) if len(names) > 1 else None
    s0 = _start_states(names, B, rng)
    st_a, st_b = u32(s0), u32(s0)
    cnt_a, cnt_b = u32(np.zeros(B)), u32(np.zeros(B))
    for step in range(steps):
        x = _logits(V, B, step, dtype)
        forced_np = _forced_for(names, host(st_a).view(np.uint32), rng, 0.1 if step == 3 else 0.0)
        forced = torch.from_numpy(forced_np).cuda()
        bm_a, bm_b = empty((B, W), torch.int32), empty((B, W), torch.int32)
        tok_a, tok_b = empty((B,), torch.int32), empty((B,), torch.int32)
        ns_a, ns_b = empty((B,), torch.int32).view(torch.uint32), empty((B,), torch.int32).view(torch.uint32)
        fl_a, fl_b = empty((B,), torch.uint8), empty((B,), torch.uint8)
        ctx_a.fill_bitmask(st_a, bm_a, gid=gid, forced=forced)
        ctx_a.mask_and_sample(x, bm_a, temp, top_p, 77, step, tok_a)
        ctx_a.accept(st_a, tok_a.view(torch.uint32), ns_a, fl_a, gid=gid, forced=forced, counts=cnt_a,
                     max_tokens=cap)
        code_a = ctx_a.status()
        ctx_b.step(st_b, x, temp, top_p, 77, step, tok_b, ns_b, fl_b, gid=gid, forced=forced, counts=cnt_b,
                   max_tokens=cap, bitmask=bm_b)
        code_b = ctx_b.status()
        assert code_a == code_b, (step, code_a, code_b)
        assert np.array_equal(host(bm_a), host(bm_b)), step
        assert np.array_equal(host(tok_a), host(tok_b)), step
        assert np.array_equal(host(ns_a), host(ns_b)), step
        assert np.array_equal(host(fl_a), host(fl_b)), step
        assert np.array_equal(host(cnt_a), host(cnt_b)), step
        st_a, st_b = ns_a, ns_b


def test_step_without_bitmask_output():
    """With no bitmask buffer the fused path keeps the mask on chip and the
    unfused path uses the context's own buffer; results are unchanged."""
    import torch
    names, V, B = ("booking",), 128256, 16
    ctx_a, ctx_b = make_ctx(names, "bpe", V), make_ctx(names, "bpe", V)
    rng = np.random.default_rng(5)
    s0 = _start_states(names, B, rng)
    for temp, top_p in ((0.7, 0.9), (0.0, 1.0)):
        x = _logits(V, B, 1, "bf16")
        outs = []
        for ctx, bm in ((ctx_a, empty((B, (V + 31) // 32), torch.int32)), (ctx_b, None)):
            tok, ns = empty((B,), torch.int32), empty((B,), torch.int32).view(torch.uint32)
            fl = empty((B,), torch.uint8)
            ctx.step(u32(s0), x, temp, top_p, 3, 1, tok, ns, fl, bitmask=bm)
            assert ctx.status() == 0
            outs.append((host(tok), host(ns), host(fl)))
        for a, b in zip(*outs):
            assert np.array_equal(a, b)


@pytest.mark.parametrize("temp,top_p", [(0.7, 0.9), (0.0, 1.0)])
def test_step_host_matches_step(temp, top_p):
    """cg_step_host (logits in page-locked host memory, ids copied back, two
    device buffers alternating) gives cg_step's results; four calls are queued
    before the first sync, so copies overlap the previous steps' kernels."""
    import torch
    names, V, B, steps = ("calc_eval", "booking"), 128256, 40, 4
    ctx_a, ctx_b = make_ctx(names, "bpe", V), make_ctx(names, "bpe", V)
    gid = u16(np.arange(B) % len(names))
    s0 = _start_states(names, B, np.random.default_rng(8))
    st_a, st_b = u32(s0), u32(s0)
    cnt_a, cnt_b = u32(np.zeros(B)), u32(np.zeros(B))
    xs = [_logits(V, B, k, "bf16") for k in range(steps)]
    hx = [x.cpu().pin_memory() for x in xs]
    htok = [torch.full((B,), -1, dtype=torch.int32).pin_memory() for _ in range(steps)]
    ns_b = [empty((B,), torch.int32).view(torch.uint32) for _ in range(steps)]
    fl_b = [empty((B,), torch.uint8) for _ in range(steps)]
    want = []
    for k in range(steps):
        tok = empty((B,), torch.int32)
        ns, fl = empty((B,), torch.int32).view(torch.uint32), empty((B,), torch.uint8)
        ctx_a.step(st_a, xs[k], temp, top_p, 5, k, tok, ns, fl, gid=gid, counts=cnt_a, max_tokens=6)
        want.append((host(tok), host(ns), host(fl)))
        st_a = ns
    for k in range(steps):
        ctx_b.step_host(st_b, hx[k], temp, top_p, 5, k, htok[k], ns_b[k], fl_b[k], gid=gid, counts=cnt_b,
                        max_tokens=6)
        st_b = ns_b[k]
    ctx_b.sync()
    assert ctx_a.status() == 0 and ctx_b.status() == 0
    for k in range(steps):
        assert np.array_equal(htok[k].numpy(), want[k][0]), k
        assert np.array_equal(host(ns_b[k]), want[k][1]), k
        assert np.array_equal(host(fl_b[k]), want[k][2]), k


@pytest.mark.parametrize("temp,top_p", [(0.7, 0.9), (0.7, 1.0)])
def test_step_host_matches_the_oracle(temp, top_p):
    """cg_step_host checked against the oracle directly: every row's id (on
    the same logits and the oracle's mask of its state), next state and flags,
    over three steps from random live states."""
    import torch
    from oracle.dfa import DEAD
    from oracle.step import VocabMatrix, accept, sample_row, token_mask
    from tests.gpu_helpers import same_token
    from tests.oracle_cache import oracle_dfa, vocab
    name, V, B, steps = "booking", 32000, 32, 3
    toks = vocab("bpe", V)
    vm = VocabMatrix(toks)
    d = oracle_dfa(name)
    ctx = make_ctx((name,), "bpe", V)
    states = _start_states((name,), B, np.random.default_rng(21))
    st = u32(states)
    for k in range(steps):
        vals, raw = make_logits(V, list(range(B)), k, 1234, 2.0, 4.0, 0.05, "bf16")
        hx = torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16).pin_memory()
        htok = torch.full((B,), -1, dtype=torch.int32).pin_memory()
        ns, fl = empty((B,), torch.int32).view(torch.uint32), empty((B,), torch.uint8)
        ctx.step_host(st, hx, temp, top_p, 5, k, htok, ns, fl)
        ctx.sync()
        assert ctx.status() == 0
        g_tok, g_ns, g_fl = htok.numpy().view(np.uint32), host(ns).view(np.uint32), host(fl)
        for b in range(B):
            s, t = int(states[b]), int(g_tok[b])
            allowed = token_mask(d, vm, s) if s != 0xFFFFFFFF else np.zeros(V, bool)
            res = sample_row(vals[b].astype(np.float64), allowed, temp, top_p, 5, b, k)
            assert same_token(t, res), (k, b, t, res.tok, res.gap, res.margin)
            want_s, want_f = accept(d, -1 if s == 0xFFFFFFFF else s, t, toks, False)
            assert g_ns[b] == (0xFFFFFFFF if want_s == DEAD else want_s) and g_fl[b] == want_f, (k, b)
        states = g_ns.copy()
        st = ns
