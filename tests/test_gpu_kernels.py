"""GPU parity of the three step kernels against the oracle (through the C ABI).

Bitmasks, next states, flags and greedy ids must be bit-exact; softmax
probabilities within 1e-5 absolute; sampled ids identical except where the
oracle's top-two Gumbel scores (or the top-p threshold) are within 1e-5."""

import numpy as np
import pytest

from oracle.dfa import DEAD
from oracle.step import (FLAG_NO_TOKEN, NO_TOKEN, VocabMatrix, accept, sample_row,
                         token_mask, unpack_bitmask)
from tests.gpu_helpers import (empty, host, logits_rows, make_ctx, oracle_bitmask, same_token,
                               u16, u32)
from tests.oracle_cache import oracle_dfa, vocab
from workloads import GRAMMARS

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
from grammar_constrained_decoding_gb300 import _lib  # noqa: E402


def _rows_for(dfas, n, rng, with_dead=True):
    gid = rng.integers(0, len(dfas), n)
    states = np.array([rng.integers(0, dfas[g].n_states) for g in gid], dtype=np.int64)
    if with_dead:
        states[::11] = -1
    return gid, states


@pytest.mark.parametrize("names,kind,V", [
    (("calc_call",), "tiny", 512),
    (("booking_200",), "bpe", 4013),
    (("calc_eval", "booking_200", "json_eval"), "bpe", 2999),
])
def test_fill_bitmask(names, kind, V):
    ctx = make_ctx(names, kind, V)
    dfas = [oracle_dfa(n) for n in names]
    vm = VocabMatrix(vocab(kind, V))
    rng = np.random.default_rng(1)
    B = 97
    gid, states = _rows_for(dfas, B, rng)
    forced = np.full(B, -1, np.int64)
    forced[5::13] = rng.integers(0, V, len(forced[5::13]))
    # a forced-only state with no forced token is a driver error: empty mask + status
    expect_missing = False
    for b in range(B):
        if forced[b] < 0 and states[b] >= 0 and dfas[gid[b]].forced_only()[states[b]]:
            expect_missing = True
    st = u32(np.where(states < 0, 0xFFFFFFFF, states).astype(np.uint32))
    W = (V + 31) // 32
    for rep in range(3):  # first call fills the cache, second reads it, third after prefill
        if rep == 2:
            ctx2 = make_ctx(names, kind, V)
            ctx2.prefill()
            ctx = ctx2
        bm = empty((B, W), torch.int32)
        ctx.fill_bitmask(st, bm, gid=u16(gid), forced=torch.as_tensor(forced.astype(np.int32)).cuda())
        code = ctx.status()
        got = host(bm).view(np.uint32)
        for b in range(B):
            want = oracle_bitmask(dfas[gid[b]], vm, int(states[b]), int(forced[b])) if states[b] >= 0 or forced[b] >= 0 \
                else np.zeros(W, np.uint32)
            if forced[b] < 0 and states[b] >= 0 and dfas[gid[b]].forced_only()[states[b]]:
                want = np.zeros(W, np.uint32)
            assert np.array_equal(got[b], want), (rep, b, gid[b], states[b], forced[b])
        assert code == (5 if expect_missing else 0)                # CG_DEV_MISSING_FORCED
    assert ctx.info()["n_classes"] > 0


def _sampler_case(V, dtype, temp, top_p, B=13, seed=3, boost=4.0, frac=0.05, density=0.6):
    ctx = make_ctx(("calc_call",), "bpe" if V > 600 else "tiny", V)
    rng = np.random.default_rng(seed)
    masks = rng.random((B, V)) < density
    masks[1] = False                      # no allowed token
    masks[2] = False
    masks[2, V - 1] = True                # one allowed token, the last id
    masks[3] = True                       # all allowed
    from oracle.step import pack_bitmask
    bm = np.stack([pack_bitmask(m) for m in masks])
    x, xt = logits_rows(V, range(B), 7, 11, 2.0, boost, frac, dtype)
    if dtype == "bf16":
        # ties: a block of equal logits
        x[4, :40] = x[4, 0]
        xt[4, :40] = xt[4, 0]
    # with probabilities requested (the per-row kernels), then without (the
    # segmented sampler for bf16 rows)
    for want_probs in (True, False):
        out = empty((B,), torch.int32)
        probs = empty((B, V), torch.float32) if want_probs else None
        ctx.mask_and_sample(xt, u32(bm), temp, top_p, 0xABCDEF0123, 5, out, probs=probs)
        assert ctx.status() == 0
        got = host(out).view(np.uint32)
        gp = host(probs) if want_probs else None
        for b in range(B):
            res = sample_row(x[b], masks[b], temp, top_p, 0xABCDEF0123, b, 5)
            if temp == 0.0:
                assert got[b] == res.tok, (want_probs, b, got[b], res.tok)
            else:
                assert same_token(int(got[b]), res), (want_probs, b, got[b], res.tok, res.gap, res.margin)
            if want_probs:
                assert np.max(np.abs(gp[b] - res.probs)) <= 1e-5, b


@pytest.mark.parametrize("V", [512, 4013, 32000])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("temp,top_p", [(0.0, 1.0), (0.7, 1.0), (0.7, 0.9), (1.3, 0.5), (0.7, 0.0)])
def test_mask_and_sample(V, dtype, temp, top_p):
    _sampler_case(V, dtype, temp, top_p)


def test_topp_nucleus_below_key_window():
    # flat, wide logits and top_p close to 1: the nucleus reaches negative
    # logits, below the per-key window, so the bisection path decides
    _sampler_case(4013, "bf16", 5.0, 0.999, boost=0.0, frac=0.0, density=0.9)


def test_sampler_statistics_match_oracle_over_many_steps():
    V, B = 64, 8
    ctx = make_ctx(("calc_call",), "tiny", 512)
    rng = np.random.default_rng(5)
    x, xt = logits_rows(512, range(B), 1, 2, 1.0, 0.0, 0.0, "bf16")
    masks = np.zeros((B, 512), bool)
    masks[:, :V] = rng.random((B, V)) < 0.8
    from oracle.step import pack_bitmask
    bm = u32(np.stack([pack_bitmask(m) for m in masks]))
    out = empty((B,), torch.int32)
    agree = 0
    total = 0
    for step in range(200):
        ctx.mask_and_sample(xt, bm, 0.8, 0.85, 77, step, out)
        got = host(out).view(np.uint32)
        for b in range(B):
            res = sample_row(x[b], masks[b], 0.8, 0.85, 77, b, step)
            assert same_token(int(got[b]), res)
            agree += int(got[b] == res.tok)
            total += 1
    assert agree >= total - 2


def test_accept():
    names = ("calc_eval", "json_eval", "booking_200")
    V = 2999
    ctx = make_ctx(names, "bpe", V)
    toks = vocab("bpe", V)
    dfas = [oracle_dfa(n) for n in names]
    vm = VocabMatrix(toks)
    rng = np.random.default_rng(9)
    B = 300
    gid, states = _rows_for(dfas, B, rng, with_dead=False)
    tok = np.zeros(B, np.int64)
    forced = np.full(B, -1, np.int64)
    for b in range(B):
        d = dfas[gid[b]]
        s = int(states[b])
        if d.forced_only()[s]:
            # a legal injected byte from this state
            syms = np.flatnonzero(d.next[s, 256:] >= 0)
            tok[b] = int(syms[0])          # single-byte token ids equal the byte
            forced[b] = tok[b]
        else:
            m = token_mask(d, vm, s)
            allowed = np.flatnonzero(m)
            tok[b] = int(rng.choice(allowed)) if allowed.size and b % 7 else int(rng.integers(0, V))
    tok[3] = NO_TOKEN
    states[8] = -1
    counts = rng.integers(0, 6, B).astype(np.uint32)
    for use_counts in (False, True):
        out_s = empty((B,), torch.int32)
        out_f = empty((B,), torch.uint8)
        cnt = u32(counts) if use_counts else None
        ctx.accept(u32(np.where(states < 0, 0xFFFFFFFF, states)), u32(tok), out_s, out_f, gid=u16(gid),
                   forced=torch.as_tensor(forced.astype(np.int32)).cuda(), counts=cnt, max_tokens=5)
        ctx.status()
        gs = host(out_s).view(np.uint32)
        gf = host(out_f)
        gc = host(cnt).view(np.uint32) if use_counts else None
        for b in range(B):
            ns, fl = accept(dfas[gid[b]], int(states[b]), int(tok[b]), toks, forced[b] >= 0)
            want_s = 0xFFFFFFFF if ns == DEAD else ns
            if use_counts:
                c = int(counts[b]) + (0 if tok[b] == NO_TOKEN else 1)
                if (fl & 1) or c >= 5:
                    if not (fl & 1):
                        fl |= _lib.CG_FLAG_CAPPED
                    want_s, c = 0, 0
                assert gc[b] == c, b
            assert gs[b] == want_s and gf[b] == fl, (b, gs[b], want_s, gf[b], fl)


def test_device_status_codes():
    # one faulty row per call: the status word keeps the first code recorded
    ctx = make_ctx(("calc_call",), "tiny", 512)
    tid = {t: i for i, t in enumerate(vocab("tiny", 512))}
    bm = empty((2, 16), torch.int32)
    ctx.fill_bitmask(u32([1, 0]), bm, gid=u16([0, 3]))
    assert ctx.status() == 6                                   # bad grammar index
    assert ctx.status() == 0                                   # cleared
    ctx.fill_bitmask(u32([10**6, 0]), bm)
    assert ctx.status() == 1                                   # state out of range
    out_s = empty((2,), torch.int32)
    out_f = empty((2,), torch.uint8)
    ctx.accept(u32([0]), u32([5000]), out_s[:1], out_f[:1])
    assert ctx.status() == 2                                   # token out of range
    ctx.accept(u32([0]), u32([tid[b"c"]]), out_s[:1], out_f[:1],
               forced=torch.tensor([tid[b"d"]], dtype=torch.int32, device="cuda"))
    assert ctx.status() == 4                                   # forced token differs
    ctx.accept(u32([0]), u32([tid[b"x"]]), out_s[:1], out_f[:1])
    assert ctx.status() == 7 and host(out_f)[0] == _lib.CG_FLAG_REJECTED
    ctx.accept(u32([0]), u32([tid[b"c"]]), out_s[:1], out_f[:1])
    assert ctx.status() == 0 and host(out_f)[0] == 0


def _topp_rows(V, B, case, rng):
    x = rng.normal(0, 2, (B, V)).astype(np.float32)
    masks = rng.random((B, V)) < 0.9
    if case == "boosted":                       # the throughput workload's distribution
        x += 4.0 * (rng.random((B, V)) < 0.05)
    elif case == "sparse":                      # few allowed tokens, small logits: list bisection
        masks = rng.random((B, V)) < 0.0002
        masks[:, 7] = True
    elif case == "flat":                        # nucleus below the candidate margin: general path
        x = rng.uniform(-1.0, 1.0, (B, V)).astype(np.float32)
    elif case == "ties":                        # every logit equal: candidate list overflows
        x[:] = 0.5
        masks[:] = True
    import torch as _t
    xt = _t.from_numpy(x).to(_t.bfloat16)
    vals = xt.to(_t.float32).numpy().astype(np.float64)
    return vals, xt.cuda(), masks


@pytest.mark.parametrize("case,temp,top_p", [("boosted", 0.7, 0.9), ("boosted", 1.0, 0.5), ("plain", 0.7, 0.9),
                                            ("sparse", 0.7, 0.9), ("flat", 2.0, 0.999), ("ties", 0.7, 0.9)])
def test_single_pass_topp_branches(case, temp, top_p):
    V, B = 128256, 12
    ctx = make_ctx(("calc_call",), "bpe", V)
    rng = np.random.default_rng(sum(case.encode()))
    x, xt, masks = _topp_rows(V, B, case, rng)
    from oracle.step import pack_bitmask
    bm = u32(np.stack([pack_bitmask(m) for m in masks]))
    for want_probs in (True, False):
        out = empty((B,), torch.int32)
        probs = empty((B, V), torch.float32) if want_probs else None
        ctx.mask_and_sample(xt, bm, temp, top_p, 99, 3, out, probs=probs)
        assert ctx.status() == 0
        got = host(out).view(np.uint32)
        for b in range(B):
            res = sample_row(x[b], masks[b], temp, top_p, 99, b, 3)
            assert same_token(int(got[b]), res), (case, want_probs, b, got[b], res.tok, res.gap, res.margin,
                                                  res.nucleus_size)
            if want_probs:
                assert np.max(np.abs(host(probs)[b] - res.probs)) <= 1e-5, (case, b)
