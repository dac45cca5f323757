"""Edge cases of the C ABI on the GPU.

* An empty batch (B = 0) is a valid call for every entry point: it returns
  CG_OK, launches nothing and leaves the outputs untouched.
* Vocabularies beyond the fused kernel's shared-memory plan (V = 262144,
  W = 8192 words of mask, and the ragged V = 262149) take the separate
  kernels; their masks, sampled ids and next states still match the oracle
  (usetacet.com/docs/grammar, "The guarantee": the mask is applied whatever
  the vocabulary size).
"""

import numpy as np
import pytest

from oracle.dfa import DEAD
from oracle.step import VocabMatrix, accept, pack_bitmask, sample_row, token_mask
from tests.gpu_helpers import empty, host, make_ctx, product_grammar, same_token, u32
from tests.oracle_cache import oracle_dfa, vocab
from workloads import make_logits

pytestmark = pytest.mark.gpu


def test_empty_batch_is_a_no_op():
    import torch
    V = 4013
    ctx = make_ctx(("calc_call",), "bpe", V)
    W = (V + 31) // 32
    z32 = torch.empty((0,), dtype=torch.int32, device="cuda").view(torch.uint32)
    zf = torch.empty((0,), dtype=torch.uint8, device="cuda")
    zt = torch.empty((0,), dtype=torch.int32, device="cuda")
    bm = torch.empty((0, W), dtype=torch.int32, device="cuda")
    x = torch.empty((0, V), dtype=torch.bfloat16, device="cuda")
    ctx.fill_bitmask(z32, bm)
    ctx.mask_and_sample(x, bm, 0.7, 0.9, 1, 0, zt)
    ctx.accept(z32, z32, z32, zf)
    ctx.step(z32, x, 0.7, 0.9, 1, 0, zt, z32, zf)
    ctx.accept_many(z32, torch.empty((0, 4), dtype=torch.int32, device="cuda").view(torch.uint32), z32, z32, z32, zf)
    assert ctx.status() == 0


@pytest.mark.parametrize("V,dtype", [(262144, "bf16"), (262149, "bf16"), (262144, "f32")])
def test_large_vocabulary_takes_the_separate_kernels(V, dtype):
    import torch
    names = ("calc_eval",)
    B, temp, top_p, seed, step = 6, 0.7, 0.9, 17, 3
    toks = vocab("bpe", V)
    dfa = oracle_dfa(names[0])
    vm = VocabMatrix(toks)
    ctx = make_ctx(names, "bpe", V)
    W = (V + 31) // 32
    live = np.flatnonzero(dfa.next[:, :256].max(axis=1) >= 0)     # states the model can continue from
    rng = np.random.default_rng(V)
    states = np.array([0] + [int(live[rng.integers(len(live))]) for _ in range(B - 1)], np.uint32)
    vals, raw = make_logits(V, range(B), step, 5, 2.0, 4.0, 0.05, dtype)
    if dtype == "bf16":
        x = torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        x = torch.from_numpy(raw).cuda()
    bm = empty((B, W), torch.int32)
    tok = empty((B,), torch.int32)
    ns, fl = empty((B,), torch.int32).view(torch.uint32), empty((B,), torch.uint8)
    ctx.step(u32(states), x, temp, top_p, seed, step, tok, ns, fl, bitmask=bm)
    assert ctx.status() == 0
    g_bm, g_tok = host(bm).view(np.uint32), host(tok).view(np.uint32)
    g_ns, g_fl = host(ns).view(np.uint32), host(fl)
    for b in range(B):
        allowed = token_mask(dfa, vm, int(states[b]))
        assert np.array_equal(g_bm[b], pack_bitmask(allowed)), b
        res = sample_row(vals[b].astype(np.float64), allowed, temp, top_p, seed, b, step)
        assert same_token(int(g_tok[b]), res), (b, int(g_tok[b]), res.tok)
        if int(g_tok[b]) == res.tok:
            want_s, want_f = accept(dfa, int(states[b]), res.tok, toks, False)
            assert g_ns[b] == (0xFFFFFFFF if want_s == DEAD else want_s) and g_fl[b] == want_f, b
