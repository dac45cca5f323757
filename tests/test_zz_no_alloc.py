"""cg_mask_and_sample_noalloc gives exactly the results of cg_mask_and_sample.

The no-allocation entry point runs the same kernels on a fixed scratch array in
the library instead of the context's allocated scratch, so the two must agree
bit for bit.  The file name puts it last in collection: it passes on its own
and after every other GPU test (the fixed scratch holds whatever the previous
calls left; nothing in it has to start at zero).
"""

import numpy as np
import pytest

from tests.gpu_helpers import empty, host, make_ctx, u32

pytestmark = pytest.mark.gpu


def _inputs(V, B, seed):
    import torch
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, 2.0, (B, V)) + 4.0 * (rng.random((B, V)) < 0.05)
    xt = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).cuda()
    W = (V + 31) // 32
    dens = np.where(np.arange(B) % 3 == 0, 0.002, 0.9)[:, None]   # sparse and dense rows
    bits = rng.random((B, W * 32)) < dens
    bits[:, V:] = False
    words = (bits.reshape(B, W, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(-1)
    return xt, u32(words.astype(np.uint32))   # bit t of word t // 32


@pytest.mark.parametrize("temp,top_p", [(0.7, 0.9), (0.7, 1.0), (0.0, 1.0)])
def test_noalloc_matches_allocating_entry_point(temp, top_p):
    import torch
    V, B = 128256, 48
    ctx = make_ctx(("calc_call",), "bpe", V)
    xt, bm = _inputs(V, B, 11)
    for step in (5, 6):   # two consecutive calls
        tok_a, tok_b = empty((B,), torch.int32), empty((B,), torch.int32)
        p_a, p_b = empty((B, V), torch.float32), empty((B, V), torch.float32)
        ctx.mask_and_sample(xt, bm, temp, top_p, 7, step, tok_a, probs=p_a)
        ctx.mask_and_sample_noalloc(xt, bm, temp, top_p, 7, step, tok_b, probs=p_b)
        assert ctx.status() == 0
        assert np.array_equal(host(tok_a), host(tok_b)), step
        assert np.array_equal(host(p_a).view(np.uint32), host(p_b).view(np.uint32)), step


def test_noalloc_rejects_oversized_batch():
    import torch
    from grammar_constrained_decoding_gb300 import CgError
    from grammar_constrained_decoding_gb300._lib import CG_E_LIMIT, CG_NOALLOC_MAX_ROWS
    V, B = 128256, CG_NOALLOC_MAX_ROWS + 1
    ctx = make_ctx(("calc_call",), "bpe", V)
    xt, bm = _inputs(V, B, 12)
    tok = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    with pytest.raises(CgError) as err:
        ctx.mask_and_sample_noalloc(xt, bm, 0.7, 0.9, 7, 0, tok)
    assert err.value.code == CG_E_LIMIT
    torch.cuda.synchronize()
    assert (host(tok) == -7).all()        # nothing was launched
    assert ctx.status() == 0


@pytest.mark.parametrize("temp,top_p", [(0.7, 0.9), (2.0, 0.999), (0.7, 1.0), (0.0, 1.0)])
def test_noalloc_full_batch_matches_oracle(temp, top_p):
    """CG_NOALLOC_MAX_ROWS rows on the fixed array, without the optional
    outputs: greedy and top_p >= 1 rows take the segmented sampler (its part of
    the fixed array), top-p rows the per-row kernels (temperature 2 with
    top_p 0.999 flattens the dense rows: their nuclei reach deep, towards or
    past the candidate margin).  Every row's id agrees with the oracle's
    (within the pages' tolerance for sampled ids) and with the allocating
    entry point, over two consecutive calls."""
    import torch
    from grammar_constrained_decoding_gb300._lib import CG_NOALLOC_MAX_ROWS
    from oracle.step import sample_row, unpack_bitmask
    from tests.gpu_helpers import same_token
    V, B = 128256, CG_NOALLOC_MAX_ROWS
    ctx = make_ctx(("calc_call",), "bpe", V)
    xt, bm = _inputs(V, B, 13)
    x = xt.float().cpu().numpy().astype(np.float64)
    masks = [unpack_bitmask(row, V) for row in host(bm).view(np.uint32)]
    for step in (5, 6):
        tok_a, tok_b = empty((B,), torch.int32), empty((B,), torch.int32)
        ctx.mask_and_sample(xt, bm, temp, top_p, 7, step, tok_a)
        ctx.mask_and_sample_noalloc(xt, bm, temp, top_p, 7, step, tok_b)
        assert ctx.status() == 0
        got = host(tok_b).view(np.uint32)
        assert np.array_equal(host(tok_a).view(np.uint32), got), step
        for b in range(B):
            res = sample_row(x[b], masks[b], temp, top_p, 7, b, step)
            if temp == 0.0:
                assert int(got[b]) == res.tok, (step, b, int(got[b]), res.tok)
            else:
                assert same_token(int(got[b]), res), (step, b, int(got[b]), res.tok, res.gap, res.margin)
