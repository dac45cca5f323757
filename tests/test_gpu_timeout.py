"""Failure detection without a fault: a bounded device wait that runs out
records CG_DEV_TIMEOUT, the host reads it, and the context stays usable.

cg_self_test_wait_timeout arms a barrier for bytes no copy delivers and waits
on it with the library's bounded wait (the one its sampling and accept
kernels use).  Nothing faults, traps or hangs: the wait gives up after its
polling limit and returns.
"""

import time

import numpy as np
import pytest

from tests.gpu_helpers import empty, host, make_ctx, oracle_bitmask, u32
from tests.oracle_cache import oracle_dfa, vocab

pytestmark = pytest.mark.gpu

CG_DEV_TIMEOUT = 8


def test_bounded_wait_runs_out_and_context_stays_usable():
    import torch
    from oracle.step import VocabMatrix
    ctx = make_ctx(("calc_call",), "tiny", 512)
    t0 = time.perf_counter()
    ctx.self_test_wait_timeout()
    code = ctx.status()
    elapsed = time.perf_counter() - t0
    assert code == CG_DEV_TIMEOUT
    assert elapsed < 10.0, elapsed
    assert ctx.status() == 0                      # read once, then cleared
    # the same context keeps working: masks for a few states match the oracle
    dfa = oracle_dfa("calc_call")
    vm = VocabMatrix(vocab("tiny", 512))
    states = np.array([0, 1, 2, 3], np.uint32)
    bm = empty((4, 16), torch.int32)
    ctx.fill_bitmask(u32(states), bm)
    assert ctx.status() == 0
    got = host(bm).view(np.uint32)
    for b, s in enumerate(states):
        assert np.array_equal(got[b], oracle_bitmask(dfa, vm, int(s))), b
