"""Evaluator-aware decoding, end to end: the oracle (oracle.driver.OracleRun)
and the GPU path (cg_step on the device, the C++ forced-token driver on the
host) decode the same rows from the same logits, step by step, and must agree
on every token, every accept flag and every forced token -- including the
steps where a row closes an arithmetic span, the host evaluates it and the
result is forced into the row (labs.miniml.ai "Evaluator aware decoding",
"The core idea"; string operations: "Not just arithmetic: string
operations").  A sampled token may differ only where the oracle reports a
tolerance case (top-two Gumbel scores or the top-p boundary within 1e-5); such
a row is not compared further.
"""

import numpy as np
import pytest

from tests.gpu_helpers import host, make_ctx, product_vocab, u16, u32
from tests.oracle_cache import oracle_dfa, vocab
from workloads import GRAMMARS, make_logits

pytestmark = pytest.mark.gpu

FORMATS = {"calc_tag": 0, "json_answer": 1, "strop_tag": 2}


@pytest.mark.parametrize("names,temp,top_p", [
    (("calc_eval", "json_eval"), 0.0, 1.0),
    (("calc_eval", "json_eval"), 0.8, 0.9),
    (("calc_eval", "booking"), 0.7, 1.0),
    (("strop_eval", "calc_eval"), 0.0, 1.0),
    (("strop_eval", "json_eval"), 0.7, 0.9),
    (("calc_structtag", "strop_eval"), 0.0, 1.0),
])
def test_trajectory_matches_oracle(names, temp, top_p):
    import torch
    from grammar_constrained_decoding_gb300 import Driver
    from oracle.driver import OracleRun, Row
    V, B, steps, cap, seed = 4096, 8, 120, 2048, 5
    specs = [GRAMMARS[n] for n in names]
    toks = vocab("bpe", V)
    run = OracleRun([oracle_dfa(n) for n in names], specs, toks, cap)
    rows = [Row(b, b % len(names)) for b in range(B)]
    ctx = make_ctx(names, "bpe", V)
    gid_np = (np.arange(B) % len(names)).astype(np.uint16)
    rules = [(s.span_open, s.span_close, FORMATS[s.result_format]) if s.result_format else (b"", b"", -1)
             for s in specs]
    drv = Driver(product_vocab("bpe", V), B, gid_np, rules)
    gid = u16(gid_np) if len(names) > 1 else None
    states = u32(np.zeros(B))
    counts = u32(np.zeros(B))
    forced_next = np.full(B, -1, np.int32)
    live = np.ones(B, bool)
    forced_steps = np.zeros(len(names), int)
    for step in range(steps):
        vals, raw = make_logits(V, list(range(B)), step, seed, 2.0, 4.0, 0.05, "bf16")
        x = torch.from_numpy(raw.view(np.int16)).cuda().view(torch.bfloat16)
        forced_used = forced_next.copy()
        tok = torch.empty(B, dtype=torch.int32, device="cuda")
        flags = torch.empty(B, dtype=torch.uint8, device="cuda")
        ctx.step(states, x, temp, top_p, seed, step, tok, states, flags, gid=gid,
                 forced=torch.from_numpy(forced_used).cuda(), counts=counts, max_tokens=cap)
        assert ctx.status() == 0, step
        t_gpu = host(tok).view(np.uint32)
        f_gpu = host(flags)
        for b in range(B):
            if not live[b]:
                continue
            assert forced_used[b] == (rows[b].queue[0] if rows[b].queue else -1), (step, b)
            rec = run.step_row(rows[b], vals[b].astype(np.float64), temp, top_p, seed, step)
            if int(t_gpu[b]) != rec["tok"]:
                assert rec["gap"] < 1e-5 or rec["margin"] < 1e-5, (step, b, int(t_gpu[b]), rec["tok"])
                live[b] = False
                continue
            assert int(f_gpu[b]) == rec["flags"], (step, b, int(f_gpu[b]), rec["flags"])
            forced_steps[b % len(names)] += rec["forced"] >= 0
        drv.update(t_gpu, f_gpu, forced_used, forced_next)
        s_gpu = host(states).view(np.uint32)
        for b in range(B):
            if live[b]:
                assert int(s_gpu[b]) == rows[b].state, (step, b, int(s_gpu[b]), rows[b].state)
    assert live.sum() >= B // 2
    if temp == 0.0:
        for k, spec in enumerate(specs):
            if spec.result_format:
                assert forced_steps[k] > 0, f"no {spec.name} row reached an evaluated span"
