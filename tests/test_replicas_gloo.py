"""The replica path (several GPUs of one node) on CPU: two gloo ranks run the
bookkeeping bench.py uses -- process group, per-rank input seeds, the maximum
over ranks of the timed duration and the job throughput -- and decode their
own rows with the oracle, independently (rows shard; nothing is exchanged)."""

import os
import socket

import numpy as np
import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    from grammar_constrained_decoding_gb300 import replicas
    from oracle.dfa import compile_grammar
    from oracle.driver import OracleRun, Row
    from workloads import GRAMMARS, make_logits
    from workloads.vocab import make_vocab
    pg = replicas.init("gloo")
    w, r, _ = replicas.rank_info()
    spec = GRAMMARS["calc_call"]
    dfa = compile_grammar(spec.kind, spec.source, spec.bounds)
    toks = make_vocab("tiny", 512, 0)
    run = OracleRun([dfa], [spec], toks, spec.bounds.max_tokens)
    seed = replicas.replica_seed(11, r)
    rows = [Row(b, 0) for b in range(2)]
    produced, first = [], None
    for step in range(40):
        for row in rows:
            x, _ = make_logits(512, [row.b], step, seed, 1.0, 0.0, 0.0, "f32")
            if first is None:
                first = x[0].copy()
            rec = run.step_row(row, x[0].astype(np.float64), 0.0, 1.0, 0, step)
            produced.append(rec["tok"])
    ms = 10.0 + 5.0 * r                       # the slower rank sets the time
    top = replicas.max_over_ranks(ms, pg)
    pg.barrier()
    out.put((r, w, seed, top, replicas.job_throughput(12, w, top), produced, first))
    pg.destroy_process_group()


def test_two_gloo_replicas():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res = sorted(res, key=lambda t: t[0])
    (r0, w0, s0, t0, v0, p0, x0), (r1, w1, s1, t1, v1, p1, x1) = res
    assert (r0, r1, w0, w1) == (0, 1, 2, 2)
    assert s0 != s1 and not np.array_equal(x0, x1)   # each replica draws its own inputs
    assert t0 == t1 == 15.0                  # max over ranks
    assert v0 == v1 == pytest.approx(12 * 2 / 15e-3)
    assert p0 != p1                          # independent rows, different tokens


def test_single_process_needs_no_group(monkeypatch):
    from grammar_constrained_decoding_gb300 import replicas
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert replicas.init("gloo") is None
    assert replicas.max_over_ranks(3.5, None) == 3.5
    assert replicas.job_throughput(100, 1, 50.0) == pytest.approx(2000.0)
