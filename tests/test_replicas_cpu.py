"""The multi-GPU path is replicas only: each rank runs its own sequences with
no data exchange, and the bench reports all ranks' tokens over the slowest
rank's time. Two gloo ranks on the CPU check that host logic and that
replicas of the integer model agree bit for bit (the oracle stands in for
the GPU library here)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist          # noqa: E402
import torch.multiprocessing as mp        # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, path, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        import oracle
        import synth
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        m = oracle.Model(path)
        s = m.new_seq(64)
        am, lg = s.feed(synth.prompt_ids(0, 0, 16, m.vocab))
        toks, h = [am], oracle.chain_hash([lg])
        for _ in range(3):
            am, lg = s.feed([toks[-1]])
            toks.append(am)
            h = oracle.chain_hash([lg], h)
        got = [None] * ws
        dist.all_gather_object(got, (toks, h.hex()))
        out[rank] = (ms, got)
    finally:
        dist.destroy_process_group()


def test_two_replicas_agree_and_time_is_the_max():
    import synth
    path = synth.ensure_artifact("tiny", 0)
    ws = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(ws, _free_port(), path, out), nprocs=ws, join=True)
    assert set(out.keys()) == {0, 1}
    for r in range(ws):
        ms, got = out[r]
        assert ms == 15.0                       # the slowest rank's time on every rank
        assert got[0] == got[1]                 # the replicas' tokens and chain hash agree
