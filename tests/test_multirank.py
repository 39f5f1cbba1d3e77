"""The multi-GPU path is replicas only: every rank forwards its own tokens
with the same weights and no data-path collective; the job's time is the
slowest rank's and its rate is the work of all ranks over that time.  The
host side of that path is exercised here with two gloo ranks on the CPU,
each running one replica through the oracle."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        import oracle
        from workloads import make_tokens, make_weights, shape
        s = shape("tiny")
        w = make_weights(s, seed=0, device="cpu")
        x = make_tokens(s, seed=bench.replica_seed(rank), device="cpu")
        out = oracle.forward(x.float().numpy(), w.Wr.numpy(), w.bias.numpy(), w.W1.float().numpy(),
                             w.W2.float().numpy(), s.K, nthreads=1)
        my_ms = 10.0 + 5.0 * rank              # a made-up per-rank time: rank 1 is the slow one
        slowest = bench._max_over_ranks(my_ms, ws, device="cpu")
        q.put((rank, slowest, out["counts"].tolist(), float(np.abs(out["y"]).sum())))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_replicas_on_gloo():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks agree on the slowest rank's time
    assert [r[1] for r in res] == [15.0, 15.0]
    # each replica routed its own tokens: different batches, same weights
    assert res[0][2] != res[1][2]
    assert sum(res[0][2]) == sum(res[1][2]) == 256 * 2
    import bench
    # whole-job rate = work of all ranks' steps / slowest time
    assert bench.aggregate(100.0, ws, 3, 15.0) == pytest.approx(100.0 * 2 * 3 / 0.015)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        config = "tiny"
        steps = 1
        warmup = 1
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
