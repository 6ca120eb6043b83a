"""The N>1 benchmark path on CPU: two gloo ranks, one replica each, with the
barrier and the max-over-ranks timing reduction bench.py uses."""
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from spec_decode_recurrent_gb300 import dist
    r, lr, w = dist.init("gloo")
    dist.barrier()
    m = dist.max_over_ranks(10.0 * (rank + 1))
    seed = dist.replica_seed(2, r)
    dist.finalize()
    q.put((r, w, m, seed))


def test_two_rank_replicas_reduce_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[2] == 20.0 for r in res)          # every rank sees the slowest rank
    assert res[0][3] != res[1][3]                  # replicas draw different inputs


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    from spec_decode_recurrent_gb300 import dist
    assert dist.world() == (0, 0, 1)
    assert dist.max_over_ranks(3.5) == 3.5
