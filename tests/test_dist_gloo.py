"""The multi-rank path of the benchmark on CPU with gloo (world size 2): each
rank draws its own batch, the timing barrier holds, the job time is the max
over ranks, and the whole-job throughput counts every rank's units.  Rows are
independent, so the per-rank results must equal the oracle on that rank's own
batch with no data exchanged."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import oracle
    from memory_fusion_gb300 import dist as mdist
    from memory_fusion_gb300 import inputs

    r = mdist.Ranks("gloo")
    assert (r.world, r.rank) == (world, rank)
    # each rank: its own seeded batch of a small softmax workload
    seed = mdist.seed_for(1, rank)
    d = inputs.gemm_inputs(64, 128, 64, seed, x_std=1.0, w_std=0.125, bias_std=None, gamma_std=None,
                           beta_std=None)
    y = oracle.gemm_rowsoftmax(d["X"], d["W"], scale=0.125)
    r.barrier()
    elapsed = 0.010 * (rank + 1)              # a stand-in per-rank time
    t = r.max(elapsed)
    thr = mdist.job_throughput(1000.0, world, t)
    out[rank] = (float(y.sum()), float(d["X"][0, 0]), t, thr)
    r.close()


@pytest.mark.timeout(120)
def test_two_gloo_ranks():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert sorted(out.keys()) == [0, 1]
    for rank in range(world):
        rows_sum, x00, t, thr = out[rank]
        assert abs(rows_sum - 64) < 1e-9           # 64 softmax rows, each summing to 1
        assert t == pytest.approx(0.020)          # max over ranks
        assert thr == pytest.approx(1000.0 * 2 / 0.020)
    assert out[0][1] != out[1][1]                 # the ranks drew different batches


def test_single_rank_defaults(monkeypatch):
    from memory_fusion_gb300 import dist as mdist
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    r = mdist.Ranks("gloo")
    assert (r.world, r.rank) == (1, 0) and r.pg is None
    assert r.max(3.5) == 3.5
    r.barrier()
    r.close()
    assert mdist.seed_for(4, 0) == 4 and mdist.seed_for(4, 2) == 2004
    assert np.isclose(mdist.job_throughput(10, 4, 2.0), 20.0)
