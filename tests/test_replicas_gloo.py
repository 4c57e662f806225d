"""Multi-rank bookkeeping of replica runs (the N > 1 path of the benchmark): barrier, the slowest
rank's step time on every rank, and the job throughput over all ranks' units, on two gloo ranks on
the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from ggml_iq_codebook_accumulate_b300 import replicas


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, step_ms, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = replicas.world_info()
        replicas.barrier()
        ms = replicas.max_over_ranks(step_ms[rank])
        replicas.barrier()
        q.put((r, w, local, ms, replicas.job_throughput(1000.0, ms * 1e-3, w)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("step_ms", [(10.0, 15.0), (7.5, 2.0)])
def test_two_gloo_ranks_take_the_slowest_rank(step_ms):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, step_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        out = sorted(q.get(timeout=180) for _ in range(2))
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    slowest = max(step_ms)
    assert [o[0] for o in out] == [0, 1]
    for r, w, local, ms, thr in out:
        assert (w, local) == (2, r)
        assert ms == slowest                       # every rank sees the job's time
        assert thr == pytest.approx(2 * 1000.0 / (slowest * 1e-3))


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert replicas.world_info() == (0, 1, 0)
    replicas.barrier()                              # no process group: nothing to wait for
    assert replicas.max_over_ranks(3.25) == 3.25
    assert replicas.job_throughput(10.0, 2.0, 1) == 5.0
    with pytest.raises(ValueError):
        replicas.job_throughput(10.0, 0.0, 1)
