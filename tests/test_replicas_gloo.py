"""The N > 1 path of bench.py on the CPU: two gloo ranks through the same
Replicas helper (barrier, max over ranks, whole-job throughput)."""

import os
import socket
import tempfile

import numpy as np


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank: int, world: int, port: int, outdir: str) -> None:
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from quantized_linear_layers_block_gb300.replicas import Replicas
    r = Replicas()
    try:
        r.barrier()
        elapsed = 1.0 + rank          # rank 1 is the slower one
        mx = r.max(elapsed)
        rate = r.throughput(100.0, elapsed)
        r.barrier()
        np.save(os.path.join(outdir, f"r{rank}.npy"), np.array([mx, rate, r.world, r.rank]))
    finally:
        r.close()


def test_two_gloo_ranks_agree_on_max_and_throughput():
    import torch.multiprocessing as mp
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_worker, args=(2, _free_port(), d), nprocs=2, join=True)
        res = [np.load(os.path.join(d, f"r{r}.npy")) for r in range(2)]
    for r, v in enumerate(res):
        assert v[0] == 2.0                  # max elapsed over the ranks
        assert v[1] == 2 * 100.0 / 2.0      # all ranks' units over the slowest time
        assert v[2] == 2 and v[3] == r


def test_single_process_is_a_noop(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    from quantized_linear_layers_block_gb300.replicas import Replicas
    r = Replicas()
    r.barrier()
    assert r.max(3.5) == 3.5 and r.throughput(10.0, 2.0) == 5.0
    r.close()
