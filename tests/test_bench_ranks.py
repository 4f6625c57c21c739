"""The replicas-only multi-rank path of bench.py: every rank runs the whole
single-GPU workload, and rank 0 reports the whole job -- the attention bytes
of all ranks over the slowest rank's attention time, and the slowest rank's
step time.  Two gloo ranks on CPU (no GPU, no kernel)."""
import os
import socket
import sys

import torch.multiprocessing as mp

from conftest import ROOT


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    local = {"value": 1.0, "ms_per_step": [0.02, 0.03][rank], "n_gpus": 1,
             "_attn": ([1e9, 3e9][rank], [0.5, 2.0][rank])}
    out = bench.combine_ranks(local)
    q.put((rank, out["value"], out["ms_per_step"], out["n_gpus"]))
    dist.destroy_process_group()


def test_combine_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(60)
        assert p.exitcode == 0
    for rank, value, ms, n in res:
        assert value == round(4e9 / 2.0 / 1e9, 2)  # every rank's bytes over the slowest rank's time
        assert ms == 0.03 and n == 2
