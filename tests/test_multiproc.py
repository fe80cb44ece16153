"""World-size-2 process groups on CPU (gloo): the replica timing reduction and
tensor-parallel reassembly through real collectives.  Each rank computes its
shard with the oracle; no GPU is involved."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from parity import oracle_ref
        from ternary_weight_linear_02_gb300 import dist_util, shard, synth
        oracle.build()
        res = {}
        # replica timing: slowest rank, whole-job throughput
        mx = dist_util.max_over_ranks(1.5 + rank)
        res["max"] = mx
        res["thr"] = dist_util.job_throughput(100.0, mx, world)
        # column parallel: all-gather of the shards' outputs
        M, N, K, gs = 3, 256, 512, 128
        x, p, s = synth.layer(M, N, K, torch.bfloat16, gs, 0.005, 0.05, ("mp", 1), "cpu", 0.01)
        full = oracle_ref(x, p, s, gs)
        pi, si = shard.split_n(p, s, [N // world] * world)[rank]
        mine = torch.from_numpy(oracle_ref(x, pi, si, gs))
        parts = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine)
        res["col_exact"] = bool(np.array_equal(torch.cat(parts, dim=1).numpy(), full))
        # row parallel: all-reduce of the partial sums
        sizes = shard.even_cuts(K, world, 128)
        pk, sk_, k0 = shard.split_k(p, s, sizes)[rank]
        part = torch.from_numpy(oracle_ref(x[:, k0:k0 + pk.shape[1] * 4].contiguous(), pk, sk_, gs))
        dist.all_reduce(part, op=dist.ReduceOp.SUM)
        res["row_err"] = float(np.max(np.abs(part.numpy() - full)) / max(np.max(np.abs(full)), 1e-30))
        q.put((rank, res))
    finally:
        dist.destroy_process_group()


def test_two_rank_replica_and_tp_reassembly():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        assert out[r]["max"] == 2.5
        assert out[r]["thr"] == pytest.approx(2 * 100.0 / 2.5e-3)
        assert out[r]["col_exact"]
        assert out[r]["row_err"] < 1e-12
