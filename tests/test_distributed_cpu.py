"""Multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Sparse decode shards by token with no exchange step, so `bench.py --gpus N`
runs N replicas, each on its own batch.  What the ranks share is host logic:
 * the job's time is the slowest rank's (max over ranks);
 * each rank decodes an independent batch of the same shape;
 * the reported value counts all ranks' work;
 * only rank 0 runs and prints the reference (oracle) arm.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        from deepseek_sparse_mla_sfa_gb300 import workloads

        # the slowest rank's time is the job's time
        t = bench.max_over_ranks(1.5 + rank, world)
        assert t == 1.5 + (world - 1)

        # every rank decodes its own batch of the same shape
        base = workloads.small("mtp", B=2, S=700, S_min=300, top_k=96)
        w = bench.rank_workload(base, rank)
        assert (w.B, w.Q, w.h, w.top_k, w.S) == (base.B, base.Q, base.h, base.top_k, base.S)
        inp = workloads.make(w, device="cpu")
        out, lse = oracle.decode(oracle.Problem(inp.q, inp.kv, inp.block_table, inp.seq_lens,
                                                  inp.topk_idx, w.Q, w.scale))
        assert np.isfinite(out).all()
        sig = torch.tensor([float(np.nansum(lse[np.isfinite(lse)])), float(inp.q.float().sum())],
                           dtype=torch.float64)
        sigs = [torch.zeros_like(sig) for _ in range(world)]
        dist.all_gather(sigs, sig)
        for a in range(world):
            for b in range(a + 1, world):
                assert not torch.equal(sigs[a], sigs[b]), "ranks decoded the same batch"

        # value counts all ranks' work over the slowest rank's time
        acc = bench.accounting(inp)
        v = bench.job_value(acc["flops"], 2.0, world)
        assert v == pytest.approx(world * acc["flops"] / 2e-3 / 1e12)

        # the reference arm runs on rank 0 only: other ranks print nothing, do nothing
        if rank != 0:
            buf = io.StringIO()
            with redirect_stdout(buf):
                bench.run_reference(type("A", (), {"config": "tiny", "steps": 1, "warmup": 0})(),
                                    world, rank)
            assert buf.getvalue() == ""
        dist.barrier()
        with open(os.path.join(result_dir, f"ok{rank}"), "w") as f:
            f.write("ok")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert sorted(os.listdir(tmp_path)) == [f"ok{r}" for r in range(world)]

