"""The N>1 bench path on CPU: two gloo ranks, each a replica of the same
workload (the path has no exchange step), reduce their timed-region lengths
to the maximum and report whole-job throughput over it."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from any_precision_bit_pw_gb300 import synth
        wl = synth.MIXTRAL_8X7B_DECODE
        # replicas draw identical inputs: the seeded generators do not depend on the rank
        x = synth.activations(wl, 0, 3)
        lg = synth.router_logits(wl, 0, 3)
        digest = torch.tensor([float(x.double().sum()), float(lg.double().sum())], dtype=torch.float64)
        peers = [torch.zeros_like(digest) for _ in range(world)]
        dist.all_gather(peers, digest)
        my_ms = 100.0 + 50.0 * rank
        dist.barrier()
        mx = bench.max_over_ranks(my_ms, world, "cpu")
        value = bench.job_throughput(wl.tokens, 10, world, mx)
        out[rank] = (mx, value, all(torch.equal(p, peers[0]) for p in peers))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        mx, value, same = res[r]
        assert mx == 150.0
        assert value == pytest.approx(32 * 10 * 2 / 0.150)
        assert same
