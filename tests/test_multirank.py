"""The bench's N>1 path on CPU with two gloo ranks: each rank's share of the
job is a batch of its own (no data moves between ranks), the step time is the
maximum over ranks, the job's throughput counts every rank's work, and the
reference arm runs on rank 0 alone."""
import contextlib
import io
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        r, world, local = bench.dist_setup()
        # this rank's batch, reduced in size; gathered to compare across ranks
        w = bench.rank_workload(bench.CAUSAL_4K, r)
        q = bench.make_inputs(w, L=256, B=1, H=2)["q"].float()
        qs = [torch.zeros_like(q) for _ in range(world)]
        dist.all_gather(qs, q)
        # the slower rank sets the step time
        ms = bench.max_over_ranks(1.5 + r, torch.device("cpu"))
        value = bench.job_throughput(1e12, ms, world)
        # the reference arm: only rank 0 works and prints
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            ran = None
            if r != 0:
                ran = bench.run_reference(None)
        results.put(dict(rank=r, world=world, local=local, seed=w.seed,
                         same_batch=bool(torch.equal(qs[0], qs[1])), ms=ms, value=value,
                         ref_return=ran, ref_out=out.getvalue()))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_shard_and_reduce():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, results)) for r in range(WORLD)]
    for p in procs:
        p.start()
    got = [results.get(timeout=240) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    by_rank = {g["rank"]: g for g in got}
    assert sorted(by_rank) == [0, 1]
    for g in got:
        assert g["world"] == WORLD and g["local"] == g["rank"]
        assert not g["same_batch"]                 # every rank draws its own batch
        assert g["ms"] == 2.5                      # the maximum over ranks, on every rank
        assert abs(g["value"] - 2 * 1e12 / 2.5 / 1e9) < 1e-9
    assert by_rank[0]["seed"] != by_rank[1]["seed"]
    assert by_rank[1]["ref_return"] is None and by_rank[1]["ref_out"] == ""


def test_single_rank_workload_is_the_configured_one():
    import bench
    assert bench.rank_workload(bench.CAUSAL_4K, 0) == bench.CAUSAL_4K
    assert bench.job_throughput(3e12, 2.0, 1) == pytest.approx(1500.0)   # TFLOP/s
