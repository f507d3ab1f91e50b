"""The multi-process path of bench.py on CPU: two gloo ranks, as torchrun
would launch them (one process per GPU on a GPU machine)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.dist_max(times[rank], world)
        bench.dist_barrier(world)
        out.put((rank, m, bench.throughput(8, 10, world, m)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_slowest_rank_sets_the_job_time(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [12.5, 40.0, 7.0][:world]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [m for _, m, _ in res] == [max(times)] * world
    # 8 tokens x 10 steps on each rank over the slowest rank's 40 ms (or 12.5 ms)
    for _, m, v in res:
        assert v == pytest.approx(8 * 10 * world / (max(times) / 1e3))


def test_accounting_matches_cost_model():
    import bench
    import oracle as O
    from deepseek_sparse_attention_lightning_gb300 import workloads as W
    spec = W.SPECS["long_128k"]
    u = bench.accounting(spec, [131072] * 8)
    assert u["layer_bytes"] == 8 * O.decode_bytes(131072)
    assert u["indexer_flops"] + u["attention_flops"] == 8 * O.decode_flops(131072)
    spec2 = W.SPECS["mtp_32k"]
    u2 = bench.accounting(spec2, [32769] * 32)
    assert u2["layer_bytes"] == O.layer_bytes([32769] * 32, 2, 2048)
