"""bench.py's multi-GPU bookkeeping, run as two gloo ranks on the CPU: every
rank times its own tree (replicas, weak scaling); the job's time is the
slowest rank's and its throughput counts the work of all ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [120.0, 150.0][rank]
    mx = bench.max_over_ranks(local, world)
    tput = bench.job_throughput(1e12, 10, world, mx)
    dist.barrier()
    results[rank] = (mx, tput)
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    port = _free_port()
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0][0] == res[1][0] == 150.0
    # 2 ranks x 10 steps x 1e12 FLOP in 0.150 s
    assert res[0][1] == pytest.approx(2 * 10 * 1e12 / 0.150 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(42.0, 1) == 42.0
    assert bench.job_throughput(2e12, 5, 1, 1000.0) == pytest.approx(10.0)


def test_expanded_chain_batches():
    """The expanded-trajectory leg splits its chains into equal contiguous
    batches only when one batch would not fit the memory budget."""
    import bench
    import prefix_tree_attention_attn_gb300 as TA
    lens = [5000, 7000, 3000, 9000, 4000, 6000, 8000, 2000]
    whole = bench.chain_batches(TA, lens, 8, 2, 128, 1e15)
    assert whole == [lens]
    tight = bench.chain_batches(TA, lens, 8, 2, 128, 2e8)
    assert len(tight) > 1 and [x for g in tight for x in g] == lens
    assert len({len(g) for g in tight[:-1]}) == 1
    one_each = bench.chain_batches(TA, lens, 8, 2, 128, 1.0)
    assert one_each == [[x] for x in lens]
