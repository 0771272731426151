"""Host logic of the multi-GPU benchmark path, run as two gloo ranks on the CPU.

Each rank draws its own batch (weak scaling) and the step time reported is the
maximum over ranks; no collective touches the data path."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    import sys

    import torch.distributed as dist

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads

    assert bench.dist_env() == (rank, rank, world)
    t = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
    b = workloads.build("r", bench.rank_seed(5, rank), [40, 20], [1, 1], 8, 2, 64, 16, "bf16")
    results[rank] = (t, b.q.tobytes()[:64], int(b.seq_lens.sum()))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_max_time_and_distinct_batches():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    assert results[0][0] == results[1][0] == 15.0      # max over ranks
    assert results[0][1] != results[1][1]              # each rank its own inputs
    assert results[0][2] == results[1][2] == 60        # same shape (weak scaling)


def test_single_process_max_is_identity():
    import bench

    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.rank_seed(2, 0) == 2 and bench.rank_seed(2, 1) != bench.rank_seed(2, 0)
