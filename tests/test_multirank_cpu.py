"""The multi-rank (torchrun) side of bench.py on CPU: two gloo ranks check the
barrier, the max-over-ranks timing and the whole-job throughput (units of all
ranks divided by the slowest rank's time), and that each rank gets its own
documents.  No GPU and no data-path collective are involved: the layer's
documents are independent, so ranks only meet at the start/stop barrier."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.barrier(w)
    secs = 1.0 + rank  # rank 1 is the slower one
    value, tmax = bench.aggregate_throughput(1000.0, secs, w)
    # inputs: each rank's own document, the shared layer weights
    from ttt_inputs import make_layer
    cfg = make_layer(16, 32, 8, 4, 2, 1e-3, dtype="bf16", seed=0, init="qwen",
                     x_seed=bench.workload_x_seed(rank, w))
    q.put((rank, value, tmax, float(cfg["x"][0, 0]), float(cfg["w_gate"][0, 0])))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, tmax, _, _ in res:
        assert tmax == pytest.approx(2.0)           # the slowest rank's time
        assert value == pytest.approx(2000.0 / 2.0)  # both ranks' units / max time
    assert res[0][3] != res[1][3]                    # different documents per rank
    assert res[0][4] == res[1][4]                    # the same layer weights


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.aggregate_throughput(500.0, 2.0, 1) == (250.0, 2.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
