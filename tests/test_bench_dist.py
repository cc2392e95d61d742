"""World-size-2 CPU (gloo) checks of the benchmark's multi-rank plumbing.

Each rank decodes its own batch (weak scaling); ranks only agree on a barrier
and on the maximum timed duration.  These tests run that plumbing with two
gloo processes on the CPU.
"""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_setup(use_gpu=False)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    # every rank draws its own batch: seeds differ per rank, shapes agree
    from decode_phase_gqa_gb300 import workloads as W
    wl = W.make_workload("smollm3", seed=1000 * rank)
    q.put((rank, m, wl.seq_lens.tolist(), wl.n_seq))
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks_agree_on_max_time_and_draw_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]
    assert res[0][3] == res[1][3] == 8
    assert res[0][2] != res[1][2]


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
