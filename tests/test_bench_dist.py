"""Multi-rank path of bench.py on CPU: two gloo ranks, as `torchrun --nproc-per-node 2`
would start them.  The PaTH path shards by (batch, head) with no data-path
collective (one replica per GPU), so what needs checking is the bookkeeping:
the barrier, the slowest-rank time and the whole-job throughput."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_info()
        bench.barrier(ws)
        # each rank "measured" a different step time; the job takes the slowest
        ms = 10.0 + 5.0 * rank
        ms_max = bench.max_over_ranks(ms, ws)
        units = 8 * 4096  # tokens one rank processes per step
        rate = bench.job_throughput(units, ms_max, ws)
        bench.barrier(ws)
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            f.write("%d %d %d %r %r\n" % (got_ws, got_rank, got_local, ms_max, rate))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws", [2])
def test_two_gloo_ranks(tmp_path, ws):
    port = _free_port()
    mp.start_processes(_rank_main, args=(ws, port, str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    rows = []
    for r in range(ws):
        with open(tmp_path / ("rank%d.txt" % r)) as f:
            rows.append(f.read().split())
    slowest = 10.0 + 5.0 * (ws - 1)
    for r, row in enumerate(rows):
        assert int(row[0]) == ws and int(row[1]) == r and int(row[2]) == r
        assert float(row[3]) == slowest  # every rank sees the same max
        # whole-job rate: all ranks' tokens over the slowest rank's time
        assert float(row[4]) == pytest.approx(ws * 8 * 4096 / (slowest * 1e-3))


def test_single_rank_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)  # no process group needed
    assert bench.job_throughput(1000, 2.0, 1) == pytest.approx(5e5)


def test_flop_split_matches_pair_count():
    """The scan/prep split covers every causal chunk pair exactly once."""
    sys.path.insert(0, ROOT)
    import bench

    B, H, L, d, C = 1, 1, 1024, 128, 128
    N = L // C
    scan, prep = bench.prefill_flops(B, H, L, d, C)
    off_pairs = N * (N - 1) // 2
    u_products = (N - 1) * (N - 2) // 2
    assert scan == 4 * C * C * d * off_pairs + 2 * C * d * d * u_products
    # QK^T + PV over the causal triangle (the 2 d L^2 count): the off-diagonal
    # pairs plus each chunk's own block
    assert 4 * C * C * d * off_pairs + 2 * C * C * d * N == 2 * d * L * L
    assert prep == 16 * L * C * d + 2 * C * C * d * N
    assert torch.isfinite(torch.tensor(scan + prep))
