"""Sequence-sharded (context-parallel) prefill, the parts that need no GPU:
the partition of the chunks over the ranks (the library's path_attn_cp_rows)
and the all-gather of the exchange blocks between ranks (two and three gloo
ranks on CPU, as torchrun would start them).

The layout the scan relies on is restated here from its documentation in
include/path_attn.h, independently of the library's code: 2 * world blocks of
nb = ceil(N / (2 * world)) chunks of 128 positions, rank r holding blocks r
and 2 * world - 1 - r, and each rank's exchange block laid out as
[Kh, Pm, V][batch * heads][2 * nb * 128][128] bf16 at its local rows."""
import math
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import dependent_positional_attention_gb300 as pa
from dependent_positional_attention_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pa_build.build()
    pa.load_library()


def blocks_of(rank, world, N):
    nb = math.ceil(N / (2 * world))
    return nb, [rank, 2 * world - 1 - rank]


@pytest.mark.parametrize("L,world", [(4096, 2), (4096, 4), (32768, 8), (1000, 3), (130, 4),
                                     (1, 2), (300, 1), (4095, 5)])
def test_ranks_cover_every_position_once_in_zigzag_blocks(L, world):
    N = math.ceil(L / 128)
    seen = []
    for r in range(world):
        rows = pa.path_attn_cp_rows(1, 1, L, world, r).tolist()
        assert len(rows) == pa.path_attn_cp_local_len(1, 1, L, world, r)
        assert rows == sorted(rows)
        nb, blks = blocks_of(r, world, N)
        expect = [p for b in blks for p in range(b * nb * 128, min((b + 1) * nb * 128, L))]
        assert rows == expect
        seen += rows
    assert sorted(seen) == list(range(L))


def test_zigzag_balances_the_causal_work():
    """Scan work of a query chunk grows with its index; with the zigzag every
    rank's total is within one block's worth of the mean."""
    L, world = 32768, 8
    N = L // 128
    work = []
    for r in range(world):
        rows = pa.path_attn_cp_rows(1, 1, L, world, r)
        chunks = sorted(set((rows // 128).tolist()))
        work.append(sum(chunks))
    assert max(work) - min(work) <= 2 * math.ceil(N / (2 * world))


def test_sizes_and_rejections():
    B, H, L = 2, 3, 1000
    for world in (1, 2, 5):
        nb = math.ceil(math.ceil(L / 128) / (2 * world))
        assert pa.path_attn_cp_exchange_bytes(B, H, L, world) == 3 * B * H * 2 * nb * 128 * 128 * 2
    with pytest.raises(pa.PathAttnError):
        pa.path_attn_cp_local_len(B, H, L, 2, 2)  # rank outside [0, world)
    bad = pa.PrefillDesc(B, H, L, 64, pa.PATH_BF16, 0.125, 0)  # head_dim 64
    assert pa.load_library().path_attn_cp_workspace_size(bad, 2) == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, L, BH, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import dependent_positional_attention_gb300 as pa

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        N = math.ceil(L / 128)
        nb = math.ceil(N / (2 * ws))
        Lq = 2 * nb * 128
        rows = pa.path_attn_cp_rows(1, BH, L, ws, rank)
        # a stand-in exchange block: section s, head h, local row l, lane j holds
        # a code of (section, head, global position) instead of Kh / Pm / V
        blk = torch.full((3, BH, Lq, 128), -1.0, dtype=torch.float64)
        for s in range(3):
            for h in range(BH):
                blk[s, h, :len(rows), :] = (s * 1e7 + h * 1e5 + rows.double()).unsqueeze(1)
        gathered = pa.cp_all_gather(blk.reshape(-1), ws).reshape(ws, 3, BH, Lq, 128)
        # the scan reads chunk c of head h from owner r = block or 2ws-1-block,
        # local chunk index (block < ws ? 0 : nb) + c % nb
        bad = 0
        for c in range(N):
            blkc = c // nb
            owner = blkc if blkc < ws else 2 * ws - 1 - blkc
            idx = (0 if blkc < ws else nb) + c - blkc * nb
            for s in range(3):
                for h in range(BH):
                    tile = gathered[owner, s, h, idx * 128:(idx + 1) * 128]
                    n = min(128, L - c * 128)
                    want = s * 1e7 + h * 1e5 + torch.arange(c * 128, c * 128 + n).double()
                    bad += int(not torch.equal(tile[:n, 0], want))
                    bad += int(not torch.equal(tile[:n, 127], want))
        dist.barrier()
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            f.write("%d %d\n" % (len(rows), bad))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws,L", [(2, 1000), (3, 1300)])
def test_exchange_blocks_gathered_where_the_scan_reads_them(tmp_path, ws, L):
    port = _free_port()
    BH = 2
    mp.start_processes(_rank_main, args=(ws, port, L, BH, str(tmp_path)), nprocs=ws, join=True,
                       start_method="spawn")
    total = 0
    for r in range(ws):
        n, bad = map(int, open(tmp_path / ("rank%d.txt" % r)).read().split())
        assert bad == 0, (r, bad)
        total += n
    assert total == L
