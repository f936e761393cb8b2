"""The bench's multi-rank logic on CPU: two gloo ranks (the path shards into
independent replicas, so the only exchange is the timing reduction).  Each rank
reports a different time; both must see the slowest, and the whole-job value
counts the bytes of every rank over that time.  The reference arm runs on rank
0 only."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank                     # rank 1 is the slow one
        t = bench.max_over_ranks(local_ms, dist, "cpu")
        out[rank] = (t, bench.whole_job_gbs(1000000, world, 4, t * 1e-3))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 4 steps x 1 MB in 15 ms
    assert res[0][1] == pytest.approx(2 * 4 * 1e6 / 15e-3 / 1e9)


def test_single_process_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_gbs(10 ** 9, 1, 1, 1.0) == pytest.approx(1.0)


def test_reference_arm_other_ranks_exit_quietly(capsys):
    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""


def test_algorithmic_bytes_match_the_roofline_table():
    """The bytes the roofline divides by, worked by hand from the layout: 4-bit
    4 bits + an FP16 scale / 32 + a 4-bit zero / 32 per weight, 2-bit 2 bits +
    FP16 S and Z / 32, outliers 4 B of index + 2 B per row, FP16 x in, FP16 y out."""
    assert bench.algorithmic_bytes("w4", 4096, 4096, 0) == 4096 * 4096 * 37 // 64 + 2 * 4096 + 2 * 4096
    assert bench.algorithmic_bytes("w4", 4096, 4096, 0) == 9715712
    assert bench.algorithmic_bytes("w2", 4096, 4096, 143) == 4096 * 4096 * 3 // 8 + 143 * (4 + 2 * 4096) + 4 * 4096
    assert bench.algorithmic_bytes("w4", 14336, 4096, 0, M=4) == 14336 * 4096 * 37 // 64 + 2 * 4096 * 4 + 2 * 14336 * 4
    layer = sum(bench.algorithmic_bytes("w4", N, K, 0) for N, K in
                ((4096, 4096), (1024, 4096), (1024, 4096), (4096, 4096), (14336, 4096), (14336, 4096), (4096, 14336)))
    assert layer == 126255104
