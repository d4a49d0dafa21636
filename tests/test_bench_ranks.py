"""The multi-process side of bench.py on CPU: two gloo ranks (the launch a
torchrun run makes, one process per GPU) agree on the slowest rank's times,
and only rank 0 of the reference arm reports."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # rank r measured (1 + r) ms per step and (10 - r) ms end to end
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank], "cpu")
        out.put((rank, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_time():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get() for _ in range(2))
    assert res[0] == res[1] == [2.0, 10.0]


def test_single_process_is_a_copy():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1.25]) == [3.5, 1.25]


def test_reference_arm_reports_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 1, 0
    assert bench.run_reference(Args(), rank=1, world=2) is None


def test_oracle_clock_times_every_piece_and_extrapolates():
    """The reference arm's clock on a small global layer and sampler: every
    piece gets a time, the estimate is positive and grows with the rows it
    extrapolates to."""
    sys.path.insert(0, ROOT)
    import bench
    import canvas_workloads as wl
    a = wl.make_attention_inputs(wl.AttnConfig("clk", B=1, C=8, prefix=(40,), D=64, Hq=2, Hkv=1, d=64,
                                               layer="global", window=0, theta=1e6, rotary_fraction=0.25,
                                               dtype="bf16", seed=1, page_tokens=64))
    s = wl.make_sample_inputs(wl.SampleConfig("clk", rows=4, C=4, V=40000, D=16, dtype="bf16", seed=2, step=0,
                                              bound=0.3, logits="normal"))
    clock = bench.OracleClock(a, s)
    assert clock.n_chunks == 3 and len(clock.pieces) == 6
    for i, piece in enumerate(clock.pieces):
        assert clock.run(piece, i) >= 0.0
    est = clock.estimate()
    assert est > 0.0
    clock.t["stats"] += 1.0       # one more second per position: 4 positions
    assert abs(clock.estimate() - est - 4.0) < 1e-9
    assert "rotation" in clock.describe() and "every piece once" in clock.describe(rotating=False)
