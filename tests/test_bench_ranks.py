"""The bench's multi-rank host logic on CPU: two gloo ranks stand in for two
GPU replicas.  The job's time is the slowest rank's, the job's throughput is
every rank's bytes over that time, and only rank 0 of the reference arm runs."""
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    import datetime

    import torch.distributed as td
    td.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                          timeout=datetime.timedelta(seconds=60))
    try:
        t = bench.reduce_max(times[rank])
        v = bench.whole_job_gbs(world, 1_000_000_000, 10, t)
        q.put((rank, t, v))
        td.barrier()
    finally:
        td.destroy_process_group()


def test_reduce_max_and_whole_job_value_over_two_gloo_ranks():
    world, times = 2, [0.5, 2.0]
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    mp.start_processes(_rank_main, args=(world, _free_port(), times, q), nprocs=world, join=True,
                       start_method="spawn")
    got = sorted(q.get() for _ in range(world))
    for rank, t, v in got:
        # every rank sees the slowest rank's time ...
        assert t == max(times)
        # ... and the value counts both ranks' 10 GB over it
        assert v == pytest.approx(world * 10.0 / max(times))


def test_single_process_needs_no_group():
    assert bench.reduce_max(1.25) == 1.25
    assert bench.whole_job_gbs(1, 2_000_000_000, 3, 2.0) == pytest.approx(3.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, layers = 1, 0, 1

    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""


def test_oracle_steps_times_exactly_the_asked_steps():
    """The reference arm's stepping on a small shape: W untimed steps, then K
    timed ones over the prepared layer sets, reported in the bench's unit."""
    import synth
    r = bench.oracle_steps(synth.TINY, n_layers=3, steps=5, warmup=2, prepared=2)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["cores"] == 1
    assert r["value"] > 0 and r["s_per_step"] > 0
    assert r["sample"].startswith("5 timed steps") and "first 2 layer sets" in r["sample"]
