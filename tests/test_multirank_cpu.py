"""The multi-rank host logic of bench.py on the CPU, two gloo ranks: heads
are independent, so N GPUs run N replicas of the workload with no exchange on
the data path; what the ranks share is the step time (the maximum over
ranks, one all-reduce) and, for the reference arm, rank 0 alone runs and
prints."""
import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], world)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_step_time_is_max_over_two_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, [1.25, 3.5], out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(2.0, 1) == 2.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the reference arm's other ranks exit without work."""
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    calls = []
    monkeypatch.setattr(bench, "_oracle_sample", lambda *a, **k: calls.append(a) or (1.0, 1.0))
    assert bench.main(["--gpus", "2", "--impl", "reference", "--steps", "1", "--warmup", "0"]) is None
    assert calls == [] and capsys.readouterr().out == ""


def test_gpus_flag_must_match_the_launched_ranks(monkeypatch, capsys):
    """--gpus N is honoured, not ignored: a run whose launcher started a
    different number of ranks stops before any work (exit status 2), so a
    replicas run cannot be reported under the wrong GPU count."""
    import pytest

    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "2", "--impl", "reference", "--steps", "1"])
    assert e.value.code == 2
    assert "--nproc-per-node 2" in capsys.readouterr().err
    assert bench.check_world(1, {}) == 1
    assert bench.check_world(4, {"WORLD_SIZE": "4"}) == 4
    with pytest.raises(SystemExit):
        bench.check_world(8, {"WORLD_SIZE": "2"})
