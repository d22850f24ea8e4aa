"""Host logic of bench.py's N > 1 path on CPU: two gloo ranks (replicas only --
the path has no data exchange), barrier, max-over-ranks timing and the
whole-job aggregate."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.dist_init(w, "gloo")
    try:
        bench.dist_barrier(w)
        # each replica processed the same units; rank 1 was slower
        elapsed = 2.0 if rank == 1 else 1.0
        slowest = bench.dist_max(elapsed, w)
        out[rank] = (slowest, bench.aggregate(w * 100.0, slowest))
        bench.dist_barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        if any(c is None for c in codes):
            for p in procs:
                p.kill()
            pytest.fail("a gloo rank did not finish")
        assert codes == [0, 0]
        res = dict(out)
    # max over ranks, and units of all ranks over that time
    assert res[0] == res[1] == (2.0, 100.0)


def test_single_process_defaults():
    import bench
    assert bench.dist_max(3.5, 1) == 3.5
    assert bench.aggregate(10.0, 4.0) == 2.5


def test_reference_arm_prints_the_contract_line(capsys):
    """bench.py --impl reference runs the CPU oracle (no GPU needed) and
    prints one JSON line with the contract's keys."""
    import json

    import bench
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1"]) in (0, None)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
