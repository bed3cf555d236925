"""Multi-process host logic on CPU (gloo, world size 2): the independent units
of a batch are split across ranks with no overlap and no gap, and the
benchmark's max-over-ranks timing reduction sees every rank.  The data path
itself has no collective: each rank relocates its own requests."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, n_units, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth

    mine = list(synth.shard(n_units, rank, world))
    got = [None] * world
    dist.all_gather_object(got, mine)
    t = bench.max_over_ranks(1.0 + rank, world)
    dist.barrier()
    if rank == 0:
        q.put((got, t))
    dist.destroy_process_group()


@pytest.mark.parametrize("n_units", [0, 1, 7, 32])
def test_shards_cover_units_once(n_units):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, n_units, q)) for r in range(2)]
    for p in procs:
        p.start()
    got, t = q.get(timeout=120)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    flat = [u for part in got for u in part]
    assert sorted(flat) == list(range(n_units))
    assert abs(len(got[0]) - len(got[1])) <= 1
    assert t == 2.0


def test_oracle_on_every_core_counts_every_unit():
    """The CPU baseline's process pool: each of its processes relocates its own
    independent sample behind one barrier, and the round reports every token."""
    import bench

    cores = bench.OracleCores(2)
    try:
        ntok, dt, what = cores.run("relocate-mla", 16, 3)
    finally:
        cores.close()
    assert ntok == 32 and dt > 0 and "16-token" in what


@pytest.mark.parametrize("kind,n", [("relocate-mla", 16), ("sweep-mla", 1),
                                    ("relocate-gqa-patch", 1), ("splice-mla-128k", 1024),
                                    ("splice-mla-4k", 0)])
def test_every_cpu_baseline_sample_runs_and_counts_its_units(kind, n):
    """Each workload's oracle sample runs and reports the metric's units of
    one call: tokens relocated, or rows moved by the splice (downstream rows
    plus stub rows)."""
    import bench

    call, units, what = bench.oracle_sample(kind, n, 5)
    call()
    if kind == "splice-mla-4k":
        assert units == 4096 - 2048 + 16
    elif kind == "relocate-mla":
        assert units == n
    assert units > 0 and what


def test_default_sequence_ends_with_the_headline():
    import bench

    assert bench.DEFAULT_SEQUENCE[-1] == "relocate-mla"
    for name in bench.DEFAULT_SEQUENCE:
        assert name in bench.WORKLOADS and name in bench.CPU_SAMPLES


def test_reference_arm_prints_one_complete_line(capsys):
    """bench.py --impl reference: the oracle on every host core, one JSON line
    with the contract's keys (no GPU needed)."""
    import json

    import bench

    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"]) == 0
    line = capsys.readouterr().out.strip().splitlines()[-1]
    d = json.loads(line)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
