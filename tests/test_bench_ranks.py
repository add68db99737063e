"""Multi-process logic of the benchmark on CPU (gloo, world size 2): the path shards by
(batch, head) with no data-path exchange, so N processes run N replicas; the timed region is
bracketed by barriers, the time is the maximum over ranks and the value counts every rank's
units.  The reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    R = bench.Ranks()
    R.init_cpu()
    R.barrier()
    ms = R.max(10.0 + 5.0 * rank)           # rank 1 is the slower replica
    value = bench.whole_job_value(R.world, 1000, ms)
    R.barrier()
    R.close()
    q.put((rank, ms, value))


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in got:
        assert ms == 15.0, "every rank sees the slowest rank's time"
        assert value == pytest.approx(2 * 1000 / 0.015), "the value counts the units of both replicas"


def test_single_process_is_its_own_world(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    R = bench.Ranks()
    R.init_cpu()
    assert R.world == 1 and R.rank == 0 and R.max(3.0) == 3.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun the other ranks exit 0 at once, without work and without output."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1"])
    assert bench.run_reference(bench.parse_args()) == 0
    assert capsys.readouterr().out == ""


def test_chunk_mode_cpu_baseline_times_the_oracle_rule():
    """The chunk-mode line's CPU baseline runs the oracle's chunk-granular rule on a bounded
    sample of heads and reports token-equivalents per second on one thread."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import synth
    w = synth.Workload("tiny_chunk", 1, 2, 96, 8, 8, 16, 8, 16, "bf16", "gauss")
    x = synth.make_inputs(w)
    cpu = bench.cpu_baseline_chunk(x, w, heads=3)
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["unit"] == "tokens/s"
    assert cpu["value"] > 0 and "2 of 2 heads" in cpu["sample"]


def test_head_slices_cover_every_head_once():
    """The contiguous head slices of every world size cover [0, total) once, in rank order;
    with world * B * Hh heads, rank r's slice is its own batch block [r B Hh, (r + 1) B Hh)."""
    for total in (1, 5, 8, 128, 257):
        for world in (1, 2, 3, 4, 8):
            owned = []
            for r in range(world):
                lo, hi = bench.head_slice(total, world, r)
                assert 0 <= lo <= hi <= total
                owned.extend(range(lo, hi))
            assert owned == list(range(total))
    for world in (1, 2, 4, 8):
        for B, Hh in ((1, 8), (4, 32), (64, 32)):
            for r in range(world):
                assert bench.head_slice(world * B * Hh, world, r) == (r * B * Hh, (r + 1) * B * Hh)


def _shard_worker(rank, world, port, q):
    """Each rank runs the oracle on its own slice of the heads of one small workload and the
    slices are gathered back into head order."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import synth
    from oracle import inc
    x = synth.gauss_inputs(1, 5, 40, 8, 8, "bf16", seed=31)
    R = bench.Ranks()
    R.init_cpu()
    lo, hi = bench.head_slice(5, R.world, R.rank)
    flat = lambda a: a.reshape(5, *a.shape[2:])[lo:hi]  # noqa: E731
    out = inc.run(flat(x.q), flat(x.k), flat(x.v), x.W, 6, 4, "bf16", nthreads=1)
    Y = R.gather_heads(out["Y"], 5)
    wpos = R.gather_heads(out["write_pos"].astype(np.int64), 5)
    R.barrier()
    R.close()
    q.put((rank, (lo, hi), Y, wpos))


def test_sharded_heads_reassemble_in_order():
    """Two gloo ranks, each with a contiguous slice of 5 heads (3 + 2): the gathered outputs
    and decision logs equal one process running every head."""
    import numpy as np
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import synth
    from oracle import inc
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_shard_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((q.get(timeout=180) for _ in range(world)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    x = synth.gauss_inputs(1, 5, 40, 8, 8, "bf16", seed=31)
    whole = inc.run(x.q.reshape(5, 40, 8), x.k.reshape(5, 40, 8), x.v.reshape(5, 40, 8), x.W, 6, 4, "bf16",
                    nthreads=1)
    assert [g[1] for g in got] == [(0, 3), (3, 5)]
    for _, _, Y, wpos in got:
        np.testing.assert_array_equal(Y, whole["Y"])
        np.testing.assert_array_equal(wpos, whole["write_pos"])


def test_traffic_figures_bind_to_the_kernel_sources(monkeypatch):
    """A DRAM-traffic figure is reported only for the kernel sources it was captured on: the
    digest of the named files must match, else the figure is null."""
    import bench
    files = ["lola_hola.cu", "lola_internal.cuh"]
    good = bench.sources_digest(files)
    monkeypatch.setitem(bench.NCU_TRAFFIC, ("k", "w"), {"sources": files, "digest": good, "bytes_per_launch": 5.0})
    assert bench.traffic("k", "w") == 5.0
    monkeypatch.setitem(bench.NCU_TRAFFIC, ("k", "w"), {"sources": files, "digest": "0" * 16, "bytes_per_launch": 5.0})
    assert bench.traffic("k", "w") is None
    assert bench.traffic("no such kernel", "w") is None
