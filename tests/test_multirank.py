"""The data-parallel path on several ranks, on the CPU with gloo (world size
2): each rank decodes its own batch with no collective on the data path, and
the bench reduces only its timings, taking the slowest rank's time and the
whole job's FLOPs.  The reference arm runs on rank 0 alone."""
import contextlib
import io
import multiprocessing as mp
import os
import socket

import pytest

import bench
from mla_latent_decode_gb300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        # ranks time different spans; every rank gets the slowest
        t = bench.slowest_rank(1.5 + 2.0 * rank, dist, "cpu")
        # each rank's batch is its own (seeded by rank): different data
        wl = synth.Workload("mr", 2, 5, 16, [300, 70])
        b = synth.make_batch(wl, seed=rank, device="cpu")
        head = b.q_nope.flatten()[:8].float().tolist()
        q.put((rank, r, w, local, t, head))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings_only():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, local, t, _ in out:
        assert (r, w, local) == (rank, world, rank)
        assert t == 3.5  # the slower rank's 1.5 + 2.0
    assert out[0][5] != out[1][5]  # independent batches per rank
    # job throughput: both ranks' work in the slowest rank's time
    assert bench.job_tflops(2e12, 10, world, 2.0) == pytest.approx(20.0)
    assert bench.slowest_rank(0.25) == 0.25  # one rank: no process group


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun every rank starts bench.py --impl reference; rank 1
    exits 0 at once and prints nothing."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.parse(["--impl", "reference", "--gpus", "2", "--steps", "1",
                             "--warmup", "0", "--config", "tiny"])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    assert buf.getvalue() == ""
