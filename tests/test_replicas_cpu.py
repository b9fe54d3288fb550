"""The multi-GPU path of bench.py on CPU: two gloo ranks. The decode path
does not shard (replicas only), so what N > 1 adds is host logic: the
max-over-ranks reduction of the timings, and rank 0 alone running and
printing the reference arm."""
import io
import os
import socket
import sys
import contextlib

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, -rank], torch.device("cpu"))
    # the reference arm: every rank but 0 returns at once and prints nothing
    buf = io.StringIO()
    args = bench.argparse.Namespace(impl="reference", gpus=world, steps=1, warmup=0,
                                    workload="tiny_f32_ctx256", no_cpu_baseline=True,
                                    no_other=True)
    rc = None
    if rank != 0:
        with contextlib.redirect_stdout(buf):
            rc = bench.run_reference(args)
    out.put((rank, got, rc, buf.getvalue()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rc, text in res:
        assert got == [2.0, 10.0, 0.0], got
        if rank != 0:
            assert rc == 0 and text == ""


def test_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks([3, 4.5], torch.device("cpu")) == [3.0, 4.5]


def test_reference_arm_times_whole_oracle_steps(capsys):
    """Rank 0 alone: each timed step is one whole oracle step, so the
    reported time per step times the step count fits inside the run."""
    import json
    import bench
    args = bench.argparse.Namespace(impl="reference", gpus=1, steps=3, warmup=1,
                                    workload="tiny_f32_ctx256", no_cpu_baseline=True,
                                    no_other=True)
    assert bench.run_reference(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "us/step"
    assert line["ms_per_step"] * line["steps"] / 1e3 <= line["wall_s"]
    assert line["cpu_baseline"]["value"] == line["value"] == line["e2e"]["value"]
