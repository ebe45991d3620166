"""The benchmark's multi-GPU host logic on CPU ranks (gloo, world size 2).

Decode requests are independent units, so ranks share nothing on the data
path: each runs its own batch, and the only collectives are the timing
barrier and a MAX over ranks of the step time.  These tests run that host
logic in two processes without a GPU.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synth  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [0.25, 0.40][rank]                # the second rank is slower
    ms = bench.max_over_ranks(local_ms, world, "cpu")
    dist.barrier()
    wl = synth.make("c0", seed=bench.rank_seed("c0", rank))
    out.put((rank, ms, bench.whole_job_rate(world, wl.n_q, ms), wl.q_idx.tobytes()[:64],
             wl.q_idx.shape))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, v0, b0, s0), (r1, ms1, v1, b1, s1) = res
    assert ms0 == ms1 == 0.40                     # every rank reports the slowest step
    assert v0 == v1 == 2 * 256 / 0.40e-3          # both ranks' rows over that time
    assert s0 == s1 and b0 != b1                  # same shapes, independent data


def test_single_rank_needs_no_collective():
    assert bench.max_over_ranks(0.3, 1, "cpu") == 0.3
    assert bench.whole_job_rate(1, 64, 0.128) == pytest.approx(500000.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the oracle arm runs on rank 0; other ranks exit at once
    without output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
