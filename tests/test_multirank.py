"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each with
its own replica time, agree on the job time (the slowest rank) and on the
whole-job throughput.  The data path has no collective (each rank runs an
independent replica), so this reduction is the only exchange."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank  # rank 1 is slower
    job_ms = bench.max_over_ranks(ms, world)
    out.put((rank, job_ms, bench.job_value(bench.STEP_FLOPS, job_ms, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_job_time():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, v0), (r1, ms1, v1) = res
    assert ms0 == ms1 == 15.0
    assert v0 == v1 == pytest.approx(2 * 7.696581394432e12 / 15e-3 / 1e12)


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference (the float64 oracle on host cores) keeps the
    JSON contract."""
    import json
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["cpu_baseline"]["kind"] == "oracle"
    assert j["value"] > 0 and j["e2e"]["h2d_bytes_per_step"] == 0
