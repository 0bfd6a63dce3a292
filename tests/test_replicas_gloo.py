"""The multi-GPU path is replicas only: every rank runs the whole workload on
its own GPU, with no exchange on the data path.  These CPU tests run the host
logic of that path as world-size-2 gloo process groups: the job time is the
slowest rank's, the throughput counts every rank's work, and the reference
arm prints from rank 0 only."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r'''
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo", rank=rank, world_size=world)
own = 100.0 + 50.0 * rank                    # each replica's own timed total (ms)
total = bench.slowest_rank_ms(own, world, "cpu")
dist.barrier()
print(json.dumps({{"rank": rank, "total": total,
                   "value": bench.job_throughput(1e9, 10, total, world)}}), flush=True)
dist.destroy_process_group()
'''


def _launch(code, world, port):
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world))
    procs = []
    for r in range(world):
        e = dict(env, RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, "-c", code], env=e, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, err = p.communicate(timeout=120)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(o)
    return outs


def test_job_time_is_the_slowest_replica():
    outs = _launch(WORKER.format(root=ROOT), 2, 29511)
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o in outs), key=lambda d: d["rank"])
    assert [d["total"] for d in res] == [150.0, 150.0]
    # 2 ranks x 1e9 MACs x 10 steps over 0.15 s
    assert all(abs(d["value"] - 2 * 1e9 * 10 / 0.15 / 1e9) < 1e-6 for d in res)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(123.0, 1, "cpu") == 123.0
    assert bench.job_throughput(5e8, 4, 1000.0, 1) == pytest.approx(2.0)


def test_reference_arm_prints_from_rank_zero_only():
    """Rank 1 of the reference arm does no work and prints nothing."""
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench, argparse; "
            "a = argparse.Namespace(workload='mlp', steps=1, warmup=0, gpus=2); "
            "bench.reference_arm(a, 1)")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
