"""The multi-rank path of bench.py on CPU with gloo, world size 2.

The layer step shards by batch: every rank runs its own batch and the only
cross-rank operations are the barrier around the timed region and the max of
the per-rank times.  These tests run those pieces in two gloo processes, and
the reference arm under torchrun, where rank 0 alone prints its line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    class A:
        pass

    w, r, _ = bench.dist_init(A())
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + rank, w)  # rank-dependent times: the slowest rank wins
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 11.0, 1: 11.0}


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "switch_tiny_f32"]
    out = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
    # the line carries the contract's keys, with the arm's own metric and workload
    for key in ("metric", "unit", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
                "dtype", "data", "config", "cpu_baseline"):
        assert key in rec, key
    assert rec["config"]["workload"] == "switch_tiny_f32" and rec["higher_is_better"] is True
    # the same config dict as the GPU arm builds for this workload, key for key
    sys.path.insert(0, ROOT)
    import bench
    from routing_permute_grouped_router_gb300 import workload as W

    assert rec["config"] == bench.workload_config("switch_tiny_f32", W.WORKLOADS["switch_tiny_f32"])
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["e2e"]["value"] == rec["value"] and rec["e2e"]["unit"] == rec["unit"]
