"""The bench's N > 1 path on CPU: world-size-2 ranks over gloo (the same torch.distributed calls the
GPU runs make over NCCL) and the reference arm under torchrun.  The layer shards by tokens with no
exchange, so the only cross-rank steps are the barrier and the max-over-ranks timing."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    W, r, _ = bench.world()
    ms = bench.max_over_ranks(1.5 + rank)            # rank 1 is the slow replica
    value = bench.job_tokens_per_s(W, 8, ms)
    dist.barrier()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": W, "ms": ms, "value": value}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["world"] == 2
        assert r["ms"] == 2.5                        # the slowest rank's time, seen by every rank
        assert abs(r["value"] - 2 * 8 / 2.5e-3) < 1e-6   # both ranks' tokens over that time


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_tokens_per_s(1, 8, 0.2) == 8 / 0.2e-3


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2", "--impl", "reference",
           "--workload", "tiny", "--steps", "2", "--warmup", "1", "--ref-seconds", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=280, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1                           # rank 0 alone runs and prints; rank 1 exits without work
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_launch_counts_match_the_measured_launch_lists():
    # kernels per forward as counted in the committed ncu launch lists (decode: 3; batched: 7;
    # prefill: 8; INT8 decode: 7) and the tiny-batch path's two launches
    import dataclasses
    sys.path.insert(0, ROOT)
    import bench
    import synth
    W = synth.WORKLOADS
    assert bench.launches_per_forward(W["decode"]) == 3
    assert bench.launches_per_forward(W["batched"]) == 7
    assert bench.launches_per_forward(W["prefill"]) == 8
    assert bench.launches_per_forward(dataclasses.replace(W["decode"], fmt="int8")) == 7
    assert bench.launches_per_forward(W["decode"], naive=True) == 2
    # NVFP4: two launches (bf16 rows, GEMM) for each of L1 and L2; the permute copies nothing (the
    # L1 conversion reads the token-order rows)
    assert bench.launches_per_forward(W["skewed"]) == 3 + 2 + 4 + 1
