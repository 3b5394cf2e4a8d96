"""The N>1 bench path on CPU: two gloo ranks exercise the barrier, the
max-over-ranks timing and the sum-over-ranks work count that bench.py uses
under torchrun (the path runs independent replicas, so these are its only
cross-rank steps), and the reference arm's rank-0-only rule."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    bench.dist_init(world, "gloo")
    bench.barrier(world)
    ms = 2.0 + rank  # rank 1 is slower
    flops = 1e12 * (rank + 1)
    t = bench.max_over_ranks(ms, world, "cpu")
    f = bench.sum_over_ranks(flops, world, "cpu")
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
        json.dump({"max_ms": t, "sum_flops": f}, fh)
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        res = json.load(open(tmp_path / f"r{r}.json"))
        assert res["max_ms"] == 3.0
        assert res["sum_flops"] == 3e12


@pytest.mark.parametrize("rank", [1])
def test_reference_arm_non_zero_rank_does_no_work(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "c1_contig_g2_m100_n256_k256", "--steps", "3",
                          "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "c1_contig_g2_m100_n256_k256", "--steps", "3",
                          "--warmup", "3", "--reference-seconds", "2"], env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0
