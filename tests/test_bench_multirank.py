"""bench.py's multi-process logic on CPU ranks (gloo, world size 2): the timed
region is the slowest rank's, the value counts every rank's bytes, and the
reference arm prints from rank 0 only."""
import os
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sec = [0.010, 0.025][rank]
        m = bench.max_over_ranks(sec, dist, "cpu")
        out[rank] = (m, bench.job_gbs(world, 100, 1_000_000, m))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    port = 29500 + (os.getpid() % 1000)
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 0.025
    assert abs(res[0][1] - 2 * 100 * 1_000_000 / 0.025 / 1e9) < 1e-9


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5) == 0.5
    assert bench.job_gbs(1, 10, 2_000_000_000, 2.0) == 10.0


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_both_arms_name_the_same_config_and_bytes():
    # the reference arm and the GPU arm print one config dict for a workload,
    # and the algorithmic bytes follow each input read once and each output
    # written once
    sys.path.insert(0, ROOT)
    import bench
    from row_wise_normalization_reduce_gb300 import workloads as W
    for w in W.ALL:
        assert bench.workload_config(w, 1) == bench.workload_config(w, 1)
        assert bench.workload_config(w, 1)["workload"] == w.name
    w = W.ADD_RMS_BF16_4096x4096
    assert bench.algorithmic_bytes(w) == 4 * 4096 * 4096 * 2 + 4096 * 2 + 4096 * 4
    w = W.LN_BF16_4096x4096
    assert bench.algorithmic_bytes(w, stats=False) == 2 * 4096 * 4096 * 2 + 2 * 4096 * 2
    w = W.BN_F32_32x64x56x56
    assert bench.algorithmic_bytes(w) == 2 * 32 * 64 * 56 * 56 * 4 + 2 * 64 * 4 + 6 * 64 * 4
    w = W.BN_BF16_32x64x56x56  # 16-bit x, y, gamma, beta; binary32 statistics
    assert bench.algorithmic_bytes(w) == 2 * 32 * 64 * 56 * 56 * 2 + 2 * 64 * 2 + 6 * 64 * 4


def test_reference_arm_line_matches_gpu_arm_keys():
    # the reference arm's JSON line (rank 0, CPU only): impl, the shared
    # config, and an e2e object with zero host<->device bytes
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "ln_f32_64x1024", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    import json
    line = json.loads(r.stdout.strip().splitlines()[-1])
    sys.path.insert(0, ROOT)
    import bench
    from row_wise_normalization_reduce_gb300 import workloads as W
    assert line["impl"] == "reference"
    assert line["config"] == bench.workload_config(W.LN_F32_64x1024, 1)
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
