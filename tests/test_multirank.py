"""Multi-rank host logic of bench.py on CPU (gloo, world_size 2).

The decode path shards by replica: every rank runs the whole workload on its
own GPU with its own seeded inputs and no collective on the data path. The
only cross-rank steps are the barrier around the timed region and the
max-over-ranks of the elapsed time, which these tests run on the gloo
backend. The reference arm is run under torchrun with two ranks: rank 0
alone prints its line and the other rank exits without work.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, result_dir):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import mla_inputs as mi

    env_ws, env_rank, env_local = bench.dist_env()
    bench.init_dist(env_ws, "gloo")
    bench.barrier(env_ws)
    # per-rank elapsed times: the whole job is as slow as its slowest rank
    ms = [3.0, 5.0, 4.0, 1.0][rank]
    ms_max = bench.max_over_ranks(ms, env_ws, "cpu")
    # each rank builds its own replica of a small workload from its own seed
    w = mi.WORKLOADS["bf16_b4_l1024"]
    inp = [mi.make_workload(w, seed_offset=bench.replica_seed_offset(env_rank, k)) for k in range(2)]
    again = mi.make_workload(w, seed_offset=bench.replica_seed_offset(env_rank, 0))
    fp = [float(x.q.float().sum()) for x in inp]
    reproducible = bool(torch.equal(inp[0].q, again.q) and torch.equal(inp[0].kv, again.kv)
                        and torch.equal(inp[0].kv_indices, again.kv_indices))
    same_shape = list(inp[0].kv_indptr.tolist())
    fps = [None] * env_ws
    torch.distributed.all_gather_object(fps, fp)
    bench.barrier(env_ws)
    torch.distributed.destroy_process_group()
    with open(os.path.join(result_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ws": env_ws, "rank": env_rank, "local": env_local, "ms_max": ms_max, "fps": fps,
                   "reproducible": reproducible, "indptr": same_shape}, f)


def test_two_ranks_barrier_max_and_independent_replicas(tmp_path):
    ws = 2
    mp.start_processes(_rank_main, args=(ws, _free_port(), str(tmp_path)), nprocs=ws, start_method="spawn",
                       join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(ws)]
    for r, d in enumerate(res):
        assert (d["ws"], d["rank"], d["local"]) == (ws, r, r)
        assert d["ms_max"] == 5.0  # max over ranks, seen identically by every rank
        assert d["reproducible"]
        assert d["fps"] == res[0]["fps"]  # every rank gathered the same view
    # same shapes on every rank, different data: independent replicas
    assert res[0]["indptr"] == res[1]["indptr"]
    fps = res[0]["fps"]
    assert len({x for pair in fps for x in pair}) == 4


def test_whole_job_value_counts_every_rank():
    import bench
    one = bench.whole_job_gbs(304_218_112, 100, 1, 6.6)
    two = bench.whole_job_gbs(304_218_112, 100, 2, 6.6)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(304_218_112 * 100 / 6.6e-3 / 1e9)
    # a slower rank lowers the whole-job figure
    assert bench.whole_job_gbs(304_218_112, 100, 2, 8.0) < two
    assert bench.replica_seed_offset(0, 0) != bench.replica_seed_offset(1, 0)
    assert bench.replica_seed_offset(0, 1) != bench.replica_seed_offset(1, 0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1",
           "--workload", "bf16_b4_l1024"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert np.isfinite(d["ms_per_step"])


def test_bench_layout_option():
    import bench
    assert bench.parse_layout("rows") == ("rows", 1, False)
    assert bench.parse_layout("rows:shuffled") == ("rows", 1, True)
    assert bench.parse_layout("pages:64") == ("pages", 64, False)
    assert bench.parse_layout("pages:8:shuffled") == ("pages", 8, True)
    for bad in ("pages", "pages:0", "pages:x", "rows:3", "pages:8:sorted", "grid"):
        with pytest.raises(SystemExit):
            bench.parse_layout(bad)
