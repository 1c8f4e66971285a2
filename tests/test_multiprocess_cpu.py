"""The multi-process plumbing of the benchmark on the host: two ranks over gloo
(the GPU runs use one process per GPU over NCCL, replicas only, with the
collective carrying nothing but the slowest rank's time).

Covers: the max over ranks, the barrier, the whole-job throughput of the
replicas, the reference arm's silent non-zero ranks, and a rank that never
reaches the barrier making the other fail within the process-group timeout
(failure detected on the host, no GPU involved).
"""
import datetime
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, mode, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    if mode == "plumbing":
        w, r, _ = bench.dist_setup(None, backend="gloo")
        assert (w, r) == (world, rank)
        bench.barrier(w)
        m = bench.dist_max(10.0 + 5.0 * rank, w)
        v = bench.aggregate_tflops(w, 1e12, 10, m)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
            json.dump({"max": m, "value": v}, fh)
        dist.destroy_process_group()
    elif mode == "dead_rank":
        dist.init_process_group("gloo", timeout=datetime.timedelta(seconds=4))
        if rank == 1:
            os._exit(0)  # leaves between steps, never reaches the barrier
        err = ""
        try:
            dist.barrier()
        except Exception as exc:  # the survivor learns of it on the host
            err = type(exc).__name__
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
            json.dump({"error": err}, fh)
        os._exit(0)


def _spawn(mode, tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, 2, port, mode, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert not p.is_alive(), "a rank hung"
    return procs


def test_two_ranks_take_the_slowest_time_and_count_both_replicas(tmp_path):
    procs = _spawn("plumbing", tmp_path)
    assert all(p.exitcode == 0 for p in procs)
    out = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert out[0]["max"] == out[1]["max"] == 15.0
    # 2 replicas x 1 TFLOP x 10 steps in the slower rank's 15 ms
    assert out[0]["value"] == pytest.approx(2 * 1e12 * 10 / 0.015 / 1e12)


def test_a_rank_that_never_joins_fails_the_other_on_the_host(tmp_path):
    _spawn("dead_rank", tmp_path)
    out = json.load(open(tmp_path / "r0.json"))
    assert out["error"], "the surviving rank did not see the missing one"


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "1", "--reference-seconds", "2", "--workload", "mlp_tp2_t512"],
                       capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0"))
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 1
    assert line["config"]["workload"] == "mlp_tp2_t512" and line["unit"] == "TFLOP/s" and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_default_workload_is_the_largest_single_gpu_layer():
    """With no flags the bench times the prefill decoder layer (T=4096, D=8192,
    64 q / 8 kv heads, F=28672, TP=8) with the one-pass ring combine."""
    sys.path.insert(0, ROOT)
    import bench
    old = sys.argv
    try:
        sys.argv = ["bench.py"]
        args = bench.parse_args()
    finally:
        sys.argv = old
    assert args.workload == "prefill_layer_tp8_t4096" and args.combine is None and args.gpus == 1
