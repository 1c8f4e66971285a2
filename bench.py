#!/usr/bin/env python3
"""Benchmark of the tensor-parallel MLP block on GB300 (one JSON line on stdout).

One step = one pass of the block's hot path over one batch of synthetic input:
the shard plan (host), the column-parallel gate/up GEMM with the fused SwiGLU
for all ranks, the row-parallel down GEMM, and the ring all-reduce of the
per-rank partials. Default workload: Llama-style MLP, T=512 tokens, D=2048,
F=8192, TP=2, bf16 inputs with fp32 accumulation. Inputs are already resident in
HBM; several input sets (each a full weight copy) are rotated so that the
working set exceeds twice the L2 (no step reads another step's weights from L2).

`--impl reference` times the fp64 CPU oracle on the same workload instead (the
CPU baseline arm). Under torchrun every rank runs an independent replica on its
own GPU (the block itself lives on one device); the value is the total over
ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
COMBINE_NAMES = {"fused": 1, "ring": 2, "ring_fused": 3}
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", default="mlp_tp2_t512")
    p.add_argument("--combine", choices=sorted(COMBINE_NAMES), default="ring")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, ValueError, KeyError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---- workload accounting ------------------------------------------------------------
def mlp_flops(w) -> dict:
    T, D, F = w["T"], w["hidden"], w["ffn"]
    gate_up = 2.0 * T * D * 2 * F
    down = 2.0 * T * F * D
    return {"gate_up": gate_up, "down": down, "total": gate_up + down}


def ring_bytes(mode: str, n: int, size_bytes: int) -> int:
    """Algorithmic HBM bytes of one all-reduce of n partials of size_bytes each."""
    if n == 1 or mode == "fused":
        return 0
    if mode == "ring":
        return 3 * (n - 1) * size_bytes + 2 * (n - 1) * size_bytes
    return 2 * n * size_bytes  # ring_fused: each partial read once, every rank written once


def launches_per_step(mode: str, n: int) -> int:
    ring = {"ring": 2 * (n - 1), "ring_fused": 1, "fused": 0}[mode] if n > 1 else 0
    return 2 + ring


# ---- clocks -------------------------------------------------------------------------
class ClockSampler:
    def __init__(self, device_index: int, path: str):
        self.path, self.proc, self.dev = path, None, device_index

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={CLOCK_QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self) -> dict:
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons, n = [], None, set(), 0
        try:
            lines = open(self.path).read().strip().splitlines()
        except OSError:
            lines = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": n}


# ---- distributed plumbing (replicas only: NCCL carries only the timing max) ----------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- traffic from the committed ncu summary ------------------------------------------
def kernel_digest() -> str:
    h = hashlib.sha256()
    for f in ("gemm_tcgen05.cu", "sm100_ptx.cuh", "tp_internal.h"):
        with open(os.path.join(ROOT, "tensor_sharded_linear_gqa_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """dram bytes per launch of the gate/up GEMM from profiles/, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", f"gemm_gate_up_swiglu_{workload}.md")
    try:
        kv = {}
        for line in open(path):
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                kv[k.strip()] = v.strip().strip("`")
        if kv.get("kernel_source_digest") != kernel_digest():
            return None
        return int(float(kv["dram_bytes_per_launch"]))
    except (OSError, KeyError, ValueError):
        return None


# ---- CPU baseline (the oracle as it stands) --------------------------------------------
CPU_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, sys.argv[1])
import oracle as O
from tensor_sharded_linear_gqa_gb300 import inputs
w = dict(inputs.WORKLOADS[sys.argv[2]])
budget, max_reps, rows = float(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5])
d = inputs.make_bf16_inputs(w)
f = {k: inputs.bf16_bits_to_f64(v) for k, v in d.items()}
if rows <= 0:
    # size the per-pass row sample so that one pass takes about -rows/1000 seconds
    target = -rows / 1000.0
    t0 = time.perf_counter()
    O.mlp_sharded(f["x"][:32], f["wg"], f["wu"], f["wd"], w["tp"])
    t32 = max(time.perf_counter() - t0, 1e-4)
    rows = int(max(1, min(w["T"], 32 * target / t32)))
x = f["x"][:rows]
times = []
t_all = time.perf_counter()
while True:
    t0 = time.perf_counter()
    O.mlp_sharded(x, f["wg"], f["wu"], f["wd"], w["tp"])
    times.append(time.perf_counter() - t0)
    if time.perf_counter() - t_all >= budget or len(times) >= max_reps:
        break
print(json.dumps({"reps": len(times), "seconds": sum(times), "times": times, "rows": rows}))
"""


def cpu_oracle_run(workload: str, seconds: float, max_reps: int, rows: int) -> dict:
    """Runs the fp64 oracle MLP block in a child process on every core this process may use.
    rows > 0: that many token rows per pass; rows <= 0: sized so a pass takes -rows ms."""
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    out = subprocess.run([sys.executable, "-c", CPU_SNIPPET, ROOT, workload, str(seconds),
                          str(max_reps), str(rows)], capture_output=True, text=True, env=env,
                         timeout=1800)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    r = json.loads(out.stdout.strip().splitlines()[-1])
    r["cores"] = cores
    return r


def cpu_baseline(w, workload: str, seconds: float) -> dict:
    rows = w["T"]
    r = cpu_oracle_run(workload, seconds, 1000, rows)
    fl = mlp_flops(dict(w, T=r["rows"]))["total"]
    val = fl * r["reps"] / r["seconds"] / 1e12
    return {"value": round(val, 6), "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
            "sample": f"{r['reps']} full passes of the fp64 oracle MLP block (T={r['rows']}, "
                      f"D={w['hidden']}, F={w['ffn']}, TP={w['tp']}: column gate/up, SwiGLU, "
                      f"row down, ring all-reduce) in {r['seconds']:.1f} s"}


# ---- native arm ----------------------------------------------------------------------
def run_native(args):
    import numpy as np
    import torch

    import tensor_sharded_linear_gqa_gb300 as tp
    from tensor_sharded_linear_gqa_gb300 import inputs

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = inputs.WORKLOADS[args.workload]
    if w["kind"] != "mlp":
        raise SystemExit("bench.py times the MLP block workloads; see --workload")
    n, T, D, F = w["tp"], w["T"], w["hidden"], w["ffn"]
    Fr = F // n
    mode = args.combine
    combine = COMBINE_NAMES[mode]
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream

    # -- inputs: one seeded host draw, copied into R device sets ---------------------------
    data = inputs.make_bf16_inputs(w)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)

    set_bytes = (2 * F * D + D * F) * 2 + T * D * 2 + T * F * 2 + n * T * D * 4
    R = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    plan0 = tp.tp_plan_create(n, D, 8 * n, 8, 128, F)
    shards = [tp.tp_plan_query_rank(plan0, r) for r in range(n)]
    sets = []
    for i in range(R):
        x = to_dev(data["x"])
        wg, wu, wd = to_dev(data["wg"]), to_dev(data["wu"]), to_dev(data["wd"])
        g = [wg[slice(*shards[r]["ranges"]["gate_proj"])] for r in range(n)]
        u = [wu[slice(*shards[r]["ranges"]["up_proj"])] for r in range(n)]
        dn = [wd[:, slice(*shards[r]["ranges"]["down_proj"])] for r in range(n)]
        hbuf = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
        h = [hbuf[:, r * Fr:(r + 1) * Fr] for r in range(n)]
        ys = [torch.empty((T, D), dtype=torch.float32, device=dev)
              for _ in range(1 if mode == "fused" else n)]
        s = {"x": x, "keep": (wg, wu, wd, hbuf), "g": g, "u": u, "d": dn, "h": h, "y": ys}
        s["gate_up"] = ("tp_gate_up_swiglu", tp.arr([x]), tp.arr(g), tp.arr(u), tp.arr(h))
        if mode == "fused":
            s["down"] = tp.Prepared("tp_row_linear", n, tp.arr(h), tp.arr(dn), tp.arr(ys),
                                    tp.TP_COMBINE_FUSED, sptr)
            s["ring"] = None
        else:
            s["down"] = tp.Prepared("tp_row_linear", n, tp.arr(h), tp.arr(dn), tp.arr(ys),
                                    tp.TP_COMBINE_NONE, sptr)
            s["ring"] = tp.Prepared("tp_allreduce_ring", n, tp.arr(ys),
                                    tp.TP_RING_STEPS if mode == "ring" else tp.TP_RING_FUSED, sptr)
        sets.append(s)

    def step(s, ev=None):
        # a1: the shard plan (host), then the device path of the block
        plan = tp.tp_plan_create(n, D, 8 * n, 8, 128, F)
        name, xa, ga, ua, ha = s["gate_up"]
        if ev:
            ev[0].record(stream)
        st = tp.raw_status(name, plan.handle, xa, ga, ua, ha, sptr)
        if st != tp.TP_OK:
            raise tp.TPError(st, name)
        if ev:
            ev[1].record(stream)
        s["down"]()
        if ev:
            ev[2].record(stream)
        if s["ring"] is not None:
            s["ring"]()
        if ev:
            ev[3].record(stream)
        tp.tp_plan_destroy(plan)

    for i in range(args.warmup):
        step(sets[i % R])
    torch.cuda.synchronize(dev)
    st, word = tp.tp_device_status(sptr)
    if st != tp.TP_OK:
        raise SystemExit(f"device status {word:#x} after warm-up")

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    out_dir = os.path.join(ROOT, "gpurun_out")
    if not os.path.isdir(out_dir):
        import tempfile
        out_dir = tempfile.gettempdir()
    clock_path = os.path.join(out_dir, f"clocks_rank{rank}.csv")
    with ClockSampler(local, clock_path) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for i in range(K):
            step(sets[i % R], evs[i])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    st, word = tp.tp_device_status(sptr)
    if st != tp.TP_OK:
        raise SystemExit(f"device status {word:#x} after the timed region")
    total_ms = t_start.elapsed_time(t_end)
    gate_ms = [e[0].elapsed_time(e[1]) for e in evs]
    down_ms = [e[1].elapsed_time(e[2]) for e in evs]
    ring_ms = [e[2].elapsed_time(e[3]) for e in evs]
    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    max_ms = dist_max(total_ms, world)

    fl = mlp_flops(w)
    value = world * fl["total"] * K / (max_ms / 1e3) / 1e12
    peaks, peak_src = load_peaks()
    gate_mean_s = statistics.mean(gate_ms) / 1e3
    achieved = fl["gate_up"] / gate_mean_s / 1e12
    part_bytes = T * D * 4
    rb = ring_bytes(mode, n, part_bytes)
    ring_mean_s = statistics.mean(ring_ms) / 1e3
    combine_gbs = rb / ring_mean_s / 1e9 if rb and ring_mean_s > 0 else None

    # -- end to end through the public block call with host buffers ------------------------
    xh = torch.from_numpy(np.ascontiguousarray(data["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty((T, D), dtype=torch.float32).pin_memory()
    ws = torch.empty(tp.tp_mlp_block_workspace_size(plan0, T), dtype=torch.uint8, device=dev)
    es = sets[0]
    for i in range(3 + args.e2e_steps):
        if i == 3:
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        es["x"].copy_(xh, non_blocking=True)
        tp.tp_mlp_block(plan0, es["x"], es["g"], es["u"], es["d"], es["y"], combine, ws, stream=sptr)
        yh.copy_(es["y"][0], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = dist_max(e0.elapsed_time(e1), world)
    e2e_value = world * fl["total"] * args.e2e_steps / (e2e_ms / 1e3) / 1e12

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = cpu_baseline(w, args.workload, args.cpu_seconds)
        except Exception as exc:  # reported, not fatal
            cpu = {"error": str(exc)[-300:]}

    traffic = committed_traffic(args.workload)
    peak = peaks["bf16_tflops"]
    line = {
        "metric": "TP MLP/attn-proj block TFLOP/s and combine GB/s on 1 GB300, % of roofline",
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(max_ms / K, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights, rounded to bf16)",
        "config": {
            "workload": args.workload, "tokens": T, "hidden": D, "ffn": F, "tp_size": n,
            "combine": mode, "flops_per_step": fl["total"],
            "l2": f"{R} rotating input sets of {set_bytes / 1e6:.1f} MB (> 2x L2 in total)",
            "parallelism": f"tp{n} logical ranks on one GPU; replicas across GPUs",
        },
        "phases_ms": {"gate_up_swiglu": round(statistics.mean(gate_ms), 5),
                      "down": round(statistics.mean(down_ms), 5),
                      "combine": round(statistics.mean(ring_ms), 5),
                      "step_sum": round(statistics.mean(step_ms), 5)},
        "combine": {"mode": mode, "gbs": round(combine_gbs, 1) if combine_gbs else None,
                    "bytes_per_step": rb, "frac_of_hbm": round(combine_gbs / peaks["hbm_gbs"], 4)
                    if combine_gbs else None, "bus_bytes_per_rank": int(2 * (n - 1) / n * part_bytes)},
        "roofline": {"kernel": "k_gemm_bf16 (gate/up + SwiGLU epilogue)", "bound": "tensor",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "algorithmic_flops_per_launch": fl["gate_up"]},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 4},
        "gpu_launches": launches_per_step(mode, n) * K,
        "clocks": clk.summary(),
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---- reference arm: the oracle on the host cores ----------------------------------------
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from tensor_sharded_linear_gqa_gb300 import inputs
    w = inputs.WORKLOADS[args.workload]
    K, W = args.steps, max(args.warmup, 0)
    # Each step is a row sample of the workload sized so that all K + W steps take
    # about two minutes on the host cores.
    per_step_ms = max(5.0, 120_000.0 / (K + W))
    r = cpu_oracle_run(args.workload, 1e9, K + W, -int(per_step_ms))
    times = r["times"][W:] or r["times"]
    per_step = sum(times) / len(times)
    rows = r["rows"]
    value = mlp_flops(dict(w, T=rows))["total"] / per_step / 1e12
    sample = (f"{rows} of {w['T']} token rows of {args.workload} per step (fp64 oracle: column "
              f"gate/up, SwiGLU, row down, ring all-reduce), {len(times)} timed passes")
    line = {"metric": "TP MLP/attn-proj block TFLOP/s and combine GB/s on 1 GB300, % of roofline",
            "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": len(times),
            "warmup": W, "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "tokens": w["T"], "hidden": w["hidden"],
                       "ffn": w["ffn"], "tp_size": w["tp"], "rows_per_step": rows},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": r["cores"],
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
