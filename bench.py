#!/usr/bin/env python3
"""Benchmark of the tensor-parallel sharded linear blocks on GB300 (one JSON line on stdout).

One step = one pass of the hot path over one batch of synthetic input. Default
workload: the large decoder-layer projections and MLP in prefill, T=4096 tokens,
D=8192, 64 q / 8 kv heads of 128, F=28672, TP=8, bf16 inputs with fp32
accumulation. A step is the shard plan (host), the q/k/v column-parallel GEMM,
the o_proj row-parallel GEMM with the ring all-reduce of its partials, the
gate/up column-parallel GEMM with the fused SwiGLU, and the down row-parallel
GEMM with its ring all-reduce. Inputs are already resident in HBM; when one
input set is smaller than twice the L2, several sets (each a full weight copy)
are rotated so that no step reads another step's weights from L2.

`--impl reference` times the fp64 CPU oracle on the same workload instead (the
CPU baseline arm). Under torchrun every rank runs an independent replica on its
own GPU (the block itself lives on one device); the value is the total over
ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import ctypes
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
COMBINE_NAMES = {"fused": 1, "ring": 2, "ring_fused": 3, "ring_shared": 4}
# Modes of the row-parallel -> reduce-scatter -> column-parallel pipeline workload.
PIPELINE_MODES = ("deferred", "gathered")
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default: about one second of GPU time for the workload)")
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", default="prefill_layer_tp8_t4096")
    p.add_argument("--combine", choices=sorted(COMBINE_NAMES) + sorted(PIPELINE_MODES), default=None,
                   help="ring_fused (default): the ring all-reduce in one pass, bit-identical to ring (N-1 step "
                        "launches per phase); ring_shared: the same with the result stored once, for ranks that "
                        "share one output on this device; fused: the ranks summed in the GEMM accumulator. The "
                        "reduce-scatter pipeline workload takes deferred (default: the column GEMM reads the "
                        "reduced chunks) or gathered (an all-gather first)")
    p.add_argument("--moe-mode", choices=["within_expert", "expert_parallel"], default="within_expert",
                   help="MoE sharding of the moe workloads")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="host seconds of the CPU baseline timed beside the native arm")
    p.add_argument("--clocks-csv", default=None,
                   help="file for the nvidia-smi clock samples of the timed region, {rank} replaced by the "
                        "rank (default: a temporary file)")
    p.add_argument("--reference-seconds", type=float, default=120.0,
                   help="host seconds that all steps of --impl reference take together")
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
    if mode == "ring_shared":
        return (n + 1) * size_bytes  # each partial read once, the one shared result written
    return 2 * n * size_bytes  # ring_fused: each partial read once, every rank written once


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
def dist_setup(args, backend: str | None = None):
    """One process per GPU from the launcher's environment. NCCL on GPUs; gloo
    (host only, for the CPU tests of this plumbing) when no GPU is visible or
    when asked for."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    """The largest of every rank's x (the job time is the slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(world: int, flops_per_step: float, steps: int, max_ms: float) -> float:
    """Whole-job throughput: the work every replica did over the slowest rank's time."""
    return world * flops_per_step * steps / (max_ms / 1e3) / 1e12


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
# Host bytes of operands the timed oracle may hold; a workload above it is not timed.
CPU_HOLD_CAP = 16 << 30


def oracle_work(w) -> str:
    """What one oracle pass computes, for the sample description."""
    kind = w["kind"]
    if kind == "layer" and w.get("attention"):
        return ("q/k/v column-parallel, causal attention core, o_proj row-parallel with its ring all-reduce, "
                "then the MLP block")
    return {"mlp": "column gate/up, SwiGLU, row down, ring all-reduce",
            "attn": "q/k/v column-parallel, o_proj row-parallel, ring all-reduce",
            "layer": "attention projections then the MLP block, each with its ring all-reduce",
            "attn_core": "causal attention of every rank's q heads with the kv heads the plan gives them",
            "moe": "every rank's share of the routed expert FFNs, ring all-reduce",
            "vocab": "vocab-parallel lookup with its ring all-gather, then the LM-head logits",
            "rs_column": "row-parallel partials, ring reduce-scatter rounded to bf16, column-parallel GEMM",
            }[kind]


def oracle_hold_bytes(w) -> int:
    """Host bytes of the inputs the timed oracle keeps widened: fp64 weights and
    activations, except the embedding table, kept as float32 (the oracle widens it
    one shard at a time)."""
    from tensor_sharded_linear_gqa_gb300 import inputs
    total = 0
    for name, shp in inputs.weight_shapes(w).items():
        count = 1
        for s in shp:
            count *= s
        total += count * (4 if name == "emb" else 8)
    T, D = w["T"], w["hidden"]
    total += 8 * T * D * 2
    if w["kind"] == "attn_core":
        total += 8 * T * (w["q_heads"] + 2 * w["kv_heads"]) * w["head_dim"]
    return total


def sample_flops(w, rows: int) -> float:
    """Algorithmic flops of one pass over the first `rows` token rows (for causal
    attention, the first `rows` queries with their keys: the same problem at T = rows)."""
    return sum(f for f, _ in phase_costs(dict(w, T=rows), "ring_fused").values())


def oracle_pass(w, moe_mode: str):
    """The workload's inputs (the same seeded bits the GPU path reads, widened
    exactly), and pass(rows): the oracle over the first `rows` token rows, which
    returns the step's outputs (rank 0's copy where every rank holds the result).
    Also returns p, the power of rows that a pass's cost grows with."""
    import numpy as np

    import oracle as O
    from tensor_sharded_linear_gqa_gb300 import inputs

    d = inputs.make_bf16_inputs(w)
    f = {}
    for k in list(d):
        if d[k].dtype == np.uint16:
            bits = d.pop(k)
            f[k] = inputs.bf16_bits_to_f64(bits).astype(np.float32 if k == "emb" else np.float64)
            del bits
    n, kind = w["tp"], w["kind"]
    hd = w.get("head_dim", 128)
    plan = None
    if kind in ("attn", "layer", "attn_core"):
        plan = O.shard_plan(n, w["hidden"], w["q_heads"], w["kv_heads"], hd, w.get("ffn", 8 * n))

    def mlp(x):
        return O.mlp_sharded(x, f["wg"], f["wu"], f["wd"], n)["y"][0]

    def attn_projections(x, rows):
        r = O.attn_proj_sharded(x, f["wq"], f["wk"], f["wv"], f["a"][:rows], f["wo"], plan, hd)
        return r["q"] + r["k"] + r["v"] + [r["y"][0]]

    def attention_layer(x):
        q = [O.linear(x, f["wq"][slice(*s.ranges["q_proj"])]) for s in plan]
        k = [O.linear(x, f["wk"][slice(*s.ranges["k_proj"])]) for s in plan]
        v = [O.linear(x, f["wv"][slice(*s.ranges["v_proj"])]) for s in plan]
        att = O.attention_core_sharded(q, k, v, plan, hd, causal=True)
        parts = [O.linear(att[r], f["wo"][:, slice(*s.ranges["o_proj"])]) for r, s in enumerate(plan)]
        y = O.ring_all_reduce([p.reshape(-1) for p in parts])[0].reshape(x.shape[0], -1)
        return q + k + v + att + [y]

    if kind == "mlp":
        return (lambda rows: [mlp(f["x"][:rows])]), 1
    if kind == "attn":
        return (lambda rows: attn_projections(f["x"][:rows], rows)), 1
    if kind == "layer":
        def layer(rows):
            x = f["x"][:rows]
            out = attention_layer(x) if w.get("attention") else attn_projections(x, rows)
            return out + [mlp(x)]
        return layer, 1
    if kind == "attn_core":
        def heads(t, rng):
            return t[:, rng[0] * hd:rng[1] * hd]
        qs = [heads(f["q"], s.q_heads) for s in plan]
        ks = [heads(f["k"], s.kv_heads) for s in plan]
        vs = [heads(f["v"], s.kv_heads) for s in plan]
        return (lambda rows: O.attention_core_sharded([t[:rows] for t in qs], [t[:rows] for t in ks],
                                                      [t[:rows] for t in vs], plan, hd, causal=True)), 2
    if kind == "moe":
        mode = O.MOE_WITHIN_EXPERT if moe_mode == "within_expert" else O.MOE_EXPERT_PARALLEL
        ids, wts = d["topk_ids"], d["topk_w"].astype(np.float64)
        return (lambda rows: O.moe_sharded(f["x"][:rows], ids[:rows], wts[:rows], f["eg"], f["eu"], f["ed"], n,
                                           mode)["y"][:1]), 1
    if kind == "vocab":
        emb, wlm, ids = O.split_rows(f["emb"], n), O.split_rows(f["wlm"], n), d["ids"]

        def vocab(rows):
            return [O.vocab_parallel_embedding(ids[:rows], emb)["y"][0],
                    O.vocab_parallel_lm_head(f["x"][:rows], wlm)["logits"]]
        return vocab, 1
    if kind == "rs_column":
        wd, wqkv = O.split_cols(f["wd"], n), O.split_rows(f["wqkv"], n)

        def rs_column(rows):
            parts = O.row_parallel(O.split_cols(f["h"][:rows], n), wd)
            return O.reduce_scatter_then_column(parts, wqkv, round_bf16=True)["y"]
        return rs_column, 1
    raise ValueError(f"no timed oracle pass for workload kind {kind}")


# Rows of every step result that the native arm saves for the oracle's check.
PARITY_ROWS = 256
PARITY_TOL = 1e-2  # max|gpu - oracle| <= 1e-2 * max|oracle| (bf16 inputs, fp32 accumulation)


def oracle_results(w, out: list) -> list:
    """The step results, in the order step_results gives the GPU's, out of one
    oracle pass's outputs (see oracle_pass)."""
    import numpy as np
    kind = w["kind"]
    if kind == "attn":
        return [out[-1]]
    if kind == "layer":
        return out[-2:]
    if kind == "attn_core":
        return [np.concatenate(out, axis=1)]
    return list(out)


def parity_errors(gpu: list, ref: list) -> list:
    """max|gpu - ref| / max|ref| over the rows both hold, per result."""
    import numpy as np
    errs = []
    for g, r in zip(gpu, ref):
        r = np.asarray(r, dtype=np.float64)
        m = min(g.shape[0], r.shape[0])
        g, r = np.asarray(g[:m], dtype=np.float64), r[:m]
        scale = float(np.max(np.abs(r))) if r.size else 0.0
        diff = float(np.max(np.abs(g - r))) if r.size else 0.0
        errs.append(diff / scale if scale > 0 else diff)
    return errs


def cpu_child(workload: str, moe_mode: str, budget: str, max_reps: str, rows: str, check: str = "") -> None:
    """Child-process body of cpu_oracle_run: times oracle passes, prints one JSON line.
    With `check` (an .npz of the GPU's first rows of every step result), the last
    pass's outputs are compared with them."""
    from tensor_sharded_linear_gqa_gb300 import inputs
    w = dict(inputs.WORKLOADS[workload])
    budget, max_reps, rows = float(budget), int(max_reps), int(rows)
    one_pass, power = oracle_pass(w, moe_mode)
    if rows <= 0:
        # Size the row sample so that one pass takes about -rows/1000 seconds: fit
        # cost = a + b * rows**power through two timed probes after a warm-up pass
        # (a is the part of a pass that does not grow with the rows).
        target = -rows / 1000.0
        r1, r2 = min(w["T"], 8), min(w["T"], 32)
        one_pass(r1)
        cost = []
        for r in (r1, r2):
            t0 = time.perf_counter()
            one_pass(r)
            cost.append(time.perf_counter() - t0)
        b = (cost[1] - cost[0]) / (r2 ** power - r1 ** power) if r2 > r1 else 0.0
        a = cost[0] - b * r1 ** power
        if b <= 0.0:  # the probes did not resolve a slope: scale the larger one
            rows = int(r2 * (target / max(cost[1], 1e-4)) ** (1.0 / power))
        elif target <= a:
            rows = r1
        else:
            rows = int(((target - a) / b) ** (1.0 / power))
    rows = max(1, min(w["T"], rows))
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        last = one_pass(rows)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all >= budget or len(times) >= max_reps:
            break
    res = {"reps": len(times), "seconds": sum(times), "times": times, "rows": rows}
    if check:
        import numpy as np
        with np.load(check) as z:
            gpu = [z[f"r{i}"] for i in range(len(z.files))]
        errs = parity_errors(gpu, oracle_results(w, last))
        res["parity"] = {"rows": min(rows, PARITY_ROWS), "max_rel_err": [float(f"{e:.3e}") for e in errs],
                         "tol": PARITY_TOL, "pass": bool(all(e <= PARITY_TOL for e in errs))}
    print(json.dumps(res))


def cpu_oracle_run(workload: str, moe_mode: str, seconds: float, max_reps: int, rows: int,
                   check: str = "") -> dict:
    """Runs the fp64 oracle over a workload in a child process on every core this
    process may use. rows > 0: that many token rows per pass (at most T); rows <= 0:
    sized so that a pass takes about -rows ms."""
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    code = "import sys; sys.path.insert(0, sys.argv[1]); import bench; bench.cpu_child(*sys.argv[2:])"
    out = subprocess.run([sys.executable, "-c", code, ROOT, workload, moe_mode, str(seconds), str(max_reps),
                          str(rows), check], capture_output=True, text=True, env=env, timeout=1800)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    r = json.loads(out.stdout.strip().splitlines()[-1])
    r["cores"] = cores
    return r


def cpu_too_large(w):
    """The reason the oracle is not timed on a workload, or None."""
    need = oracle_hold_bytes(w)
    if need > CPU_HOLD_CAP:
        return (f"the oracle would hold {need / 2**30:.1f} GiB of widened inputs on the host "
                f"(cap {CPU_HOLD_CAP / 2**30:.0f} GiB)")
    return None


def cpu_baseline(w, workload: str, moe_mode: str, seconds: float, check: str = "") -> tuple:
    """The oracle as it stands, timed for about `seconds` on a bounded row sample
    (whole passes when a pass over all T rows takes under a quarter of that).
    Returns (the cpu_baseline object, the parity check of the GPU's saved rows or None)."""
    why = cpu_too_large(w)
    if why:
        return {"unavailable": why}, None
    r = cpu_oracle_run(workload, moe_mode, seconds, 1000, -int(seconds * 250), check)
    rows = r["rows"]
    val = sample_flops(w, rows) * r["reps"] / r["seconds"] / 1e12
    what = "full passes" if rows == w["T"] else f"passes over {rows} of its {w['T']} token rows"
    return ({"value": round(val, 6), "unit": "TFLOP/s", "cores": r["cores"], "kind": "oracle",
             "sample": f"{r['reps']} {what} of the fp64 oracle on {workload} ({oracle_work(w)}) "
                       f"in {r['seconds']:.1f} s"}, r.get("parity"))


# ---- native arm ----------------------------------------------------------------------
class DeviceSet:
    """One copy of a workload's inputs, weights and outputs in HBM, sharded per the plan,
    with the step's C calls marshalled once."""

    def __init__(self, tp, torch, w, data, plan, shards, dev, sptr, mode, moe_mode="within_expert"):
        import numpy as np
        n, T = w["tp"], w["T"]
        D = w["hidden"]
        self.keep = []

        def to_dev(bits):
            t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)
            self.keep.append(t)
            return t

        def rng(r, name):
            return slice(*shards[r]["ranges"][name])

        self.calls = []  # (phase name, callable)
        self.step_calls = []  # block calls that replace the leading phase calls in the timed step
        self.x = to_dev(data["x"])
        self.e2e = {}
        if w["kind"] in ("attn", "layer"):
            hd = w["head_dim"]
            rep = shards[0]["kv_replicated"]
            nkv = 1 if rep else n
            wq, wk, wv, wo = (to_dev(data[k]) for k in ("wq", "wk", "wv", "wo"))
            # with the attention core, A is its output; else an explicit input
            self.attention = bool(w.get("attention"))
            self.a = (torch.empty((T, w["q_heads"] * hd), dtype=torch.bfloat16, device=dev) if self.attention
                      else to_dev(data["a"]))
            self.keep.append(self.a)
            q_w = [wq[rng(r, "q_proj")] for r in range(n)]
            k_w = [wk[rng(r, "k_proj")] for r in range(nkv)]
            v_w = [wv[rng(r, "v_proj")] for r in range(nkv)]
            a_r = [self.a[:, rng(r, "o_proj")] for r in range(n)]
            o_w = [wo[:, rng(r, "o_proj")] for r in range(n)]
            q = [torch.empty((T, t.shape[0]), dtype=torch.bfloat16, device=dev) for t in q_w]
            k = [torch.empty((T, t.shape[0]), dtype=torch.bfloat16, device=dev) for t in k_w]
            v = [torch.empty((T, t.shape[0]), dtype=torch.bfloat16, device=dev) for t in v_w]
            yo = [torch.empty((T, D), device=dev) for _ in range(1 if mode == "fused" else n)]
            self.keep += q + k + v + yo
            self.calls.append(("qkv", ("tp_qkv_proj", tp.arr([self.x]), tp.arr(q_w), tp.arr(k_w), tp.arr(v_w),
                                       tp.arr(q), tp.arr(k), tp.arr(v))))
            self.aws = None
            if self.attention:
                self.aws = torch.empty(tp.tp_attn_core_workspace_size(plan, T), dtype=torch.uint8, device=dev)
                self.keep.append(self.aws)
                self.calls.append(("attn_core", tp.Prepared(
                    "tp_attn_core", plan.handle, tp.arr(q), tp.arr(k), tp.arr(v), tp.arr(a_r), 1,
                    self.aws.data_ptr(), self.aws.numel(), sptr)))
            # o_proj row-parallel with its combine, one public call (the library may
            # fold the ring into the GEMM)
            self.calls.append(("o_proj", tp.Prepared("tp_row_linear", n, tp.arr(a_r), tp.arr(o_w), tp.arr(yo),
                                                     COMBINE_NAMES[mode], sptr)))
            if not self.attention:
                # the timed step makes the block call, q/k/v and o_proj in one
                # (the phase pass times the two halves on their own)
                self.step_calls = [("attn_proj", ("tp_attn_proj", tp.arr([self.x]), tp.arr(q_w), tp.arr(k_w),
                                                  tp.arr(v_w), tp.arr(q), tp.arr(k), tp.arr(v), tp.arr(a_r),
                                                  tp.arr(o_w), tp.arr(yo), COMBINE_NAMES[mode]))]
            self.e2e["attn"] = (q_w, k_w, v_w, q, k, v, a_r, o_w, yo)
        if w["kind"] in ("mlp", "layer"):
            F = w["ffn"]
            Fr = F // n
            wg, wu, wd = (to_dev(data[k]) for k in ("wg", "wu", "wd"))
            g = [wg[rng(r, "gate_proj")] for r in range(n)]
            u = [wu[rng(r, "up_proj")] for r in range(n)]
            dn = [wd[:, rng(r, "down_proj")] for r in range(n)]
            hbuf = torch.empty((T, F), dtype=torch.bfloat16, device=dev)
            h = [hbuf[:, r * Fr:(r + 1) * Fr] for r in range(n)]
            ym = [torch.empty((T, D), device=dev) for _ in range(1 if mode == "fused" else n)]
            self.keep += [hbuf] + ym
            self.calls.append(("gate_up", ("tp_gate_up_swiglu", tp.arr([self.x]), tp.arr(g), tp.arr(u),
                                           tp.arr(h))))
            self.calls.append(("down", tp.Prepared("tp_row_linear", n, tp.arr(h), tp.arr(dn), tp.arr(ym),
                                                   COMBINE_NAMES[mode], sptr)))
            # the timed step makes the block call (gate/up and down with its combine)
            self.mws = torch.empty(tp.tp_mlp_block_workspace_size(plan, T), dtype=torch.uint8, device=dev)
            self.keep.append(self.mws)
            self.step_calls.append(("mlp_block", ("tp_mlp_block", tp.arr([self.x]), tp.arr(g), tp.arr(u), tp.arr(dn),
                                                  tp.arr(ym), COMBINE_NAMES[mode], self.mws.data_ptr(),
                                                  self.mws.numel())))
            self.e2e["mlp"] = (g, u, dn, ym)
        if w["kind"] == "attn_core":
            hd = w["head_dim"]
            rep = shards[0]["kv_replicated"]
            self.aq, self.ak, self.av = to_dev(data["q"]), to_dev(data["k"]), to_dev(data["v"])
            ws = torch.empty(tp.tp_attn_core_workspace_size(plan, T), dtype=torch.uint8, device=dev)
            aout = torch.empty((T, w["q_heads"] * hd), dtype=torch.bfloat16, device=dev)
            self.keep += [ws, aout]

            def cols(t, heads):
                return t[:, heads[0] * hd:heads[1] * hd]

            def attn_calls(qb, kb, vb, ob):
                """The public attention-core call over every rank's q heads (causal)."""
                qs = [cols(qb, shards[r]["q_heads"]) for r in range(n)]
                outs = [cols(ob, shards[r]["q_heads"]) for r in range(n)]
                ks = [kb] if rep else [cols(kb, shards[r]["kv_heads"]) for r in range(n)]
                vs = [vb] if rep else [cols(vb, shards[r]["kv_heads"]) for r in range(n)]
                return [("attn_core", tp.Prepared("tp_attn_core", plan.handle, tp.arr(qs), tp.arr(ks), tp.arr(vs),
                                                  tp.arr(outs), 1, ws.data_ptr(), ws.numel(), sptr))]

            self.calls += attn_calls(self.aq, self.ak, self.av, aout)
            self.e2e["attn_core"] = (attn_calls, aout)
        if w["kind"] == "moe":
            E, F, k = w["experts"], w["ffn"], w["top_k"]
            within = moe_mode == "within_expert"
            eg, eu, ed = data["eg"], data["eu"], data["ed"]
            if within:  # rank r: every expert's F/N slice, stacked by expert
                fs = F // n
                g = [np.concatenate([eg[e, r * fs:(r + 1) * fs] for e in range(E)]) for r in range(n)]
                u = [np.concatenate([eu[e, r * fs:(r + 1) * fs] for e in range(E)]) for r in range(n)]
                dn = [np.concatenate([ed[e][:, r * fs:(r + 1) * fs] for e in range(E)]) for r in range(n)]
            else:       # rank r: experts r, r+N, ... whole
                g = [np.concatenate([eg[e] for e in range(r, E, n)]) for r in range(n)]
                u = [np.concatenate([eu[e] for e in range(r, E, n)]) for r in range(n)]
                dn = [np.concatenate([ed[e] for e in range(r, E, n)]) for r in range(n)]
            g, u, dn = [to_dev(t) for t in g], [to_dev(t) for t in u], [to_dev(t) for t in dn]
            self.rid = torch.from_numpy(data["topk_ids"]).to(dev)
            self.rw = torch.from_numpy(data["topk_w"]).to(dev)
            self.dims = tp.moe_dims(n, tp.TP_MOE_WITHIN_EXPERT if within else tp.TP_MOE_EXPERT_PARALLEL, E, k, D, F)
            ws = torch.empty(tp.tp_moe_workspace_size(self.dims, T), dtype=torch.uint8, device=dev)
            self.keep += [self.rid, self.rw, ws]
            combine_id = COMBINE_NAMES[mode]

            def moe_calls(xbuf, rid, rw, ys):
                """The public MoE block call: routing, gather, expert GEMMs, weighted
                combine and the all-reduce, all on the device."""
                xs = tp.tensor(xbuf)
                self.keep.append(xs)
                return [("moe_block", tp.Prepared(
                    "tp_moe_block", ctypes.byref(self.dims), ctypes.byref(xs), rid.data_ptr(), rw.data_ptr(),
                    tp.arr(g), tp.arr(u), tp.arr(dn), tp.arr(ys), combine_id, ws.data_ptr(), ws.numel(), sptr))]

            ys = [torch.empty((T, D), device=dev) for _ in range(1 if mode == "fused" else n)]
            self.keep += ys
            self.calls += moe_calls(self.x, self.rid, self.rw, ys)
            self.e2e["moe"] = (moe_calls, ys)
        if w["kind"] == "vocab":
            V = w["vocab"]
            per_v = V // n
            emb, wlm = to_dev(data["emb"]), to_dev(data["wlm"])
            emb_r = [emb[r * per_v:(r + 1) * per_v] for r in range(n)]
            wlm_r = [wlm[r * per_v:(r + 1) * per_v] for r in range(n)]
            self.ids = torch.from_numpy(data["ids"]).to(dev)
            self.keep.append(self.ids)

            def vocab_calls(ids, xbuf, x0, logits):
                """The lookup of the token ids (one shared output copy), then the LM-head
                logits of the hidden states, gathered into one [T x V] f32 tensor."""
                xs = tp.tensor(xbuf)
                self.keep.append(xs)
                return [("embed", tp.Prepared("tp_vocab_embedding", n, tp.ids_ptr(ids), ids.numel(),
                                              tp.arr(emb_r), tp.arr([x0]), 1, sptr)),
                        ("lm_head", tp.Prepared("tp_vocab_lm_head", n, ctypes.byref(xs), tp.arr(wlm_r),
                                                tp.arr([logits]), 1, sptr))]

            x0 = torch.empty((T, D), dtype=torch.bfloat16, device=dev)
            logits = torch.empty((T, V), device=dev)
            self.keep += [x0, logits]
            self.calls += vocab_calls(self.ids, self.x, x0, logits)
            self.e2e["vocab"] = (vocab_calls, x0, logits)
        if w["kind"] == "rs_column":
            F = w["ffn"]
            Fr = F // n
            self.h = to_dev(data["h"])
            wd, wqkv = to_dev(data["wd"]), to_dev(data["wqkv"])
            per = wqkv.shape[0] // n
            wd_r = [wd[:, r * Fr:(r + 1) * Fr] for r in range(n)]
            wc_r = [wqkv[r * per:(r + 1) * per] for r in range(n)]
            parts = [torch.empty((T, D), device=dev) for _ in range(n)]
            chunks = [torch.empty((T, D), dtype=torch.bfloat16, device=dev) for _ in range(n)]
            xfull = torch.empty((T, D), dtype=torch.bfloat16, device=dev) if mode == "gathered" else None
            self.keep += parts + chunks + [xfull]
            self._xs = tp.tensor(xfull) if xfull is not None else None

            def pipeline_calls(hbuf, ys):
                """Row-parallel partials, the ring reduce-scatter into bf16 chunks, then the
                column-parallel GEMM: over the chunks in place (deferred) or over an
                all-gathered copy (gathered). The intermediates are shared: every call
                runs on one stream."""
                h_r = [hbuf[:, r * Fr:(r + 1) * Fr] for r in range(n)]
                calls = [("row", tp.Prepared("tp_row_linear", n, tp.arr(h_r), tp.arr(wd_r), tp.arr(parts),
                                             tp.TP_COMBINE_NONE, sptr)),
                         ("combine_rs", tp.Prepared("tp_reduce_scatter_bf16", n, tp.arr(parts), tp.arr(chunks),
                                                    sptr))]
                if mode == "gathered":
                    shards_rs = [chunks[r][r * T // n:(r + 1) * T // n] for r in range(n)]
                    calls.append(("combine_ag", tp.Prepared("tp_all_gather", n, tp.arr(shards_rs),
                                                            tp.arr([xfull]), 1, 0, sptr)))
                    calls.append(("column", tp.Prepared("tp_column_linear", n, ctypes.byref(self._xs),
                                                        tp.arr(wc_r), tp.arr(ys), 0, sptr)))
                else:
                    calls.append(("column", tp.Prepared("tp_column_linear_chunks", n, tp.arr(chunks),
                                                        tp.arr(wc_r), tp.arr(ys), 0, sptr)))
                return calls

            ys = [torch.empty((T, per), dtype=torch.bfloat16, device=dev) for _ in range(n)]
            self.keep += ys
            self.calls += pipeline_calls(self.h, ys)
            self.e2e["rs_column"] = (pipeline_calls, ys)


def result_copies(mode: str, n: int) -> int:
    """f32 result tensors a row-parallel layer with its combine writes: one per rank
    after a ring all-reduce, one for the fused sum or the shared ring result."""
    return 1 if mode in ("fused", "ring_shared") or n == 1 else n


def phase_costs(w, mode):
    """Algorithmic flops and HBM bytes of every phase of one step (weights counted once;
    a replicated K/V projection is computed once). A row-parallel phase includes its
    combine: its bytes are its operands and the combined result (the ring's own
    traffic, when it runs as a separate pass, is measured on its own; see
    combine_loop)."""
    n, T, D = w["tp"], w["T"], w["hidden"]
    out = {}
    part = T * D * 4
    nparts = result_copies(mode, n)
    if w["kind"] in ("attn", "layer"):
        hd, hq, hkv = w["head_dim"], w["q_heads"], w["kv_heads"]
        cols = (hq + 2 * hkv) * hd
        out["qkv"] = (2.0 * T * D * cols, cols * D * 2 + T * D * 2 + T * cols * 2)
        out["o_proj"] = (2.0 * T * hq * hd * D, D * hq * hd * 2 + T * hq * hd * 2 + nparts * part)
    if w["kind"] in ("mlp", "layer"):
        F = w["ffn"]
        out["gate_up"] = (4.0 * T * D * F, 2 * F * D * 2 + T * D * 2 + T * F * 2)
        out["down"] = (2.0 * T * F * D, D * F * 2 + T * F * 2 + nparts * part)
    if w["kind"] == "layer" and w.get("attention"):
        hd, hq, hkv = w["head_dim"], w["q_heads"], w["kv_heads"]
        out["attn_core"] = (4.0 * hd * hq * T * (T + 1) / 2,
                            T * hq * hd * 2 * 2 + T * hkv * hd * 2 * 2 + 2 * T * hkv * hd * 2)
    if w["kind"] == "attn_core":
        hd, hq, hkv = w["head_dim"], w["q_heads"], w["kv_heads"]
        # causal: query i meets keys 0..i; QK^T and PV, 2 flops a multiply-add each
        out["attn_core"] = (4.0 * hd * hq * T * (T + 1) / 2,
                            T * hq * hd * 2 * 2 + T * hkv * hd * 2 * 2 + 2 * T * hkv * hd * 2)
    if w["kind"] == "moe":
        E, F, k = w["experts"], w["ffn"], w["top_k"]
        a = T * k
        # weights once, X, the routed copy of X and H written and read, f32 partials and outputs
        out["moe_block"] = (6.0 * a * D * F, 3 * E * F * D * 2 + T * D * 2 + 2 * a * D * 2 + 2 * a * F * 2 +
                            2 * (n if mode != "fused" else 1) * a * D * 4 + ring_bytes(mode, n, part))
    if w["kind"] == "vocab":
        V = w["vocab"]
        out["embed"] = (0.0, T * D * 2 * 2 + T * 4)        # rows read once and written once, ids
        out["lm_head"] = (2.0 * T * D * V, V * D * 2 + T * D * 2 + T * V * 4)
    if w["kind"] == "rs_column":
        F, hd = w["ffn"], w["head_dim"]
        per = (w["q_heads"] // n + 2 * max(1, w["kv_heads"] // n)) * hd
        S = T * D
        out["row"] = (2.0 * T * F * D, D * F * 2 + T * F * 2 + n * part)
        out["combine_rs"] = (0.0, n * S * 4 + S * 2)          # every partial read once, bf16 chunks written
        if mode == "gathered":
            out["combine_ag"] = (0.0, S * 2 * 2)               # bf16 chunks read, full copy written
        out["column"] = (2.0 * T * D * n * per, n * per * D * 2 + S * 2 + T * n * per * 2)
    return out


def combine_loop(tp, torch, dev, stream, n, rows, cols, mode, hbm_gbs):
    """The ring all-reduce alone: tp_allreduce_ring in the step's ring mode on N f32
    buffers of one partial's shape, back to back over enough buffer sets that the
    working set exceeds twice the L2 (so the figure is HBM's, not L2's), one pair
    of CUDA events around the loop. Algorithmic bytes: ring_bytes."""
    ring_mode = {"ring": tp.TP_RING_STEPS, "ring_fused": tp.TP_RING_FUSED,
                 "ring_shared": tp.TP_RING_FUSED_SHARED}[mode]
    part = rows * cols * 4
    nsets = 1 if n * part >= 2 * L2_BYTES else -(-2 * L2_BYTES // (n * part)) + 1
    bufs = [[torch.zeros((rows, cols), device=dev) for _ in range(n)] for _ in range(nsets)]
    calls = [tp.Prepared("tp_allreduce_ring", n, tp.arr(b), ring_mode, stream.cuda_stream) for b in bufs]
    for c in calls[:3]:
        c()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    calls[0]()
    torch.cuda.synchronize(dev)
    once = max(time.perf_counter() - t0, 1e-6)
    reps = max(len(calls), min(2000, int(0.3 / once)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = tp.tp_launch_count()
    e0.record(stream)
    for i in range(reps):
        calls[i % nsets]()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / reps
    b = ring_bytes(mode, n, part)
    gbs = b / (ms / 1e3) / 1e9
    del bufs, calls
    return {"gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_gbs, 4), "bytes_per_call": b,
            "launch_ms": round(ms, 5), "kernels_per_call": (tp.tp_launch_count() - l0) / reps,
            "bus_bytes_per_rank": 2 * (n - 1) * part // n,
            "timing": f"tp_allreduce_ring alone, {reps} calls over {nsets} set(s) of {n} x {part / 2**20:.0f} MiB"}


def run_native(args):
    import numpy as np
    import torch

    import tensor_sharded_linear_gqa_gb300 as tp
    from tensor_sharded_linear_gqa_gb300 import inputs

    world, rank, local = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = inputs.WORKLOADS[args.workload]
    if w["kind"] == "linear_fp32":
        raise SystemExit("bench.py times the bf16 block workloads")
    n, T, D = w["tp"], w["T"], w["hidden"]
    mode = args.combine
    # a stream of its own (not the legacy default stream), so that the end-to-end
    # loop can also be captured into a CUDA graph
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    sptr = stream.cuda_stream
    plan_args = (n, D, w.get("q_heads", 8 * n), w.get("kv_heads", 8), w.get("head_dim", 128),
                 w.get("ffn", 8 * n))
    plan0 = tp.tp_plan_create(*plan_args)
    shards = [tp.tp_plan_query_rank(plan0, r) for r in range(n)]

    data = inputs.make_bf16_inputs(w)
    costs = phase_costs(w, mode)
    set_bytes = sum(b for (_f, b) in costs.values() if b) + T * D * 2
    R = max(1, -(-2 * L2_BYTES // set_bytes) + (1 if set_bytes < 2 * L2_BYTES else 0))
    sets = [DeviceSet(tp, torch, w, data, plan0, shards, dev, sptr, mode, args.moe_mode) for _ in range(R)]
    names = [nm for (nm, _c) in sets[0].calls]

    def step(s, ev=None):
        # a1: the shard plan (host), then every device phase of the step in order:
        # the timed step makes the block calls (step_calls stand for the phase
        # calls they cover); the phase pass (ev given) makes the phase calls
        plan = tp.tp_plan_create(*plan_args)
        calls = s.calls
        if ev is None and s.step_calls:
            covered = {"attn_proj": ("qkv", "o_proj"), "mlp_block": ("gate_up", "down")}
            block_of = {nm: (b, c) for (b, c) in s.step_calls for nm in covered[b]}
            # each block call where its first phase call stood, the other phase calls kept
            calls, placed = [], set()
            for nm, c in s.calls:
                if nm not in block_of:
                    calls.append((nm, c))
                elif block_of[nm][0] not in placed:
                    placed.add(block_of[nm][0])
                    calls.append(block_of[nm])
        for i, (name, call) in enumerate(calls):
            if ev:
                ev[i].record(stream)
            if isinstance(call, tuple):  # plan-bound call: marshal the fresh plan handle
                st = tp.raw_status(call[0], plan.handle, *call[1:], sptr)
                if st != tp.TP_OK:
                    raise tp.TPError(st, call[0])
            else:
                call()
        if ev:
            ev[len(s.calls)].record(stream)
        tp.tp_plan_destroy(plan)

    for i in range(args.warmup):
        step(sets[i % R])
    torch.cuda.synchronize(dev)
    st, word = tp.tp_device_status(sptr)
    if st != tp.TP_OK:
        raise SystemExit(f"device status {word:#x} after warm-up")

    K = args.steps
    nev = len(names) + 1
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if args.clocks_csv:
        clock_path = args.clocks_csv.replace("{rank}", str(rank))
    else:
        import tempfile
        fd, clock_path = tempfile.mkstemp(prefix=f"clocks_rank{rank}_", suffix=".csv")
        os.close(fd)
    launches0 = tp.tp_launch_count()
    with ClockSampler(local, clock_path) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for i in range(K):
            step(sets[i % R])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    launches = tp.tp_launch_count() - launches0  # every kernel the K timed steps enqueued
    st, word = tp.tp_device_status(sptr)
    if st != tp.TP_OK:
        raise SystemExit(f"device status {word:#x} after the timed region")
    total_ms = t_start.elapsed_time(t_end)
    max_ms = dist_max(total_ms, world)
    # Per-phase breakdown, for the shares only: a second pass of the same steps
    # with CUDA events between the phases (events between kernels also stop the
    # next kernel's early launch, so this pass runs slower than the timed region).
    P = min(K, 500)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(P)]
    for i in range(P):
        step(sets[i % R], evs[i])
    torch.cuda.synchronize(dev)
    phase_ms = {nm: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) for i, nm in enumerate(names)}
    step_ms = statistics.mean(e[0].elapsed_time(e[-1]) for e in evs)

    flops_step = sum(f for (f, _b) in costs.values())
    value = aggregate_tflops(world, flops_step, K, max_ms)
    peaks, peak_src = load_peaks()

    # Roofline of the dominant kernel: its public call alone, back to back over the
    # rotating input sets, one pair of events around the whole loop on the
    # launching stream. The gate/up GEMM where there is an MLP, else q/k/v, the
    # row GEMM, the LM head, the MoE block or the attention core.
    rk = next(k for k in ("gate_up", "qkv", "row", "lm_head", "moe_block", "attn_core") if k in phase_ms)
    ri = names.index(rk)
    rf, rb = costs[rk]
    kr = max(20, min(K * 4, int(0.5e3 / max(phase_ms[rk], 1e-3))))  # about half a second

    def call_phase(s_, i_):
        name_, call_ = s_.calls[i_]
        if isinstance(call_, tuple):
            st_ = tp.raw_status(call_[0], plan0.handle, *call_[1:], sptr)
            if st_ != tp.TP_OK:
                raise tp.TPError(st_, call_[0])
        else:
            call_()

    for i in range(3):
        call_phase(sets[i % R], ri)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = tp.tp_launch_count()
    e0.record(stream)
    for i in range(kr):
        call_phase(sets[i % R], ri)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    r_launch_calls = (tp.tp_launch_count() - l0) / kr
    r_s = e0.elapsed_time(e1) / kr / 1e3
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    kname = {"attn_core": "k_attention (with the V transpose)",
             "moe_block": "tp_moe_block (routing, gather, expert GEMMs, combine)"}.get(rk, f"k_gemm_bf16* ({rk})")
    timing = (f"{kr} back-to-back calls of the phase's public call over {R} input set(s), "
              f"CUDA events around the loop on the launching stream")
    if rf / rb >= ridge:
        roof = {"kernel": kname, "bound": "tensor", "achieved": round(rf / r_s / 1e12, 2),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(rf / r_s / 1e12 / peaks["bf16_tflops"], 4),
                "peak_source": f"{peak_src} bf16_tflops (burst)", "algorithmic_flops_per_launch": rf}
    else:
        roof = {"kernel": kname, "bound": "hbm", "achieved": round(rb / r_s / 1e9, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(rb / r_s / 1e9 / peaks["hbm_gbs"], 4),
                "peak_source": f"{peak_src} hbm_gbs", "algorithmic_bytes_per_launch": rb}
    roof["traffic"] = committed_traffic(args.workload) if rk == "gate_up" else None
    roof["launch_ms"] = round(r_s * 1e3, 5)
    roof["timing"] = timing
    roof["kernels_per_call"] = r_launch_calls

    comb = {}  # every data-movement phase of the step (the lookup, the pipeline's collectives) against HBM
    for nm in names:
        if costs[nm][0] == 0:
            b = costs[nm][1]
            gbs = b / (phase_ms[nm] / 1e3) / 1e9 if phase_ms[nm] > 0 else None
            comb[nm] = {"gbs": round(gbs, 1), "bytes_per_step": b,
                        "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    if w["kind"] in ("attn", "layer", "mlp") and n > 1 and mode != "fused":
        comb["allreduce"] = combine_loop(tp, torch, dev, stream, n, T, D, mode, peaks["hbm_gbs"])

    # -- end to end through the public block calls with host buffers ---------------------
    s0 = sets[0]
    in_key = "h" if "rs_column" in s0.e2e else "x"
    x0 = s0.h if in_key == "h" else s0.x
    xh = torch.from_numpy(np.ascontiguousarray(data[in_key]).view(np.int16)).view(torch.bfloat16).pin_memory()
    ah = (torch.from_numpy(np.ascontiguousarray(data["a"]).view(np.int16)).view(torch.bfloat16).pin_memory()
          if "a" in data else None)
    outs_h = []
    idh = torch.from_numpy(data["ids"]).pin_memory() if "vocab" in s0.e2e else None
    h2d = xh.numel() * 2 + (ah.numel() * 2 if ah is not None else 0) + (idh.numel() * 4 if idh is not None else 0)
    copy_x = "attn_core" not in s0.e2e  # the attention core takes q, k, v instead of x
    if "attn_core" in s0.e2e:
        qkvh = [torch.from_numpy(np.ascontiguousarray(data[key]).view(np.int16)).view(torch.bfloat16).pin_memory()
                for key in ("q", "k", "v")]
        h2d = sum(t.numel() * 2 for t in qkvh)
    if "moe" in s0.e2e:
        rih = torch.from_numpy(data["topk_ids"]).pin_memory()
        rwh = torch.from_numpy(data["topk_w"]).pin_memory()
        h2d += rih.numel() * 4 + rwh.numel() * 4
    d2h = 0
    if "attn" in s0.e2e:
        outs_h.append(torch.empty((T, D), dtype=torch.float32).pin_memory())
        d2h += T * D * 4
    if "mlp" in s0.e2e:
        outs_h.append(torch.empty((T, D), dtype=torch.float32).pin_memory())
        d2h += T * D * 4
        ws = torch.empty(tp.tp_mlp_block_workspace_size(plan0, T), dtype=torch.uint8, device=dev)
    if "attn_core" in s0.e2e:
        ao = s0.e2e["attn_core"][1]
        outs_h.append(torch.empty(tuple(ao.shape), dtype=torch.bfloat16).pin_memory())  # every rank's A
        d2h += ao.numel() * 2
    if "moe" in s0.e2e:
        outs_h.append(torch.empty((T, D), dtype=torch.float32).pin_memory())  # the layer output
        d2h += T * D * 4
    if "vocab" in s0.e2e:
        # the looked-up rows and the full f32 logits come back
        for t in s0.e2e["vocab"][1:]:
            outs_h.append(torch.empty(tuple(t.shape), dtype=t.dtype).pin_memory())
            d2h += t.numel() * t.element_size()
    if "rs_column" in s0.e2e:
        # every rank's column-parallel output comes back: each holds its own heads
        for t in s0.e2e["rs_column"][1]:
            outs_h.append(torch.empty(tuple(t.shape), dtype=torch.bfloat16).pin_memory())
            d2h += t.numel() * 2
    combine_id = COMBINE_NAMES.get(mode)

    # Two activation slots (inputs, outputs, workspace) over the same weights, so
    # that step i's compute overlaps step i+1's input copy and step i-1's output
    # copy, each on its own copy stream: what a serving loop does with the public
    # calls. Every step's copies still run inside the timed region.
    def make_slot(first):
        sl = {"x": x0 if first else torch.empty_like(x0)}
        if "attn" in s0.e2e:
            sl["a"] = s0.a if first else torch.empty_like(s0.a)
            sl["yo"] = s0.e2e["attn"][8] if first else [torch.empty_like(t) for t in s0.e2e["attn"][8]]
        if "mlp" in s0.e2e:
            sl["ym"] = s0.e2e["mlp"][3] if first else [torch.empty_like(t) for t in s0.e2e["mlp"][3]]
            sl["ws"] = ws if first else torch.empty_like(ws)
        if "attn_core" in s0.e2e:
            sl["qkv"] = [s0.aq, s0.ak, s0.av] if first else [torch.empty_like(t) for t in (s0.aq, s0.ak, s0.av)]
            ao = s0.e2e["attn_core"][1]
            sl["aout"] = ao if first else torch.empty_like(ao)
        if "moe" in s0.e2e:
            sl["rid"] = s0.rid if first else torch.empty_like(s0.rid)
            sl["rw"] = s0.rw if first else torch.empty_like(s0.rw)
            ym0 = s0.e2e["moe"][1]
            sl["ymoe"] = ym0 if first else [torch.empty_like(t) for t in ym0]
        if "vocab" in s0.e2e:
            _f, x00, lg0 = s0.e2e["vocab"]
            sl["ids"] = s0.ids if first else torch.empty_like(s0.ids)
            sl["vo"] = [x00, lg0] if first else [torch.empty_like(x00), torch.empty_like(lg0)]
        if "rs_column" in s0.e2e:
            ys0 = s0.e2e["rs_column"][1]
            sl["ys"] = ys0 if first else [torch.empty_like(t) for t in ys0]
        sl["outs_h"] = outs_h if first else [torch.empty_like(t).pin_memory() for t in outs_h]
        return sl

    slots = [make_slot(True), make_slot(False)]
    # The public block calls, with each slot's arguments marshalled once
    # (tp.Prepared): a step then costs one ctypes call per block on the host.
    for sl in slots:
        sl["calls"] = []
        if "attn" in s0.e2e:
            q_w, k_w, v_w, q, k, v, _a_r, o_w, _yo = s0.e2e["attn"]
            a_r = [sl["a"][:, slice(*shards[r]["ranges"]["o_proj"])] for r in range(n)]
            xs = tp.tensor(sl["x"])
            sl["keep"] = [xs]
            if s0.attention:
                # q/k/v projections, the attention core into this slot's A, o_proj + combine
                sl["calls"].append(tp.Prepared(
                    "tp_qkv_proj", plan0.handle, ctypes.byref(xs), tp.arr(q_w), tp.arr(k_w), tp.arr(v_w),
                    tp.arr(q), tp.arr(k), tp.arr(v), sptr))
                sl["calls"].append(tp.Prepared(
                    "tp_attn_core", plan0.handle, tp.arr(q), tp.arr(k), tp.arr(v), tp.arr(a_r), 1,
                    s0.aws.data_ptr(), s0.aws.numel(), sptr))
                sl["calls"].append(tp.Prepared(
                    "tp_row_linear", n, tp.arr(a_r), tp.arr(o_w), tp.arr(sl["yo"]), combine_id, sptr))
            else:
                sl["calls"].append(tp.Prepared(
                    "tp_attn_proj", plan0.handle, ctypes.byref(xs), tp.arr(q_w), tp.arr(k_w), tp.arr(v_w),
                    tp.arr(q), tp.arr(k), tp.arr(v), tp.arr(a_r), tp.arr(o_w), tp.arr(sl["yo"]), combine_id, sptr))
        if "mlp" in s0.e2e:
            g, u, dn, _ym = s0.e2e["mlp"]
            xs = tp.tensor(sl["x"])
            sl["calls"].append(tp.Prepared(
                "tp_mlp_block", plan0.handle, ctypes.byref(xs), tp.arr(g), tp.arr(u), tp.arr(dn),
                tp.arr(sl["ym"]), combine_id, sl["ws"].data_ptr(), sl["ws"].numel(), sptr))
        if "rs_column" in s0.e2e:
            sl["calls"] += [c for (_nm, c) in s0.e2e["rs_column"][0](sl["x"], sl["ys"])]
        if "vocab" in s0.e2e:
            sl["calls"] += [c for (_nm, c) in s0.e2e["vocab"][0](sl["ids"], sl["x"], *sl["vo"])]
        if "moe" in s0.e2e:
            sl["calls"] += [c for (_nm, c) in s0.e2e["moe"][0](sl["x"], sl["rid"], sl["rw"], sl["ymoe"])]
        if "attn_core" in s0.e2e:
            sl["calls"] += [c for (_nm, c) in s0.e2e["attn_core"][0](*sl["qkv"], sl["aout"])]

    def compute(sl):
        for call in sl["calls"]:
            call()

    def results(sl):
        return (([sl["yo"][0]] if "attn" in s0.e2e else []) + ([sl["ym"][0]] if "mlp" in s0.e2e else []) +
                (list(sl["ys"]) if "rs_column" in s0.e2e else []) +
                (list(sl["vo"]) if "vocab" in s0.e2e else []) +
                ([sl["ymoe"][0]] if "moe" in s0.e2e else []) +
                ([sl["aout"]] if "attn_core" in s0.e2e else []))

    def serial_step():
        sl = slots[0]
        if copy_x:
            sl["x"].copy_(xh, non_blocking=True)
        if ah is not None:
            sl["a"].copy_(ah, non_blocking=True)
        if "ids" in sl:
            sl["ids"].copy_(idh, non_blocking=True)
        if "rid" in sl:
            sl["rid"].copy_(rih, non_blocking=True)
            sl["rw"].copy_(rwh, non_blocking=True)
        if "qkv" in sl:
            for dbuf, hbuf in zip(sl["qkv"], qkvh):
                dbuf.copy_(hbuf, non_blocking=True)
        compute(sl)
        for hbuf, dbuf in zip(sl["outs_h"], results(sl)):
            hbuf.copy_(dbuf, non_blocking=True)

    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipelined_step(i):
        b = i % 2
        sl = slots[b]
        if i >= 2:
            h2d_s.wait_event(ev_done[b])  # step i-2 has finished reading this slot's inputs
        with torch.cuda.stream(h2d_s):
            if copy_x:
                sl["x"].copy_(xh, non_blocking=True)
            if ah is not None:
                sl["a"].copy_(ah, non_blocking=True)
            if "ids" in sl:
                sl["ids"].copy_(idh, non_blocking=True)
            if "rid" in sl:
                sl["rid"].copy_(rih, non_blocking=True)
                sl["rw"].copy_(rwh, non_blocking=True)
            if "qkv" in sl:
                for dbuf, hbuf in zip(sl["qkv"], qkvh):
                    dbuf.copy_(hbuf, non_blocking=True)
            ev_in[b].record(h2d_s)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # step i-2's outputs have reached the host
        compute(sl)
        ev_done[b].record(stream)
        d2h_s.wait_event(ev_done[b])
        with torch.cuda.stream(d2h_s):
            for hbuf, dbuf in zip(sl["outs_h"], results(sl)):
                hbuf.copy_(dbuf, non_blocking=True)
            ev_out[b].record(d2h_s)

    def timed(run, steps):
        for i in range(3):
            run(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_s.wait_event(e0)
        for i in range(steps):
            run(i)
        for ev in ev_out:
            stream.wait_event(ev)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return dist_max(e0.elapsed_time(e1), world)

    e2e_ms = timed(pipelined_step, args.e2e_steps)
    # e2e.value is this loop's figure (the graph replay below is a side field)
    e2e_value = world * flops_step * args.e2e_steps / (e2e_ms / 1e3) / 1e12


    serial_ms = timed(lambda i: serial_step(), args.e2e_steps)
    serial_value = world * flops_step * args.e2e_steps / (serial_ms / 1e3) / 1e12

    # Last, since its events end up recorded inside a capture: the same pipelined
    # loop captured into a CUDA graph of G steps (both slots, every copy and
    # public call of each step) and replayed. The host issues one launch per G
    # steps instead of a few per step. Replays run back to back on the stream, so
    # copies overlap compute inside a graph but not across two.
    G = 20
    e2e_graph = {"graph": False}
    try:
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            fork = torch.cuda.Event()
            fork.record(stream)  # bring the copy streams into the capture
            h2d_s.wait_event(fork)
            d2h_s.wait_event(fork)
            for i in range(G):
                pipelined_step(i)
            for ev in ev_out:
                stream.wait_event(ev)  # join the copy streams back into the capture
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize(dev)
        reps = max(1, args.e2e_steps // G)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(reps):
            graph.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        g_ms = dist_max(g0.elapsed_time(g1), world)
        e2e_graph = {"graph": True, "steps_per_graph": G,
                     "value": round(world * flops_step * reps * G / (g_ms / 1e3) / 1e12, 3)}
    except Exception as exc:  # the stream loop's figure stands
        e2e_graph = {"graph": False, "error": str(exc)[-200:]}
        torch.cuda.synchronize(dev)
    st, word = tp.tp_device_status(sptr)
    if st != tp.TP_OK:
        raise SystemExit(f"device status {word:#x} after the end-to-end runs")

    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # The first rows of every step result of input set 0 (the last timed step's,
        # rewritten with the same values by the end-to-end loop), for the oracle
        # child to check against the same rows of its own pass.
        import tempfile
        fd, check = tempfile.mkstemp(prefix="bench_rows_", suffix=".npz")
        os.close(fd)
        try:
            rows_out = {}
            for i, t in enumerate(results(slots[0])):
                rows_out[f"r{i}"] = t[:PARITY_ROWS].float().cpu().numpy()
            np.savez(check, **rows_out)
            cpu, parity = cpu_baseline(w, args.workload, args.moe_mode, args.cpu_seconds, check)
        except Exception as exc:  # reported, not fatal
            cpu = {"error": str(exc)[-300:]}
        finally:
            os.unlink(check)

    config = {"workload": args.workload, "tokens": T, "hidden": D, "tp_size": n, "combine": mode,
              "flops_per_step": flops_step,
              "l2": (f"{R} rotating input sets of {set_bytes / 1e6:.1f} MB (> 2x L2 in total)" if R > 1 else
                     f"one input set of {set_bytes / 1e6:.1f} MB (> 2x L2)"),
              "parallelism": f"tp{n} logical ranks on one GPU; replicas across GPUs"}
    if w["kind"] == "vocab":
        config["combine"] = "all-gather of the looked-up rows and of the logits (in the kernels)"
    if w["kind"] == "moe":
        config["moe_mode"] = args.moe_mode
    for k in ("ffn", "q_heads", "kv_heads", "head_dim", "vocab", "experts", "top_k"):
        if k in w:
            config[k] = w[k]
    line = {
        "metric": "TP MLP/attn-proj block TFLOP/s and combine GB/s on 1 GB300, % of roofline",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(max_ms / K, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights, rounded to bf16)",
        "config": config,
        "phases_ms": {**{nm: round(v, 5) for nm, v in phase_ms.items()}, "step_sum": round(step_ms, 5),
                      "pass_steps": P},
        "combine": comb,
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "loop": "pipelined stream loop (two activation slots, copies on two copy streams)",
                "cuda_graph": e2e_graph,
                "d2h_bytes_per_step": d2h, "pipelined": True,
                "serial_value": round(serial_value, 3)},
        "gpu_launches": launches,
        "launches_per_step": launches / K,
        "clocks": clk.summary(),
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    line["parity"] = parity  # None when the oracle did not run beside this arm
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
    if w["kind"] == "linear_fp32":
        raise SystemExit("bench.py times the bf16 block workloads")
    why = cpu_too_large(w)
    if why:
        print(json.dumps({"impl": "reference", "unavailable": why}), flush=True)
        return
    K, W = args.steps, max(args.warmup, 0)
    # Each step is a row sample of the workload sized so that all K + W steps take
    # about --reference-seconds (two minutes by default) on the host cores.
    per_step_ms = max(5.0, 1000.0 * args.reference_seconds / (K + W))
    r = cpu_oracle_run(args.workload, args.moe_mode, 1e9, K + W, -int(per_step_ms))
    times = r["times"][W:] or r["times"]
    per_step = sum(times) / len(times)
    rows = r["rows"]
    value = sample_flops(w, rows) / per_step / 1e12
    sample = (f"{rows} of {w['T']} token rows of {args.workload} per step (fp64 oracle: {oracle_work(w)}), "
              f"{len(times)} timed passes")
    config = {"workload": args.workload, "tokens": w["T"], "hidden": w["hidden"], "tp_size": w["tp"],
              "rows_per_step": rows}
    for key in ("ffn", "q_heads", "kv_heads", "head_dim", "experts", "top_k", "vocab"):
        if key in w:
            config[key] = w[key]
    if w["kind"] == "moe":
        config["moe_mode"] = args.moe_mode
    line = {"metric": "TP MLP/attn-proj block TFLOP/s and combine GB/s on 1 GB300, % of roofline",
            "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": len(times),
            "warmup": W, "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config, "impl": "reference",
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": r["cores"],
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


DEFAULT_STEPS = {"mlp_tp2_t512": 10000, "attn_gqa_tp4_t2048": 3000, "decode_gqa_rep_tp8_t64": 6000,
                 "prefill_layer_tp8_t4096": 200, "rs_column_tp8_t4096": 600, "vocab_tp8_t4096": 200,
                 "moe_mixtral_tp8_t4096": 400, "attn_core_tp8_t4096": 1000, "decoder_layer_tp8_t4096": 200}


def main():
    args = parse_args()
    from tensor_sharded_linear_gqa_gb300 import inputs as _inputs
    kind = _inputs.WORKLOADS.get(args.workload, {}).get("kind")
    if args.combine is None:
        args.combine = "deferred" if kind == "rs_column" else "ring_fused"
    if (kind == "rs_column") != (args.combine in PIPELINE_MODES):
        raise SystemExit(f"--combine {args.combine} does not apply to workload {args.workload}")
    if args.steps is None:
        args.steps = DEFAULT_STEPS.get(args.workload, 1000) if args.impl == "native" else 20
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
