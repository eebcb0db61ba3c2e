#!/usr/bin/env python
"""Benchmark of the hybrid compressed-attention hot path on B300.

Default workload: CSA layer decode, batch 32, 65536-token context (16384
precompressed m=4 entries, bf16 indexer keys 8x64, top-128, 128-token
window, 64 query heads of dim 128).  One step = one CSA-layer decode for the
whole batch: lightning indexer + top-k, sparse MQA over the 128 selected
entries, window MQA, log-sum-exp merge to bf16.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload csa_decode|hca_decode|pair_decode|csa_prefill|hca_prefill]

Timing: steps are CUDA-graph replays on one stream, timed with CUDA events
after W warm-up steps, synchronised on both sides; consecutive steps use
different input sets (4 sets, more bytes than L2 holds) so each step reads
its keys from HBM.  Under torchrun every rank runs the same per-GPU work
(weak scaling, no data-path collective); rank 0 prints one JSON line with
the maximum time over ranks.  `--impl reference` times the fp64 CPU oracle
on the host cores instead (a bounded sample per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "decode queries/s and prefill tokens/s per layer; achieved HBM GB/s & tensor-pipe %"
NSETS = 4


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; the barrier and max-time reduction only)
# ---------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        rows = [l.split(",") for l in open(self.f.name).read().strip().splitlines() if l.strip()]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows if len(r) >= 9 for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


KERNEL_SOURCES = {"k_index_score": ["common.cuh", "index.cuh"]}


def csrc_hash(kernel: str):
    """Hash of the source files that define `kernel` (a profile goes stale when they change)."""
    d = os.path.join(ROOT, "long_context_compressed_15_b300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(f.encode())
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches these sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(f"{workload}:{kernel}")
    if not d or d.get("csrc_sha") != csrc_hash(kernel):
        return None
    return d.get("dram_bytes_per_launch")


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return 1


def time_graph(graph_runs, stream):
    """graph_runs: list of callables (graph replays); returns seconds (CUDA events)."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for g in graph_runs:
        g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


# ---------------------------------------------------------------------------
# workload: CSA decode (batch 32, 16384 entries)
# ---------------------------------------------------------------------------
class CsaDecodeBench:
    unit = "queries/s"
    name = "csa_decode"

    def __init__(self):
        from datagen.workloads import CsaDecode
        self.cfg = CsaDecode()

    def config(self):
        c = self.cfg
        return {"workload": "csa_decode: CSA layer decode, batch 32, 65536-token context, 16384 m=4 entries, "
                            "bf16 indexer keys 8x64, top-128, window 128, 64 heads x 128",
                "batch": c.B, "context_tokens": c.ctx, "entries": c.N, "H": c.H, "D": c.D, "HI": c.HI,
                "DI": c.DI, "k": c.k, "W": c.W, "l2": f"{NSETS} rotating input sets "
                f"({NSETS * self.step_bytes() / 1e6:.0f} MB touched > 126 MB L2)",
                "parallelism": "replicas (one independent batch per GPU)"}

    def units_per_step(self):
        return self.cfg.B

    def step_bytes(self):
        c = self.cfg
        per_q = (c.N * c.DI * 2 + c.HI * c.DI * 2 + c.HI * 4        # indexer keys + query + weights
                 + c.k * 2 * c.D * 2 + c.W * 2 * c.D * 2              # gathered entries + window rows
                 + c.H * c.D * 2 * 2 + c.k * 4)                       # q in, out, idx
        return c.B * per_q

    def setup(self, dev):
        from long_context_compressed_15_b300.layers import CsaLayerPlan
        c = self.cfg
        self.sets = [c.make(dev, rot=r) for r in range(NSETS)]
        self.plan = CsaLayerPlan(c.B, 1, c.H, c.D, c.N, c.k, c.W, device=dev)
        self.pos = torch.full((c.B,), c.q_pos, dtype=torch.int64, device=dev)
        self.raw0 = torch.full((c.B,), c.raw_pos0, dtype=torch.int64, device=dev)
        self.nval = torch.full((c.B,), c.N, dtype=torch.int32, device=dev)
        self.scores = torch.empty((c.B, 1, c.N), dtype=torch.float32, device=dev)

    def step(self, r):
        s = self.sets[r]
        return self.plan(s["q"], s["qI"], s["w"], self.pos, s["kI"], self.nval, s["Kc"], s["Vc"],
                         s["Kr"], s["Vr"], self.raw0)

    # dominant kernel: indexer scoring (streams 2 MiB of keys per query)
    dominant = "k_index_score"

    def dominant_launch(self, r):
        import long_context_compressed_15_b300 as lcc
        s = self.sets[r]
        lcc.lightning_index_scores(s["qI"], s["w"], self.pos, s["kI"], self.nval, 4, scores=self.scores)

    def dominant_bytes(self):
        c = self.cfg
        return c.B * (c.N * c.DI * 2 + c.HI * c.DI * 2 + c.HI * 4 + c.N * 4)

    # end to end through the public API: queries in from pinned host memory, output back
    def e2e_setup(self):
        s = self.sets[0]
        self.h_in = {k: s[k].cpu().pin_memory() for k in ("q", "qI", "w")}
        self.h_out = torch.empty(self.plan.out.shape, dtype=torch.bfloat16).pin_memory()
        return sum(v.numel() * v.element_size() for v in self.h_in.values()), \
            self.h_out.numel() * self.h_out.element_size()

    def e2e_step(self, graph0):
        s = self.sets[0]
        for k, v in self.h_in.items():
            s[k].copy_(v, non_blocking=True)
        graph0.replay()
        self.h_out.copy_(self.plan.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    # fp64 oracle on a bounded sample of the workload
    def oracle_sample(self, budget_s, max_queries=None):
        import datagen
        import oracle
        from datagen import workloads as wl
        from oracle import runs
        c = self.cfg
        s = c.seed
        done, t_oracle = 0, 0.0
        b = 0
        while t_oracle < budget_s and (max_queries is None or done < max_queries):
            bb = b % c.B
            kI = _host_rows(s, wl.T_KI, bb, c.N, c.DI)
            qI = _host_rows(s, wl.T_QI, bb, c.HI, c.DI)
            w = datagen.uniform_f32(s, wl.T_W, (c.B, c.HI)).numpy()[bb].astype(np.float64)
            q = _host_rows(s, wl.T_Q, bb, c.H, c.D, c.q_scale)
            Kr = _host_rows(s, wl.T_KR, bb, c.W, c.D)
            Vr = _host_rows(s, wl.T_VR, bb, c.W, c.D)
            t0 = time.perf_counter()
            sc = oracle.index_scores(qI, w, kI)
            idx, _ = oracle.topk_select(sc, c.k)
            t_oracle += time.perf_counter() - t0
            Kc = _host_entry_rows(s, wl.T_KC, bb * c.N + idx, c.D)
            Vc = _host_entry_rows(s, wl.T_VC, bb * c.N + idx, c.D)
            t0 = time.perf_counter()
            cO, cL = oracle.attend(q, Kc, Vc)
            sw = runs.swa_branch(q, c.q_pos, Kr, Vr, c.raw_pos0, c.W)
            oracle.merge([cO, sw["O"]], [cL, sw["lse"]])
            t_oracle += time.perf_counter() - t0
            done += 1
            b += 1
        return done, t_oracle, f"{done} decode queries of the batch (inputs regenerated on the host, untimed)"


def _host_rows(seed, tid, b, n, d, scale=1.0):
    """Rows [b*n, (b+1)*n) of a [*, d] bf16 tensor, as float64."""
    import datagen
    from oracle import runs
    idx = torch.arange(b * n * d, (b + 1) * n * d, dtype=torch.int64)
    t = datagen.normal_bf16_at(seed, tid, idx, scale).reshape(n, d)
    return runs.f64(t.view(torch.int16).numpy().view(np.uint16))


def _host_entry_rows(seed, tid, rows, d):
    import datagen
    from oracle import runs
    rows = torch.as_tensor(np.asarray(rows, dtype=np.int64))
    idx = (rows[:, None] * d + torch.arange(d)[None, :]).reshape(-1)
    t = datagen.normal_bf16_at(seed, tid, idx).reshape(-1, d)
    return runs.f64(t.view(torch.int16).numpy().view(np.uint16))


WORKLOADS = {"csa_decode": CsaDecodeBench}


# ---------------------------------------------------------------------------
def run_ours(args, ws, rank, local):
    import long_context_compressed_15_b300 as lcc
    from long_context_compressed_15_b300 import build
    build.build()
    lcc.load()
    dev = f"cuda:{local}"
    wb = WORKLOADS[args.workload]()
    wb.setup(dev)
    stream = torch.cuda.current_stream()
    G = 64  # steps per graph (a multiple of the number of input sets)
    for r in range(NSETS):  # eager warm-up of every set (also sets kernel attributes)
        wb.step(r)
    torch.cuda.synchronize()
    lcc.sync_status()
    # graphs: one per input set (single steps) and one of G steps
    singles = []
    n0 = lcc.launch_count()
    for r in range(NSETS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            wb.step(r)
        singles.append(g)
    launches_per_step = (lcc.launch_count() - n0) / NSETS
    big = torch.cuda.CUDAGraph()
    with torch.cuda.graph(big):
        for i in range(G):
            wb.step(i % NSETS)
    stream = torch.cuda.current_stream()

    def schedule(n):
        return [big] * (n // G) + [singles[i % NSETS] for i in range(n % G)]

    time_graph(schedule(args.warmup), stream)
    barrier(ws)
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    t = time_graph(schedule(args.steps), stream)
    ck = clocks.stop()
    barrier(ws)
    lcc.sync_status()
    t = max_over_ranks(t, ws)
    units = wb.units_per_step() * args.steps * ws
    value = units / t

    # dominant kernel alone, same rotation, CUDA events on its stream
    dg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dg):
        for i in range(G):
            wb.dominant_launch(i % NSETS)
    time_graph([dg] * 2, stream)
    reps = max(4, min(64, args.steps // G))
    td = time_graph([dg] * reps, stream) / (reps * G)
    pk = peaks()
    achieved = wb.dominant_bytes() / td / 1e9
    roofline = {"bound": "hbm", "kernel": wb.dominant, "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": ncu_traffic(wb.dominant, wb.name), "peak_source": pk["source"],
                "launch_us": round(td * 1e6, 3),
                "step_hbm_gbs": round(wb.step_bytes() * args.steps / t / 1e9, 1)}

    # end to end through the public API
    h2d, d2h = wb.e2e_setup()
    n_e2e = max(3, min(200, args.steps))
    for _ in range(3):
        wb.e2e_step(singles[0])
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        wb.e2e_step(singles[0])
    te = time.perf_counter() - t0
    te = max_over_ranks(te, ws)
    e2e = {"value": round(wb.units_per_step() * n_e2e * ws / te, 1), "unit": wb.unit, "steps": n_e2e,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "note": "per step: pinned H2D of the step's queries, graph replay, D2H of the bf16 output, sync"}

    line = {"metric": METRIC, "value": round(value, 1), "unit": wb.unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": wb.config(), "clocks": ck, "e2e": e2e,
            "gpu_launches": int(round(launches_per_step * args.steps)), "roofline": roofline}
    if rank == 0 and not args.no_cpu_baseline:
        n, tc, what = wb.oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": round(n / tc, 3), "unit": wb.unit, "cores": blas_threads(),
                                "kind": "oracle", "sample": what}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, ws, rank):
    if rank != 0:
        return
    wb = WORKLOADS[args.workload]()
    per_step = 1
    wb.oracle_sample(float("inf"), max_queries=min(args.warmup, 3) * per_step)
    t0 = time.perf_counter()
    n, tc, what = wb.oracle_sample(float("inf"), max_queries=args.steps * per_step)
    wall = time.perf_counter() - t0
    value = n / tc
    cores = blas_threads()
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": wb.unit, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tc / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wb.config(),
            "cpu_baseline": {"value": round(value, 3), "unit": wb.unit, "cores": cores, "kind": "oracle",
                             "sample": f"one query of the batch per step; {what}"},
            "e2e": {"value": round(n / wall, 3), "unit": wb.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8192)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="csa_decode")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        ws, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
        run_reference(args, ws, rank)
        return
    ws, rank, local = dist_setup()
    run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
