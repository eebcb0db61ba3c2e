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

End to end (`e2e`): the same metric through the public API with every
step's inputs copied in from pinned host memory and its output copied back.
Decode workloads run it as a serving pipeline (copies on a second stream
beside the neighbouring steps' compute, 16 steps per graph); the line also
carries the per-step synchronised variant.  Prefill workloads copy, run and
read back one step at a time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import sys
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
    """Polls SM clock and clock-event reasons through NVML on a host thread.

    Samples are taken every `period` seconds between start() and stop(), plus
    one on demand (sample_now, called right after the timed steps are
    enqueued, while the device is still running them), so even a timed region
    of a few milliseconds has samples.  Nothing is set on the device."""
    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
               ("sw_power_cap", 0x4), ("hw_power_brake_slowdown", 0x80))

    def __init__(self, device: int, period: float = 0.002):
        import ctypes
        import threading
        self.period = period
        self.samples = []
        self.stop_ev = threading.Event()
        self.th = None
        self.h = None
        self.err = None
        try:  # NVML's C API through ctypes (the driver ships libnvidia-ml)
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device), ctypes.byref(h)) != 0:
                    raise RuntimeError("no NVML handle for the device")
            self.nv, self.h, self.ct = nv, h, ctypes
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            nv.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx))  # 1 = SM clock domain
            self.max_mhz = float(mx.value)
        except Exception as e:  # no NVML: report the clocks as unavailable
            self.h = None
            self.err = f"nvml unavailable: {type(e).__name__}: {e}"

    def sample_now(self):
        if self.h is None:
            return
        ct = self.ct
        sm, r = ct.c_uint(), ct.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, ct.c_int(1), ct.byref(sm)) == 0 and \
                self.reasons_fn(self.h, ct.byref(r)) == 0:
            self.samples.append((float(sm.value), int(r.value)))
        else:
            self.err = "nvml query failed"

    def _loop(self):
        while not self.stop_ev.is_set():
            self.sample_now()
            self.stop_ev.wait(self.period)

    def start(self):
        import threading
        if self.h is not None:
            self.th = threading.Thread(target=self._loop, daemon=True)
            self.th.start()

    def stop(self):
        if self.th is not None:
            self.stop_ev.set()
            self.th.join()
        busy = [(s, r) for s, r in self.samples if not r & 0x1]  # drop samples taken while the GPU idled
        if self.h is None or not busy:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [self.err or "no samples under load"],
                    "samples": 0}
        sm = [s for s, _ in busy]
        reasons = sorted({n for _, r in busy for n, bit in self.REASONS if r & bit})
        return {"sm_mhz": float(np.median(sm)), "sm_min_mhz": min(sm), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(busy), "idle_samples": len(self.samples) - len(busy),
                "source": "nvml"}


# ---------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


KERNEL_SOURCES = {"k_index_tc": ["common.cuh", "tc.cuh", "index_tc.cuh"]}


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


def _oracle_worker(job):
    """One oracle process: its share of the sampled queries, single-threaded."""
    name, budget_s, max_queries, first, stride = job
    torch.set_num_threads(1)
    return WORKLOADS[name]().oracle_sample(budget_s, max_queries, first=first, stride=stride)


def oracle_on_host_cores(name, budget_s, max_queries=None):
    """The fp64 oracle on every host core this process may use: one spawned
    single-threaded process per core (up to 32), each on its own batch rows.
    Returns (queries, aggregate queries/s, description, workers, cpu_count)."""
    import multiprocessing as mp
    ncpu = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    nw = max(1, min(ncpu, 32))
    per = None if max_queries is None else max(1, -(-max_queries // nw))
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        # spawn, not fork: this process has already used the GPU
        with mp.get_context("spawn").Pool(nw) as pool:
            res = pool.map(_oracle_worker, [(name, budget_s, per, i, nw) for i in range(nw)])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    n = sum(r[0] for r in res)
    rate = sum(r[0] / r[1] for r in res if r[1] > 0)
    return n, rate, f"{n} {res[0][2]}; {nw} single-threaded worker processes", nw, os.cpu_count()


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return 1


def time_graph(graph_runs, stream, on_enqueued=None):
    """graph_runs: list of callables (graph replays); returns seconds (CUDA events).
    on_enqueued runs on the host after the last replay is enqueued, while the
    device is still executing the timed steps."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    # keep the device busy (~0.5 ms, outside the timed region) while the host
    # enqueues the replays, so that the region holds no launch gap
    torch.cuda._sleep(1000000)
    start.record(stream)
    for g in graph_runs:
        g.replay()
    end.record(stream)
    if on_enqueued is not None:
        on_enqueued()
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


# ---------------------------------------------------------------------------
# workloads.  Each defines one step (graph-capturable), the units it
# processes, the dominant kernel and its algorithmic bytes or FLOPs.
# ---------------------------------------------------------------------------
def _visible_pairs(T, m, q0=0, n_cap=None):
    """Sum over queries t in [q0, q0+T) of the visible compressed entries."""
    t = np.arange(q0, q0 + T, dtype=np.int64)
    v = (t + 1) // m
    if n_cap is not None:
        v = np.minimum(v, n_cap)
    return int(v.sum())


def _window_pairs(T, W, q0=0, raw_pos0=0):
    t = np.arange(q0, q0 + T, dtype=np.int64)
    lo = np.maximum(np.maximum(t - W + 1, 0), raw_pos0)
    return int((t - lo + 1).sum())


class CsaDecodeBench:
    e2e_pipeline = True  # small per-step copies: measure end to end as a serving pipeline
    unit = "queries/s"
    name = "csa_decode"
    rotate = True

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
        self.sets = [pack_inputs(c.make(dev, rot=r), ("q", "qI", "w")) for r in range(NSETS)]
        self.plan = CsaLayerPlan(c.B, 1, c.H, c.D, c.N, c.k, c.W, device=dev, m=c.m)
        # for the end-to-end pipeline: one plan (index lists, output, workspace) per input set, so that a
        # step's output can be read back while the next step runs
        self.plans = [self.plan] + [CsaLayerPlan(c.B, 1, c.H, c.D, c.N, c.k, c.W, device=dev, m=c.m)
                                    for _ in range(NSETS - 1)]
        self.pos = torch.full((c.B,), c.q_pos, dtype=torch.int64, device=dev)
        self.raw0 = torch.full((c.B,), c.raw_pos0, dtype=torch.int64, device=dev)
        self.nval = torch.full((c.B,), c.N, dtype=torch.int32, device=dev)
        self.scores = torch.empty((c.B, 1, c.N), dtype=torch.float32, device=dev)

    graph_steps = 64

    def run_steps(self, i0, n):
        for i in range(i0, i0 + n):
            s = self.sets[i % NSETS]
            self.plan(s["q"], s["qI"], s["w"], self.pos, s["kI"], self.nval, s["Kc"], s["Vc"],
                      s["Kr"], s["Vr"], self.raw0)

    def run_set(self, k):
        """One step on input set k with plan k (the end-to-end pipeline reads plan k's output back)."""
        s = self.sets[k % NSETS]
        self.plans[k % NSETS](s["q"], s["qI"], s["w"], self.pos, s["kI"], self.nval, s["Kc"], s["Vc"],
                              s["Kr"], s["Vr"], self.raw0)

    # dominant kernel: indexer scoring (streams 2 MiB of keys per query)
    dominant = "k_index_tc"
    bound = "hbm"

    def dominant_steps(self, i0, n):
        import long_context_compressed_15_b300 as lcc
        for i in range(i0, i0 + n):
            s = self.sets[i % NSETS]
            lcc.lightning_index_scores(s["qI"], s["w"], self.pos, s["kI"], self.nval, self.cfg.m, scores=self.scores)

    def dominant_work(self):
        """Algorithmic bytes of one indexer launch: keys, indexer query and head weights."""
        c = self.cfg
        return c.B * (c.N * c.DI * 2 + c.HI * c.DI * 2 + c.HI * 4)

    def dominant_extra_bytes(self):
        """Bytes the launch also moves that the roofline does not count: the fp32 scores it writes."""
        c = self.cfg
        return c.B * c.N * 4

    # end to end: the step's queries come from pinned host memory, the layer output goes back
    def e2e_io(self, k=0):
        """The step's inputs (one contiguous block: queries, indexer queries, weights) and its output."""
        return [self.sets[k % NSETS]["_in"]], self.plans[k % NSETS].out

    # fp64 oracle on a bounded sample of the workload
    def oracle_sample(self, budget_s, max_queries=None, first=0, stride=1):
        """fp64 oracle on decode queries of batch rows first, first+stride, ... (cycling)."""
        import datagen
        import oracle
        from datagen import workloads as wl
        from oracle import runs
        c = self.cfg
        s = c.seed
        done, t_oracle = 0, 0.0
        b = first
        cache = {}   # inputs of the batch rows this process cycles over, regenerated once
        while t_oracle < budget_s and (max_queries is None or done < max_queries):
            bb = b % c.B
            if bb not in cache:
                cache[bb] = dict(
                    kI=_host_rows(s, wl.T_KI, bb, c.N, c.DI), qI=_host_rows(s, wl.T_QI, bb, c.HI, c.DI),
                    w=datagen.uniform_f32(s, wl.T_W, (c.B, c.HI)).numpy()[bb].astype(np.float64),
                    q=_host_rows(s, wl.T_Q, bb, c.H, c.D, c.q_scale), Kr=_host_rows(s, wl.T_KR, bb, c.W, c.D),
                    Vr=_host_rows(s, wl.T_VR, bb, c.W, c.D))
            kI, qI, w, q, Kr, Vr = (cache[bb][x] for x in ("kI", "qI", "w", "q", "Kr", "Vr"))
            t0 = time.perf_counter()
            sc = oracle.index_scores(qI, w, kI)
            idx, _ = oracle.topk_select(sc, c.k)
            t_oracle += time.perf_counter() - t0
            key = (bb, tuple(idx.tolist()))
            if key not in cache:
                cache[key] = (_host_entry_rows(s, wl.T_KC, bb * c.N + idx, c.D),
                              _host_entry_rows(s, wl.T_VC, bb * c.N + idx, c.D))
            Kc, Vc = cache[key]
            t0 = time.perf_counter()
            cO, cL = oracle.attend(q, Kc, Vc)
            sw = runs.swa_branch(q, c.q_pos, Kr, Vr, c.raw_pos0, c.W)
            oracle.merge([cO, sw["O"]], [cL, sw["lse"]])
            t_oracle += time.perf_counter() - t0
            done += 1
            b += stride
        return done, t_oracle, ("decode queries of the batch (each process regenerates the inputs of its "
                                "batch rows once on the host, untimed, then repeats their queries)")



class DsaDecodeBench(CsaDecodeBench):
    """The DSA comparator of csa_decode: the same batch and context with m = 1, so
    the indexer scores all 65536 raw tokens of each sequence (4x the entries)."""
    name = "dsa_decode"

    def __init__(self):
        from datagen.workloads import DsaDecode
        self.cfg = DsaDecode()

    def config(self):
        d = super().config()
        d["workload"] = ("dsa_decode: the DSA comparator of csa_decode -- CSA layer decode with m=1 (the "
                         "indexer scores all 65536 raw tokens), batch 32, bf16 indexer keys 8x64, top-128, "
                         "window 128, 64 heads x 128")
        return d


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


class HcaDecodeBench:
    """HCA layer decode at 1M context: batch 8, 8192 m=128 entries + 128-token window."""
    e2e_pipeline = True
    unit = "queries/s"
    name = "hca_decode"
    dominant = "k_attn_tc<RANGE+window>+k_split_combine"
    bound = "hbm"
    graph_steps = 64

    def __init__(self):
        from datagen.workloads import HcaDecode
        self.cfg = HcaDecode()

    def config(self):
        c = self.cfg
        return {"workload": "hca_decode: HCA layer decode, batch 8, 1048576-token context, 8192 m=128 entries, "
                            "window 128, 64 heads x 128", "batch": c.B, "entries": c.N,
                "l2": f"{NSETS} rotating input sets"}

    def units_per_step(self):
        return self.cfg.B

    def setup(self, dev):
        from long_context_compressed_15_b300.layers import HcaLayerPlan
        c = self.cfg
        self.sets = [c.make(dev, rot=r) for r in range(NSETS)]
        self.plan = HcaLayerPlan(c.B, 1, c.H, c.D, c.N, c.W, device=dev)
        # for the end-to-end pipeline: one plan (output, workspace) per input set
        self.plans = [self.plan] + [HcaLayerPlan(c.B, 1, c.H, c.D, c.N, c.W, device=dev) for _ in range(NSETS - 1)]
        self.pos = torch.full((c.B,), c.q_pos, dtype=torch.int64, device=dev)
        self.raw0 = torch.full((c.B,), c.raw_pos0, dtype=torch.int64, device=dev)
        self.nval = torch.full((c.B,), c.N, dtype=torch.int32, device=dev)

    def run_steps(self, i0, n):
        for i in range(i0, i0 + n):
            s = self.sets[i % NSETS]
            self.plan(s["q"], self.pos, s["Kc"], s["Vc"], self.nval, s["Kr"], s["Vr"], self.raw0)

    def run_set(self, k):
        s = self.sets[k % NSETS]
        self.plans[k % NSETS](s["q"], self.pos, s["Kc"], s["Vc"], self.nval, s["Kr"], s["Vr"], self.raw0)

    def dominant_steps(self, i0, n):
        self.run_steps(i0, n)

    def dominant_work(self):
        c = self.cfg
        return c.B * ((c.N + c.W) * 2 * c.D * 2 + 2 * c.H * c.D * 2)

    def e2e_io(self, k=0):
        return [self.sets[k % NSETS]["q"]], self.plans[k % NSETS].out


class PairDecodeBench:
    """Interleaved CSA/HCA layer pair decode at 1M context, batch 4, NVFP4 indexer keys, 64 steps."""
    unit = "queries/s"
    name = "pair_decode"
    dominant = "k_index_tc_fp4"
    bound = "hbm"
    graph_steps = 64

    def __init__(self):
        from datagen.workloads import PairDecode
        self.cfg = PairDecode()

    def config(self):
        c = self.cfg
        return {"workload": "pair_decode: CSA+HCA layer pair decode, batch 4, 1048576-token context, "
                            "262144 CSA entries with NVFP4 indexer keys 8x64, 8192 HCA entries, top-128, "
                            "window 128, one new token per step (a CSA block pooled every 4 steps)",
                "batch": c.B, "steps_per_run": c.steps, "unit_note": "one query per sequence per step, "
                "counted once for the layer pair"}

    def units_per_step(self):
        return self.cfg.B

    def setup(self, dev):
        from long_context_compressed_15_b300.layers import PairDecodePlan
        c = self.cfg
        g = self.g = c.make(dev)
        B, W = c.B, c.W
        self.plan = PairDecodePlan(B, c.H, c.D, c.Ncap_csa, c.N_hca, c.k, W, device=dev)
        raw0 = torch.full((B,), c.raw_pos0, dtype=torch.int64, device=dev)
        # caches as they stand before step 0 (each step's token is appended by the library)
        self.csa_c = dict(Kr=g["Kr"], Vr=g["Vr"], gate=g["gate"], raw_pos0=raw0, Kc=g["Kc"], Vc=g["Vc"],
                          n_valid=torch.full((B,), c.N_csa, dtype=torch.int32, device=dev), kI=g["kI_packed"],
                          kI_scale=g["kI_scale"])
        self.hca_c = dict(Kr=g["Kr_h"], Vr=g["Vr_h"], gate=g["gate_h"], raw_pos0=raw0, Kc=g["Kc_h"], Vc=g["Vc_h"],
                          n_valid=torch.full((B,), c.N_hca, dtype=torch.int32, device=dev))
        self.pos = [torch.full((B,), c.ctx + s, dtype=torch.int64, device=dev) for s in range(c.steps)]
        self.new = []
        for s in range(c.steps):
            r = W + s
            j = min((c.ctx + s + 1) // c.m_csa - 1, c.Ncap_csa - 1)   # entry this token would complete
            self.new.append((
                dict(k=g["Kr"][:, r].contiguous(), v=g["Vr"][:, r].contiguous(), g=g["gate"][:, r].contiguous(),
                     kI=g["kI_packed"][:, j].contiguous(), kI_scale=g["kI_scale"][:, j].contiguous()),
                dict(k=g["Kr_h"][:, r].contiguous(), v=g["Vr_h"][:, r].contiguous(),
                     g=g["gate_h"][:, r].contiguous())))
        self.scores = torch.empty((c.B, 1, c.Ncap_csa), dtype=torch.float32, device=dev)

    def _step(self, s):
        g = self.g
        new_c, new_h = self.new[s]
        self.plan(self.pos[s], g["q"][s][:, None], g["qI"][s][:, None], g["w"][s][:, None], new_c, new_h,
                  self.csa_c, self.hca_c)

    def run_steps(self, i0, n):
        for i in range(i0, i0 + n):
            self._step(i % self.cfg.steps)

    def dominant_steps(self, i0, n):
        import long_context_compressed_15_b300 as lcc
        c, g = self.cfg, self.g
        for i in range(i0, i0 + n):
            s = i % c.steps
            lcc.lightning_index_scores(g["qI"][s][:, None], g["w"][s][:, None], self.pos[s], g["kI_packed"],
                                       c.N_csa, c.m_csa, kI_scale=g["kI_scale"], scores=self.scores)

    def dominant_work(self):
        """Algorithmic bytes of one indexer launch: NVFP4 keys + scales, indexer query, head weights."""
        c = self.cfg
        return c.B * (c.N_csa * (c.DI // 2 + c.DI // 16) + c.HI * c.DI * 2 + c.HI * 4)

    def dominant_extra_bytes(self):
        c = self.cfg
        return c.B * c.N_csa * 4

    def e2e_io(self):
        g = self.g
        new_c, new_h = self.new[0]
        return [g["q"][0], g["qI"][0], g["w"][0], new_c["k"], new_c["v"], new_c["g"], new_h["k"], new_h["v"],
                new_h["g"]], self.plan.hca.out


class CsaPrefillBench:
    """CSA layer prefill of one 131072-token sequence (pool, indexer + top-k, sparse + window attention)."""
    unit = "tokens/s"
    name = "csa_prefill"
    dominant = "k_index_topk_pw"
    bound = "tensor"
    graph_steps = 1

    def __init__(self):
        from datagen.workloads import CsaPrefill
        self.cfg = CsaPrefill()

    def config(self):
        c = self.cfg
        return {"workload": "csa_prefill: CSA layer prefill, 131072 tokens, causal, m=4 (32768 entries), "
                            "indexer 8x64 top-128, window 128, 64 heads x 128", "tokens": c.T}

    def units_per_step(self):
        return self.cfg.T

    def setup(self, dev):
        from long_context_compressed_15_b300.layers import CsaLayerPlan
        c = self.cfg
        self.g = c.make(dev)
        self.Kc = torch.empty((1, c.N, c.D), dtype=torch.bfloat16, device=dev)
        self.Vc = torch.empty_like(self.Kc)
        self.plan = CsaLayerPlan(1, c.T, c.H, c.D, c.N, c.k, c.W, device=dev)

    def run_steps(self, i0, n):
        import long_context_compressed_15_b300 as lcc
        c, g = self.cfg, self.g
        for _ in range(n):
            lcc.csa_compress(g["K"], g["V"], g["gate"], self.Kc, self.Vc)
            self.plan(g["q"], g["qI"], g["w"], 0, g["kI"], c.N, self.Kc, self.Vc, g["K"], g["V"], 0)

    def dominant_steps(self, i0, n):
        import long_context_compressed_15_b300 as lcc
        c, g = self.cfg, self.g
        for _ in range(n):
            lcc.lightning_index_topk(g["qI"], g["w"], 0, g["kI"], c.N, c.m, c.k, idx=self.plan.idx,
                                     workspace=self.plan.ws)

    def dominant_work(self):
        c = self.cfg
        return 2.0 * c.HI * c.DI * _visible_pairs(c.T, c.m)

    def e2e_io(self):
        g = self.g
        return [g["K"], g["V"], g["gate"], g["q"], g["qI"], g["w"], g["kI"]], self.plan.out

    def extra(self):
        import long_context_compressed_15_b300 as lcc
        c, g = self.cfg, self.g
        t = np.arange(c.T, dtype=np.int64)
        sel = np.minimum((t + 1) // c.m, c.k).sum()
        d = {"indexer_tflop": round(self.dominant_work() / 1e12, 3),
             "attention_tflop": round(4.0 * c.H * c.D * (sel + _window_pairs(c.T, c.W)) / 1e12, 3)}
        # the pooling kernel alone (HBM-bound), each launch after an L2 flush
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=g["K"].device)
        stream = torch.cuda.current_stream()
        times = []
        for i in range(6):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            lcc.csa_compress(g["K"], g["V"], g["gate"], self.Kc, self.Vc)
            e1.record(stream)
            e1.synchronize()
            if i >= 2:
                times.append(e0.elapsed_time(e1) / 1e3)
        del flush
        tp = float(np.median(times))
        nbytes = c.B * (c.T * c.D * 2 * 2 + c.T * 4 + c.N * c.D * 2 * 2)  # K, V, gates in; pooled K, V out
        hbm = peaks()["hbm_gbs"]
        d["pool"] = {"kernel": "k_pool_small<4,128,2>", "bound": "hbm", "bytes": nbytes, "launch_us": round(tp * 1e6, 3),
                     "achieved_gbs": round(nbytes / tp / 1e9, 1), "frac": round(nbytes / tp / 1e9 / hbm, 4),
                     "timing": "one launch after an L2 flush, median of 4"}
        d["fp4_indexer"] = self.fp4_indexer(stream)
        return d

    def fp4_indexer(self, stream):
        """The indexer in FP4 over the same prefill: the query quantised to NVFP4 and
        NVFP4 keys (quantiser + key expansion + the fused indexer/top-k), against the
        bf16 indexer call, each timed alone with CUDA events (median of 4 after 2)."""
        import datagen
        import long_context_compressed_15_b300 as lcc
        c, g = self.cfg, self.g
        dev = g["qI"].device
        kp, ks = datagen.nvfp4_normal(c.seed, 77, c.N, c.DI, device=dev)
        kp, ks = kp.reshape(1, c.N, c.DI // 2), ks.reshape(1, c.N, c.DI // 16)
        ws4 = torch.empty(lcc.fp4_index_topk_workspace(1, c.T, c.HI, c.DI, c.N, c.k), dtype=torch.uint8, device=dev)
        idx4 = torch.empty_like(self.plan.idx)

        def fp4():
            lcc.fp4_index_topk(g["qI"], g["w"], 0, kp, ks, c.N, c.m, c.k, idx=idx4, workspace=ws4)

        def bf16():
            self.dominant_steps(0, 1)

        def timed(fn):
            times = []
            for i in range(6):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                if i >= 2:
                    times.append(e0.elapsed_time(e1) / 1e3)
            return float(np.median(times))

        t4, t16 = timed(fp4), timed(bf16)
        lcc.sync_status()
        del ws4
        work = self.dominant_work()
        return {"call": "lcc_fp4_index_topk (k_nvfp4_quant + k_nvfp4_expand + k_index_topk_pw)",
                "ms": round(t4 * 1e3, 3), "tflops": round(work / t4 / 1e12, 1),
                "bf16_indexer_ms": round(t16 * 1e3, 3), "fp4_over_bf16_time": round(t4 / t16, 4),
                "keys": "NVFP4 N(0,1) keys, 32768 entries; query quantised to NVFP4 by the call"}


class HcaPrefillBench:
    """HCA layer prefill of a 32768-token chunk on a 1M-token context (pool 256 blocks, dense + window)."""
    unit = "tokens/s"
    name = "hca_prefill"
    dominant = "k_attn_tc<RANGE+window>"
    bound = "tensor"
    graph_steps = 1

    def __init__(self):
        from datagen.workloads import HcaPrefill
        self.cfg = HcaPrefill()

    def config(self):
        c = self.cfg
        return {"workload": "hca_prefill: HCA layer prefill of a 32768-token chunk at position 1048576, "
                            "256 new m=128 blocks pooled, 8448 entries, window 128, 64 heads x 128",
                "tokens": c.Tc}

    def units_per_step(self):
        return self.cfg.Tc

    def setup(self, dev):
        from long_context_compressed_15_b300.layers import HcaLayerPlan
        c = self.cfg
        self.g = c.make(dev)
        self.plan = HcaLayerPlan(1, c.Tc, c.H, c.D, c.Ncap, c.W, device=dev)
        self.r0 = c.W - 1

    def run_steps(self, i0, n):
        import long_context_compressed_15_b300 as lcc
        c, g, r0 = self.cfg, self.g, self.r0
        for _ in range(n):
            lcc.hca_compress(g["Kr"][:, r0:], g["Vr"][:, r0:], g["gate"][:, r0:], g["Kc"][:, c.N0:],
                             g["Vc"][:, c.N0:], n_blocks=c.Tc // c.m)
            self.plan(g["q"], c.q_pos0, g["Kc"], g["Vc"], c.Ncap, g["Kr"], g["Vr"], c.raw_pos0)

    def dominant_steps(self, i0, n):
        c, g = self.cfg, self.g
        for _ in range(n):
            self.plan(g["q"], c.q_pos0, g["Kc"], g["Vc"], c.Ncap, g["Kr"], g["Vr"], c.raw_pos0)

    def dominant_work(self):
        c = self.cfg
        keys = _visible_pairs(c.Tc, c.m, q0=c.ctx, n_cap=c.Ncap) + _window_pairs(c.Tc, c.W, q0=c.ctx,
                                                                                  raw_pos0=c.raw_pos0)
        return 4.0 * c.H * c.D * keys

    def e2e_io(self):
        g = self.g
        return [g["Kr"], g["Vr"], g["gate"], g["q"]], self.plan.out


WORKLOADS = {"csa_decode": CsaDecodeBench, "dsa_decode": DsaDecodeBench, "hca_decode": HcaDecodeBench,
             "pair_decode": PairDecodeBench, "csa_prefill": CsaPrefillBench, "hca_prefill": HcaPrefillBench}


def dsa_comparison(csa, dsa):
    """CSA (m=4) against the DSA comparator (m=1) on the same decode batch: measured
    step times and the algorithmic indexer bytes / FLOPs and cache bytes per token."""
    from datagen.workloads import CsaDecode, DsaDecode
    c, d = CsaDecode(), DsaDecode()
    kv_row = 2 * c.D * 2
    idx_c, idx_d = c.N * c.DI * 2, d.N * d.DI * 2
    return {"step_time_ratio_csa_over_dsa": round(csa["ms_per_step"] / dsa["ms_per_step"], 4),
            "indexer_bytes_ratio": round(idx_c / idx_d, 4),
            "indexer_flops_ratio": round((2 * c.HI * c.DI * c.N) / (2 * d.HI * d.DI * d.N), 4),
            "cache_bytes_per_token": {"csa_m4_bf16_keys": (kv_row + c.DI * 2) / 4,
                                      "csa_m4_nvfp4_keys": (kv_row + c.DI // 2 + c.DI // 16) / 4,
                                      "hca_m128": kv_row / 128, "dsa_m1_bf16_keys": kv_row + d.DI * 2},
            "note": "same batch, context, k and window; cache bytes exclude the fixed raw window"}


# ---------------------------------------------------------------------------
def capture(fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


class Schedule:
    """Graphs of G steps plus graphs of the remainder, replayed to run exactly n steps."""

    def __init__(self, wb):
        self.wb = wb
        self.G = wb.graph_steps
        self.big = capture(lambda: wb.run_steps(0, self.G))
        self.rem = {}

    def runs(self, n):
        r = n % self.G
        if r and r not in self.rem:
            self.rem[r] = capture(lambda: self.wb.run_steps(0, r))
        return [self.big] * (n // self.G) + ([self.rem[r]] if r else [])


def roofline_of(wb, stream, reps_hint, pk):
    """Dominant kernel alone, in a graph on the bench stream, timed with CUDA events."""
    G = wb.graph_steps
    dg = capture(lambda: wb.dominant_steps(0, G))
    time_graph([dg], stream)
    reps = max(2, reps_hint)
    td = time_graph([dg] * reps, stream) / (reps * G)
    work = wb.dominant_work()
    if wb.bound == "hbm":
        achieved, peak, unit = work / td / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = work / td / 1e12, pk["bf16_tflops"], "TFLOP/s"
    d = {"bound": wb.bound, "kernel": wb.dominant, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "traffic": ncu_traffic(wb.dominant, wb.name),
         "peak_source": pk["source"], "launch_us": round(td * 1e6, 3), "work_per_launch": work}
    if hasattr(wb, "dominant_extra_bytes"):
        d["extra_bytes"] = wb.dominant_extra_bytes()
        d["extra_note"] = "bytes the launch also writes (fp32 scores for the top-k), not counted in achieved"
    return d


def pack_inputs(d, names):
    """Re-home the per-step input tensors `names` of d as views of one contiguous device block (d["_in"]),
    so that a step's inputs arrive from the host in one copy."""
    tens = [d[n] for n in names]
    nbytes = [t.numel() * t.element_size() for t in tens]
    offs = [0]
    for n in nbytes:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    blk = torch.empty(offs[-1], dtype=torch.uint8, device=tens[0].device)
    for n, t, o, b in zip(names, tens, offs, nbytes):
        v = blk[o:o + b].view(t.dtype).view(t.shape)
        v.copy_(t)
        d[n] = v
    d["_in"] = blk
    return d


def e2e_of(wb, ws, n_steps):
    """The same metric through the public API: per step, the step's inputs are copied in from pinned
    host memory, the step runs and the layer output is read back, synchronised.  The copies and the
    step are captured into one CUDA graph (the copies are real pinned-host transfers on every replay),
    so a step costs one graph launch and one synchronisation."""
    ins, out = wb.e2e_io()
    h_in = [t.cpu().pin_memory() for t in ins]
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def io_step():
        for d, h in zip(ins, h_in):
            d.copy_(h, non_blocking=True)
        wb.run_steps(0, 1)
        h_out.copy_(out, non_blocking=True)
    g1 = capture(io_step)

    def one():
        g1.replay()
        torch.cuda.current_stream().synchronize()
    for _ in range(2):
        one()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n_steps):
        one()
    te = max_over_ranks(time.perf_counter() - t0, ws)
    return {"value": round(wb.units_per_step() * n_steps * ws / te, 1), "unit": wb.unit, "steps": n_steps,
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in h_in),
            "d2h_bytes_per_step": h_out.numel() * h_out.element_size(),
            "note": "per step: one graph replay holding the pinned H2D copies of the step's inputs, the "
                    "step and the D2H copy of the bf16 output, then a synchronisation"}


def e2e_pipelined(wb, ws, n_steps, depth=16, nbuf=NSETS):
    """The same metric through the public API as a serving pipeline: every step's inputs are copied in
    from pinned host memory (one copy, on an upload stream) into the next of `nbuf` input sets that the
    steps rotate through, and its layer output (each set has its own) is copied back to pinned host
    memory on a download stream, while the compute stream runs the neighbouring steps.  `depth` such
    steps are one CUDA graph (the copies are real transfers on every replay); the timed region is whole
    replays, synchronised at the end."""
    io = [wb.e2e_io(k) for k in range(nbuf)]
    h_in = [[t.cpu().pin_memory() for t in io[k][0]] for k in range(nbuf)]
    h_out = [torch.empty(io[k][1].shape, dtype=io[k][1].dtype).pin_memory() for k in range(nbuf)]
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_loaded = [torch.cuda.Event() for _ in range(nbuf)]
    ev_done = [torch.cuda.Event() for _ in range(nbuf)]
    ev_read = [torch.cuda.Event() for _ in range(nbuf)]

    def body():
        main = torch.cuda.current_stream()
        up.wait_stream(main)
        down.wait_stream(main)
        for i in range(depth):
            k = i % nbuf
            if i >= nbuf:
                up.wait_event(ev_done[k])             # set k's step i - nbuf has finished with it
            with torch.cuda.stream(up):
                for d, h in zip(io[k][0], h_in[k]):
                    d.copy_(h, non_blocking=True)
                ev_loaded[k].record(up)
            main.wait_event(ev_loaded[k])
            if i >= nbuf:
                main.wait_event(ev_read[k])           # set k's previous output read back
            wb.run_set(k)
            ev_done[k].record(main)
            down.wait_event(ev_done[k])
            with torch.cuda.stream(down):
                h_out[k].copy_(io[k][1], non_blocking=True)
                ev_read[k].record(down)
        main.wait_stream(up)
        main.wait_stream(down)
    g = capture(body)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, (n_steps + depth - 1) // depth)
    t0 = time.perf_counter()
    for _ in range(reps):
        g.replay()
    torch.cuda.synchronize()
    te = max_over_ranks(time.perf_counter() - t0, ws)
    steps = reps * depth
    return {"value": round(wb.units_per_step() * steps * ws / te, 1), "unit": wb.unit, "steps": steps,
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in h_in[0]),
            "d2h_bytes_per_step": h_out[0].numel() * h_out[0].element_size(),
            "note": f"serving pipeline: per step the pinned H2D copy of the step's inputs (upload stream, into "
                    f"the next of {nbuf} input sets) and the D2H copy of its bf16 output (download stream) run "
                    f"beside the neighbouring steps' compute; {depth} steps per CUDA graph, synchronised after "
                    f"the last replay"}


T0 = time.perf_counter()
T0 = time.perf_counter()


def phase(msg):
    """Progress of the run on stderr (wall seconds since start)."""
    print(f"[bench {time.perf_counter() - T0:7.1f}s] {msg}", file=sys.stderr, flush=True)


def measure_secondary(name, dev, stream, pk):
    """A short measurement of another workload (throughput + its dominant kernel's roofline)."""
    import long_context_compressed_15_b300 as lcc
    phase(f"secondary {name}")
    wb = WORKLOADS[name]()
    wb.setup(dev)
    G = wb.graph_steps
    wb.run_steps(0, min(G, NSETS))
    torch.cuda.synchronize()
    lcc.sync_status()
    n0 = lcc.launch_count()
    sch = Schedule(wb)
    launches = lcc.launch_count() - n0
    time_graph(sch.runs(G), stream)
    t1 = time_graph(sch.runs(G), stream)
    reps = max(3, int(math.ceil(0.3 / max(t1, 1e-6))))
    t = time_graph(sch.runs(G * reps), stream)
    lcc.sync_status()
    steps = G * reps
    d = {"value": round(wb.units_per_step() * steps / t, 1), "unit": wb.unit, "steps": steps,
         "ms_per_step": round(t / steps * 1e3, 5), "gpu_launches_per_step": round(launches / G, 2),
         "config": wb.config(), "roofline": roofline_of(wb, stream, reps, pk)}
    if hasattr(wb, "extra"):
        d.update(wb.extra())
    del wb, sch
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return d


def run_ours(args, ws, rank, local):
    import long_context_compressed_15_b300 as lcc
    from long_context_compressed_15_b300 import build
    build.build()
    lcc.load()
    dev = f"cuda:{local}"
    pk = peaks()
    wb = WORKLOADS[args.workload]()
    phase(f"setup {args.workload}")
    wb.setup(dev)
    stream = torch.cuda.current_stream()
    G = wb.graph_steps
    wb.run_steps(0, min(G, NSETS))  # eager warm-up (also sets kernel attributes)
    torch.cuda.synchronize()
    lcc.sync_status()
    n0 = lcc.launch_count()
    sch = Schedule(wb)
    launches_per_step = (lcc.launch_count() - n0) / G
    sch.runs(args.steps)
    sch.runs(args.warmup)

    time_graph(sch.runs(args.warmup), stream)
    barrier(ws)
    clocks = ClockSampler(torch.cuda.current_device())
    runs = sch.runs(args.steps)
    clocks.start()
    t = time_graph(runs, stream, on_enqueued=clocks.sample_now)
    ck = clocks.stop()
    barrier(ws)
    lcc.sync_status()
    t = max_over_ranks(t, ws)
    value = wb.units_per_step() * args.steps * ws / t

    # the same step repeated for at least 0.3 s, with its own clock samples, to
    # steady a short headline region
    n_rep = G * max(1, int(math.ceil(0.3 / max(t / args.steps, 1e-9) / G)))
    clocks_r = ClockSampler(torch.cuda.current_device())
    runs_r = sch.runs(n_rep)
    clocks_r.start()
    t_rep = time_graph(runs_r, stream, on_enqueued=clocks_r.sample_now)
    ck_r = clocks_r.stop()
    lcc.sync_status()
    t_rep = max_over_ranks(t_rep, ws)
    repeat = {"steps": n_rep, "seconds": round(t_rep, 4), "value": round(wb.units_per_step() * n_rep * ws / t_rep, 1),
              "ms_per_step": round(t_rep / n_rep * 1e3, 5), "clocks": ck_r}

    phase("roofline")
    roofline = roofline_of(wb, stream, max(4, min(64, args.steps // G)), pk)
    if hasattr(wb, "step_bytes"):
        roofline["step_hbm_gbs"] = round(wb.step_bytes() * args.steps / t / 1e9, 1)
    phase("e2e")
    e2e_sync = e2e_of(wb, ws, max(3, min(200, args.steps)))
    if getattr(wb, "e2e_pipeline", False):
        e2e = e2e_pipelined(wb, ws, max(16, min(512, args.steps)))
        e2e["per_step_synchronised"] = {k: e2e_sync[k] for k in ("value", "steps", "note")}
    else:
        e2e = e2e_sync

    line = {"metric": METRIC, "value": round(value, 1), "unit": wb.unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": wb.config(), "clocks": ck, "repeat": repeat, "e2e": e2e,
            "gpu_launches": int(round(launches_per_step * args.steps)), "roofline": roofline}
    if hasattr(wb, "extra"):
        line["config"].update(wb.extra())
    if rank == 0 and not args.no_cpu_baseline and hasattr(wb, "oracle_sample"):
        phase("cpu baseline")
        n, rate, what, nw, ncpu = oracle_on_host_cores(args.workload, args.cpu_budget)
        line["cpu_baseline"] = {"value": round(rate, 3), "unit": wb.unit, "cores": nw, "host_cpu_count": ncpu,
                                "kind": "oracle", "sample": f"about {args.cpu_budget:g} s of oracle work per "
                                f"worker: {what}"}
    if not args.no_secondary:
        del wb, sch
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        line["workloads"] = {}
        for name in WORKLOADS:
            if name != args.workload:
                line["workloads"][name] = measure_secondary(name, dev, stream, pk)
        w = line["workloads"]
        if args.workload == "csa_decode" and "dsa_decode" in w:
            w["dsa_decode"]["vs_csa_decode"] = dsa_comparison({"ms_per_step": line["ms_per_step"]}, w["dsa_decode"])
    phase("done")
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, ws, rank):
    if rank != 0:
        return
    wb = WORKLOADS[args.workload]()
    if not hasattr(wb, "oracle_sample"):
        print(json.dumps({"impl": "reference", "unavailable": f"no timed oracle sample for {args.workload}; "
                          "the reference arm times the fp64 oracle on csa_decode"}), flush=True)
        return
    per_step = 1
    wb.oracle_sample(float("inf"), max_queries=min(args.warmup, 3) * per_step)
    t0 = time.perf_counter()
    n, value, what, nw, ncpu = oracle_on_host_cores(args.workload, float("inf"), max_queries=args.steps * per_step)
    wall = time.perf_counter() - t0
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": wb.unit, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step / value * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": wb.config(),
            "cpu_baseline": {"value": round(value, 3), "unit": wb.unit, "cores": nw, "host_cpu_count": ncpu,
                             "kind": "oracle", "sample": f"one query of the batch per step; {what}"},
            "e2e": {"value": round(n / wall, 3), "unit": wb.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                    "note": "queries / wall time of the whole sampled run, process start-up included"}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=8192)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="csa_decode")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work per process for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the short measurements of the other workloads")
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
