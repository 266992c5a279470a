#!/usr/bin/env python
"""Benchmark of the hybrid attention decode step at 1M-token context.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload (default): the full V4-Pro-shaped hybrid layer decode, batch 8, each
sequence with 1,048,576 cached tokens -> 262,144 CSA entries (top-1024 via a
64x128 indexer), 8,192 HCA entries and the last 128 raw tokens for SWA; 128
heads x 512, RoPE on 64 dims, sinks.  One step = one pass of every row of the
hot path: the incremental compression of the entries the newest token
completes, indexer scores, top-k, the three attention branches (with their
split combines) and the sink merge.  Inputs: seeded synthetic N(0,1) bf16.

Timing: W eager warm-up steps, then the K timed steps run as R replays (R
up to 10, dividing K) of one CUDA graph of K / R steps, with a CUDA event on
the launching stream between replays; the whole timed region sits between a
barrier + synchronize on each side, and the line reports the median, min and
max per-step time of the replays beside the whole-region figure.  A second
graph of the same steps with events around every call gives the per-call
times.  The per-step input (616 MB, mostly indexer keys) is larger than L2,
so no flush is added.  The `e2e` figure repeats the K steps through the same
public calls with the step's inputs copied from pinned host memory and the
output copied back inside the timed region.  Under torchrun every rank runs
the same per-GPU workload on its own GPU (weak scaling, no collective on the
data path); the time is the max over ranks.

--impl reference times the fp64 CPU oracle (test infrastructure, the only
reference this layer has) on one sequence of the same workload per step.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "hybrid-attn decode tokens/s @1M ctx (1 B300), HBM GB/s & % roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="hybrid_decode_1m")
    ap.add_argument("--batch", type=int, default=0, help="override B (profiling only)")
    ap.add_argument("--context", type=int, default=0, help="override L (profiling only)")
    ap.add_argument("--indexer-keys", default="bf16", choices=["bf16", "fp8", "mxfp4"],
                    help="indexer key cache: bf16, or E4M3 codes with a row scale")
    ap.add_argument("--stack", type=int, default=0,
                    help="time the decode step of N attention layers in the pages' pattern "
                         "(2 SWA, then CSA and HCA alternating; 61 for V4-Pro) instead of one "
                         "hybrid layer")
    ap.add_argument("--cache-build", action="store_true",
                    help="time building the CSA and HCA caches of one 1M-token sequence "
                         "straight from V4-Pro hidden states (d_model 7168)")
    ap.add_argument("--quantize-keys", default="", choices=["", "fp8", "mxfp4"],
                    help="time quantising the bf16 indexer key cache of the 1M-token decode "
                         "workload (8 x 262,144 rows of 128) to E4M3 rows or MXFP4 blocks")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--dense-sms", type=int, default=0,
                    help="SMs for the HCA+SWA attention beside the indexer (0: the layer's "
                         "cost model; profiling only)")
    ap.add_argument("--soak-ms", type=float, default=1500.0,
                    help="replay time under the clock sampler before the timed region")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6400.0, 1800.0, "fallback"


def workload(args):
    from sparse_attention_26_b300 import synth
    wl = synth.WORKLOADS[args.workload]
    kw = {}
    if args.batch:
        kw["B"] = args.batch
    if args.context:
        kw["L"] = args.context
    return synth.scaled(wl, **kw) if kw else wl


def step_bytes(wl, keys="bf16"):
    """Algorithmic HBM bytes of one decode step with T queries per sequence
    (the T newest tokens): per sequence, the indexer keys of every visible
    entry, every visible HCA row and the W+T-1 window rows once (the queries
    share them); per query, its k gathered CSA rows, q, iq, w and the output;
    plus the incremental compression reads/writes of the newest entries."""
    B, L, D, dI, T = wl.B, wl.L, wl.D, wl.dI, wl.T
    n_csa, n_hca = L // wl.m_csa, L // wl.m_hca
    per = 0
    if "csa" in wl.branches:
        key = key_bytes(dI, keys)
        per += n_csa * key + T * (min(wl.k, n_csa) * D * 2 + wl.HI * dI * 2 + wl.HI * 4)
        per += wl.w_csa * (D + dI + 1) * 2 + D * 2 + key
    if "hca" in wl.branches:
        per += n_hca * D * 2 + wl.w_hca * (D + 1) * 2 + D * 2
    if "swa" in wl.branches:
        per += (wl.W + T - 1) * D * 2
    per += T * (2 * wl.H * D * 2 + wl.H * 4)
    return B * per


def key_bytes(dI, keys):
    """HBM bytes of one indexer key: bf16 values, E4M3 codes and an fp32 row
    scale, or MXFP4 codes (two per byte) and an E8M0 scale per 32."""
    if keys == "bf16":
        return dI * 2
    if keys == "fp8":
        return dI + 4
    return dI // 2 + dI // 32


def indexer_bytes(wl, keys="bf16"):
    """Algorithmic bytes of one indexer launch: every visible indexer key
    read once per sequence (its queries share the scan) -- dI bf16 values,
    or dI E4M3 codes plus an fp32 row scale --, and the queries and weights.
    The fp32 scores the launch writes are implementation overhead (the
    selection's intermediate), counted apart by indexer_overhead_bytes."""
    n_csa = wl.L // wl.m_csa
    key = key_bytes(wl.dI, keys)
    return wl.B * (n_csa * key + wl.T * (wl.HI * wl.dI * 2 + wl.HI * 4))


def indexer_overhead_bytes(wl):
    """The fp32 score each (query, visible entry) pair writes for top-k."""
    return wl.B * wl.T * (wl.L // wl.m_csa) * 4


# DRAM traffic of indexer_score_kernel (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu capture of an 8 x 65,536-entry launch
# per key format (bf16 keys: 137.39 MB; E4M3 keys: 70.47 MB; MXFP4 keys:
# 35.94 MB), per entry processed; it applies only to the kernel sources it
# was taken on, checked by hash, and to one query per sequence, else the
# bench reports null.
INDEXER_TRAFFIC = {
    "bytes_per_entry": {"bf16": 137.392e6 / (8 * 65536), "fp8": 70.469e6 / (8 * 65536),
                        "mxfp4": 35.942e6 / (8 * 65536)},
    "sources": ["indexer.cu", "common.cuh"],
    "sha256": "bb3161b662091452e42a3d6f15e8f8ddc0b63598163f6dc1bd11b66ec3ccb335",
    "profile": "profiles/indexer_score_kernel_decode_8x65536.md",
}


def step_flops(wl):
    """Algorithmic flops of one pass over the T queries at positions
    [L-T, L) (causal-exact): 2*HI*dI per (query, visible entry) for the
    indexer, 4*H*D per (query, key) for each attention branch (QK^T and PV
    share the key rows); per sequence, times B."""
    import numpy as np
    t = np.arange(wl.L - wl.T, wl.L, dtype=np.int64)
    vis_c = np.minimum((t + 1) // wl.m_csa, wl.L // wl.m_csa)
    fl = {}
    if "csa" in wl.branches:
        fl["indexer"] = float(2 * wl.HI * wl.dI * vis_c.sum())
        fl["sparse"] = float(4 * wl.H * wl.D * np.minimum(vis_c, wl.k).sum())
    if "hca" in wl.branches:
        fl["hca"] = float(4 * wl.H * wl.D * ((t + 1) // wl.m_hca).sum())
    if "swa" in wl.branches:
        fl["swa"] = float(4 * wl.H * wl.D * np.minimum(t + 1, wl.W).sum())
    return {k: v * wl.B for k, v in fl.items()}


def measured_bf16_burst():
    """The bf16 peak for a kernel timed alone or inside a short pass."""
    hbm, tf, src = peaks()
    if src == "measured":
        return tf, "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    return tf, "fallback 1.8 PFLOP/s burst"


def measured_bf16_sustained():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return 1400.0


def kernel_roofline(wl, keys, per_kernel, hbm, src):
    """The roofline object of the dominant kernel.  Decode with CSA: the
    indexer against HBM (its keys are the dominant bytes).  Decode without
    CSA: the HCA attention at the ridge, with both fractions.  Prefill: the
    slowest call of the pass against the bf16 tensor peak (the sustained
    figure: it runs inside a long step)."""
    peak_src = (f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured"
                else "fallback 6.4 TB/s")
    if wl.T <= 2 and "csa" in wl.branches:
        ib = indexer_bytes(wl, keys)
        idx_ms = per_kernel["indexer"]
        achieved = ib / (idx_ms / 1e3) / 1e9
        return {"bound": "hbm", "kernel": "indexer_score_kernel", "achieved": achieved,
                "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": indexer_traffic(wl, keys),
                "traffic_source": "ncu dram bytes of an 8 x 65,536-entry launch scaled by "
                                  "entries (" + INDEXER_TRAFFIC["profile"] + ")",
                "peak_source": peak_src, "algorithmic_bytes_per_launch": ib,
                "overhead_bytes_per_launch": indexer_overhead_bytes(wl),
                "overhead": "fp32 scores written for top-k (not algorithmic)",
                "avg_launch_ms": idx_ms}
    fl = step_flops(wl)
    if wl.T <= 2:
        tf, tf_src = measured_bf16_burst()
        # HCA decode: every visible entry once per sequence, the queries and outputs
        n_h = wl.L // wl.m_hca
        by = wl.B * (n_h * wl.D * 2 + wl.T * (2 * wl.H * wl.D * 2 + wl.H * 4))
        name = "hca" if "hca" in per_kernel else "attn_fused"
        ms = per_kernel[name]
        a_gbs = by / (ms / 1e3) / 1e9
        a_tf = fl["hca"] / (ms / 1e3) / 1e12
        kern = "attn_kernel<kHca>" if name == "hca" else "attn_kernel<kFused> (HCA segment)"
        return {"bound": "hbm", "kernel": kern, "achieved": a_gbs, "peak": hbm,
                "unit": "GB/s", "frac": a_gbs / hbm, "traffic": None, "peak_source": peak_src,
                "algorithmic_bytes_per_launch": by, "avg_launch_ms": ms,
                "tensor": {"achieved": a_tf, "peak": tf, "unit": "TFLOP/s", "frac": a_tf / tf,
                           "flops_per_launch": fl["hca"]},
                "note": "at the ridge: both the HBM and the tensor fraction are given"}
    # a prefill pass lasts milliseconds, not seconds: the burst peak applies
    tf, tf_src = measured_bf16_burst()
    # the fused attention covers every attention branch in one launch
    fl = dict(fl)
    if "attn_fused" in per_kernel:
        fl["attn_fused"] = sum(v for n, v in fl.items() if n in ("sparse", "hca", "swa"))
    calls = {n: per_kernel[n] for n in fl if n in per_kernel}
    name = max(calls, key=calls.get)
    ms = calls[name]
    achieved = fl[name] / (ms / 1e3) / 1e12
    kern = {"indexer": "indexer_score_kernel", "sparse": "attn_kernel<kSparse>",
            "hca": "attn_kernel<kHca>", "swa": "attn_kernel<kSwa>",
            "attn_fused": "attn_kernel<kFused> (or the branch kind of a single key set; the "
                          "layer output written in the kernel)"}[name]
    return {"bound": "tensor", "kernel": kern, "achieved": achieved, "peak": tf,
            "unit": "TFLOP/s", "frac": achieved / tf, "traffic": None,
            "peak_source": tf_src,
            "flops_per_launch": fl[name], "avg_launch_ms": ms,
            "by_call": {n: {"ms": per_kernel[n], "tflops": fl[n] / (per_kernel[n] / 1e3) / 1e12}
                        for n in calls}}


def indexer_traffic(wl, keys="bf16"):
    """Per-launch DRAM bytes scaled from the recorded capture, or None when
    the indexer sources have changed since it was taken."""
    import hashlib
    h = hashlib.sha256()
    for f in INDEXER_TRAFFIC["sources"]:
        with open(os.path.join(ROOT, "sparse_attention_26_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if h.hexdigest() != INDEXER_TRAFFIC["sha256"]:
        return None
    if wl.T != 1 or keys not in INDEXER_TRAFFIC["bytes_per_entry"]:
        return None  # the capture is of one query per sequence, per key format
    return INDEXER_TRAFFIC["bytes_per_entry"][keys] * wl.B * (wl.L // wl.m_csa)


INDEXER_KEYS = {"bf16": "bf16", "fp8": "e4m3 codes + fp32 row scale (queries quantised alike)",
                "mxfp4": "mxfp4: e2m1 codes + e8m0 scale per 32 (queries quantised alike)"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons),
                "window": "soak replays of the same graph immediately before and during the "
                          "timed region"}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif args.impl == "ours":
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x):
    """Largest x over the ranks (the job time is the slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed_replays(K, max_replays=10):
    """(R, g): the K timed steps run as R replays of a graph of g = K / R
    steps, R the largest divisor of K up to max_replays, each replay timed on
    its own so that the line reports a median and a spread."""
    R = max(r for r in range(1, min(K, max_replays) + 1) if K % r == 0)
    return R, K // R


def job_throughput(world, units_per_rank, local_ms):
    """Whole-job throughput: the units every rank processed divided by the
    slowest rank's time.  Returns (units per second, max ms)."""
    ms = max_over_ranks(world, local_ms)
    return units_per_rank * world / (ms / 1e3), ms


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample_setup(wl, seed=0):
    """One sequence of the workload for the fp64 oracle, on seeded synthetic
    caches of the full size (values drawn directly; timing does not depend on
    them).  Raw tokens are materialised only where the step reads them."""
    import numpy as np
    import torch
    g = np.random.default_rng(seed)

    def bf(shape):
        x = torch.from_numpy(g.standard_normal(shape, dtype=np.float32)).to(torch.bfloat16)
        return x.view(torch.int16).numpy().view(np.uint16)

    L, D, dI = wl.L, wl.D, wl.dI
    n_csa, n_hca = L // wl.m_csa, L // wl.m_hca
    tail = max(wl.W, wl.w_hca, wl.w_csa) + 8
    kv_raw = np.zeros((1, L, D), np.uint16)
    ik_raw = np.zeros((1, L, dI), np.uint16)
    kv_raw[0, L - tail:] = bf((tail, D))
    ik_raw[0, L - tail:] = bf((tail, dI))
    s = dict(
        kv_raw=kv_raw, ik_raw=ik_raw,
        gate_csa=bf((1, L)), gate_hca=bf((1, L)),
        kv_c=bf((1, n_csa, D)) if "csa" in wl.branches else None,
        ik_c=bf((1, n_csa, dI)) if "csa" in wl.branches else None,
        kv_h=bf((1, max(n_hca, 1), D)),
        q=bf((1, 1, wl.H, D)), iq=bf((1, 1, wl.HI, dI)),
        w=g.standard_normal((1, 1, wl.HI)).astype(np.float32),
        sink=g.standard_normal(wl.H).astype(np.float32),
        pos=np.array([[L - 1]], np.int32),
    )
    return s


def oracle_step(wl, s, compress=True):
    """The decode step of one sequence through the oracle's stages (the query
    at s["pos"], by default L-1, and the entries its token completes)."""
    import oracle as orc
    L, t = wl.L, int(s["pos"][0, 0])
    o_list, l_list = [], []
    if "csa" in wl.branches:
        j = (t + 1) // wl.m_csa - 1
        if compress and (t + 1) % wl.m_csa == 0:
            orc.compress(s["kv_raw"], s["gate_csa"], wl.m_csa, wl.w_csa, wl.r, j, j + 1,
                         ik_raw=s["ik_raw"])
        sc = orc.indexer_scores(s["iq"], s["w"], s["ik_c"], s["pos"], wl.m_csa)
        idx = orc.topk(sc, s["pos"], wl.m_csa, wl.k)
        o, l = orc.attention(orc.KIND_SPARSE, s["q"], s["kv_c"], s["pos"], idx=idx, r=wl.r)
        o_list.append(o)
        l_list.append(l)
    if "hca" in wl.branches:
        j = (t + 1) // wl.m_hca - 1
        if compress and (t + 1) % wl.m_hca == 0:
            orc.compress(s["kv_raw"], s["gate_hca"], wl.m_hca, wl.w_hca, wl.r, j, j + 1)
        o, l = orc.attention(orc.KIND_HCA, s["q"], s["kv_h"], s["pos"], m=wl.m_hca, r=wl.r)
        o_list.append(o)
        l_list.append(l)
    if "swa" in wl.branches:
        o, l = orc.attention(orc.KIND_SWA, s["q"], s["kv_raw"], s["pos"], W=wl.W, r=wl.r)
        o_list.append(o)
        l_list.append(l)
    orc.merge(o_list, l_list, s["sink"], s["pos"], wl.r)
    return L


def cpu_baseline_prefill(wl, n_sample=None):
    """The oracle on one prefill pass of one sequence: the compression of
    every entry the pass's T tokens complete, timed in full, plus the
    per-query work timed on n_sample evenly spaced queries and extrapolated
    linearly to all T (the per-query cost grows with the causal prefix, so
    the sample spans it)."""
    import numpy as np

    import oracle as orc
    from sparse_attention_26_b300.layer import HybridLayer

    if n_sample is None:
        n_sample = 8 if "hca" in wl.branches and wl.L > (1 << 17) else 64
    s = oracle_sample_setup(wl)
    shapes = HybridLayer.__new__(HybridLayer)
    shapes.wl = wl
    t0 = time.perf_counter()
    for kind, m, w, ik in (("csa", wl.m_csa, wl.w_csa, s["ik_raw"]), ("hca", wl.m_hca, wl.w_hca,
                                                                     None)):
        if kind in wl.branches:
            j0, j1 = shapes.new_entries(kind, wl.L - 1, wl.T)
            if j1 > j0:
                orc.compress(s["kv_raw"], s["gate_" + kind], m, w, wl.r, j0, j1, ik_raw=ik)
    t_comp = time.perf_counter() - t0
    ts = np.unique(np.linspace(wl.L - wl.T, wl.L - 1, n_sample).round().astype(np.int64))
    t0 = time.perf_counter()
    for t in ts:
        s["pos"] = np.array([[t]], np.int32)
        oracle_step(wl, s, compress=False)
    per_query = (time.perf_counter() - t0) / len(ts)
    per_pass = t_comp + per_query * wl.T
    return {"value": wl.T / per_pass, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "host": host_cpu(),
            "sample": f"extrapolated: one sequence's prefill pass of {wl.name} = the compression "
                      f"of its new entries (timed in full, {t_comp:.2f} s) + {wl.T} queries x "
                      f"{per_query:.3f} s per query (mean of {len(ts)} evenly spaced queries), "
                      "single-threaded fp64 C, seeded synthetic caches",
            "seconds_per_pass": per_pass}


def host_cpu():
    """The host the oracle baseline ran on: CPU model and logical cores."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"cpu_model": model, "nproc": os.cpu_count()}


def cpu_baseline(wl, steps=1):
    if wl.T > 2:
        return cpu_baseline_prefill(wl)
    s = oracle_sample_setup(wl)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_step(wl, s)
    dt = (time.perf_counter() - t0) / steps
    return {"value": 1.0 / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "host": host_cpu(),
            "sample": f"1 query of 1 of {wl.B} sequences, 1 decode step of {wl.name} at "
                      f"full size ({wl.L}-token context: {wl.L // wl.m_csa} indexer entries, "
                      f"top-{wl.k}, "
                      f"{wl.L // wl.m_hca} HCA entries, {wl.W} SWA tokens), single-threaded "
                      "fp64 C, seeded synthetic caches",
            "seconds_per_token": dt}


# ---------------------------------------------------------------- reference arm
def run_reference(args, world, rank, budget_s=150.0):
    """The oracle on a bounded sample per step: one sequence at a context of
    L' <= L tokens (a prefix of the cache), with L' chosen so that the whole
    --steps/--warmup run fits `budget_s`; tokens/s is scaled by the work
    fraction step_bytes(L') / step_bytes(L) (indexer, HCA scans and the rest
    grow linearly with the context)."""
    if rank != 0:
        return
    from sparse_attention_26_b300 import synth
    wl = workload(args)
    one = synth.scaled(wl, B=1)

    def at(L):
        L = max(wl.m_hca * 8, (L // wl.m_hca) * wl.m_hca)
        return synth.scaled(one, L=L)

    # calibrate on 1/64 of the context
    cal = at(wl.L // 64)
    s = oracle_sample_setup(cal)
    t0 = time.perf_counter()
    oracle_step(cal, s)
    t_cal = time.perf_counter() - t0
    est_full = t_cal * step_bytes(one) / step_bytes(cal)
    n = max(1, args.steps + args.warmup)
    frac = min(1.0, budget_s / n / est_full)
    smp = at(int(wl.L * frac))
    s = oracle_sample_setup(smp)
    for _ in range(args.warmup):
        oracle_step(smp, s)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(smp, s)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    work = step_bytes(smp) / step_bytes(one)
    v = work / dt
    sample = (f"each step: 1 decode token of one sequence at context {smp.L} of {wl.L} "
              f"(work fraction {work:.4f}, tokens/s scaled by it), single-threaded fp64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 / v, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(wl, sample=sample),
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_cpu()},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def l2_note(wl, keys="bf16"):
    """How the timed inputs relate to the 126 MB L2 (no flush is added)."""
    if wl.T <= 2:
        sb = step_bytes(wl, keys)
        return f"per-step algorithmic input {sb / 1e6:.1f} MB > 126 MB L2 (no flush)"
    # a prefill pass streams its queries once and re-reads the caches for
    # every query: the caches are L2-resident by design
    q_bytes = wl.B * wl.T * (wl.H * wl.D * 2 + (wl.HI * (wl.dI * 2 + 4)
                                                  if "csa" in wl.branches else 0))
    cache = 0
    if "csa" in wl.branches:
        cache += wl.B * (wl.L // wl.m_csa) * (wl.D + wl.dI) * 2
    if "hca" in wl.branches:
        cache += wl.B * (wl.L // wl.m_hca) * wl.D * 2
    return (f"per-pass streamed queries {q_bytes / 1e6:.1f} MB > 126 MB L2; the compressed "
            f"caches ({cache / 1e6:.1f} MB) are re-read by every query and stay L2-resident "
            "by design (no flush)")


def config_dict(wl, keys="bf16", **extra):
    d = {"workload": wl.name, "batch": wl.B, "context_tokens": wl.L, "queries_per_seq": wl.T,
         "heads": wl.H, "head_dim": wl.D, "rope_dims": wl.r, "indexer": f"{wl.HI}x{wl.dI}",
         "top_k": wl.k, "csa_entries": wl.L // wl.m_csa, "hca_entries": wl.L // wl.m_hca,
         "swa_window": wl.W, "branches": list(wl.branches), "l2": l2_note(wl, keys)}
    d.update(extra)
    return d


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import torch
    from sparse_attention_26_b300 import hattn, synth
    from sparse_attention_26_b300.layer import HybridLayer

    hattn.lib()
    dev = torch.device("cuda", local)
    wl = workload(args)
    inp = synth.make_inputs(wl, seed=0, device=dev)
    raw = {k: inp[k] for k in ["kv_raw", "ik_raw", "gate_csa", "gate_hca"]}
    layer = HybridLayer(wl, raw, device=dev, indexer_keys=args.indexer_keys)
    layer.override_dense_sms = args.dense_sms
    q, iq, w, pos, sink = inp["q"], inp["iq"], inp["w"], inp["pos"], inp["sink"]
    t_new = wl.L - 1
    torch.cuda.synchronize()
    hattn.check_status()

    side = torch.cuda.Stream(device=dev)  # HCA + SWA, concurrent with the CSA chain
    for _ in range(args.warmup):
        layer.step(q, iq, w, pos, sink, t_new=t_new, side_stream=side)
    torch.cuda.synchronize()
    hattn.check_status()

    K = args.steps
    R, gsteps = timed_replays(K)
    names = layer.event_names(wl.T)
    mk = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
    rep_ev = [mk() for _ in range(R + 1)]
    n_call = min(K, 10)
    kev = [{n: (mk(), mk()) for n in names} for _ in range(n_call)]
    stream = torch.cuda.Stream(device=dev)
    # The timed graph holds g = K / R steps with no event inside, so each
    # call's kernel can start as a dependent launch of the one before it; it
    # is replayed R times with an event between replays.  A second graph
    # records events around every call (which makes each launch wait for the
    # previous one) for the per-call times and the indexer's roofline.
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        for i in range(gsteps):
            layer.step(q, iq, w, pos, sink, t_new=t_new, side_stream=side)
    g_calls = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_calls, stream=stream, capture_error_mode="relaxed"):
        for i in range(n_call):
            layer.step(q, iq, w, pos, sink, t_new=t_new, events=kev[i], side_stream=side)
    torch.cuda.synchronize()
    g.replay()  # one untimed replay of each captured graph
    g_calls.replay()
    torch.cuda.synchronize()
    hattn.check_status()

    # clock sampling: soak replays, then the timed replays
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.perf_counter() + args.soak_ms / 1e3
    while time.perf_counter() < t_end:
        g.replay()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        rep_ev[0].record(stream)
        for i in range(R):
            g.replay()
            rep_ev[i + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    hattn.check_status()
    g_calls.replay()
    torch.cuda.synchronize()
    hattn.check_status()

    value, total_ms = job_throughput(world, wl.B * wl.T * K, rep_ev[0].elapsed_time(rep_ev[R]))
    ms_step = total_ms / K
    rep_ms = [rep_ev[i].elapsed_time(rep_ev[i + 1]) / gsteps for i in range(R)]
    timing = {"timed_steps": K, "replays": R, "steps_per_replay": gsteps,
              "ms_per_step_median": statistics.median(rep_ms),
              "ms_per_step_min": min(rep_ms), "ms_per_step_max": max(rep_ms),
              "how": "CUDA events on the launching stream between graph replays; value and "
                     "ms_per_step from the whole timed region (this rank), max over ranks"}
    per_kernel = {n: statistics.mean(kev[i][n][0].elapsed_time(kev[i][n][1])
                                     for i in range(n_call))
                  for n in names}

    hbm, bf16, src = peaks()
    keys = args.indexer_keys
    sb = step_bytes(wl, keys)
    roofline = kernel_roofline(wl, keys, per_kernel, hbm, src)
    step_roof = {"alg_bytes_per_step": sb, "achieved_gbs": sb / (ms_step / 1e3) / 1e9,
                 "frac_of_measured_hbm": sb / (ms_step / 1e3) / 1e9 / hbm,
                 "roofline_ms_per_step": sb / (hbm * 1e9) * 1e3}
    if wl.T > 2:
        fl = step_flops(wl)
        tot = sum(fl.values())
        burst, _ = measured_bf16_burst()
        step_roof = {"alg_flops_per_step": tot, "flops_by_branch": fl,
                     "achieved_tflops": tot / (ms_step / 1e3) / 1e12,
                     "frac_of_measured_bf16_burst": tot / (ms_step / 1e3) / 1e12 / burst,
                     "roofline_ms_per_step": tot / (burst * 1e12) * 1e3}

    # e2e: host buffers in, output back to host, inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, world, layer, inp, wl, t_new, stream, side)

    launches = layer.launches_per_step(wl.T, t_new, side_stream=True) * K
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "fp8": "bf16 (indexer QK: e4m3)",
                  "mxfp4": "bf16 (indexer QK: mxfp4)"}[keys], "data": "synthetic",
        "config": config_dict(wl, keys,
                              parallelism=f"replicas x{world}" if world > 1 else "1 GPU",
                              step_roofline=step_roof, indexer_keys=INDEXER_KEYS[keys],
                              per_call_ms=per_kernel, timing=timing),
        "roofline": roofline, "clocks": clocks, "gpu_launches": launches,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)


def stack_bytes(wl, kinds):
    """Algorithmic HBM bytes of one decode step of the layer stack: per
    layer and sequence, its query in and output out, the new token's rows
    into the ring, the W window rows; a CSA layer adds every indexer key, the
    k gathered entries and the compression of the newest entry, an HCA layer
    every visible HCA entry and the compression of the newest entry."""
    B, L, D, dI, W = wl.B, wl.L, wl.D, wl.dI, wl.W
    n_csa, n_hca = L // wl.m_csa, L // wl.m_hca
    per = 0
    for kind in kinds:
        per += 2 * wl.H * D * 2 + wl.H * 4 + W * D * 2 + (D + 1) * 2
        if kind == "csa":
            per += n_csa * dI * 2 + min(wl.k, n_csa) * D * 2 + wl.HI * dI * 2 + wl.HI * 4
            per += dI * 2 + wl.w_csa * (D + dI + 1) * 2 + (D + dI) * 2
        elif kind == "hca":
            per += n_hca * D * 2 + wl.w_hca * (D + 1) * 2 + D * 2
    return B * per


def run_stack(args, world, rank, local):
    """The decode step of args.stack attention layers at the 1M shapes: every
    layer appends the new token to its 256-row ring, compresses the entries
    it completes (t = L-1 completes a CSA and an HCA entry) and runs its
    fused attention and merge.  The compressed caches stand for a built 1M
    context and are drawn directly (seeded N(0,1) bf16): the work of a step
    does not depend on their values."""
    import torch
    from sparse_attention_26_b300 import hattn
    from sparse_attention_26_b300.stack import DecodeStack, layer_pattern

    hattn.lib()
    dev = torch.device("cuda", local)
    wl = workload(args)
    kinds = layer_pattern(args.stack)
    stack = DecodeStack(kinds, B=wl.B, H=wl.H, D=wl.D, r=wl.r, HI=wl.HI, dI=wl.dI, k=wl.k,
                        L_max=wl.L, W=wl.W, device=dev)
    for l in range(len(kinds)):
        stack.fill_random(l, 1000 + l)
    g = torch.Generator(device=dev)
    g.manual_seed(7)

    def rnd(shape, dtype=torch.bfloat16):
        return torch.randn(shape, generator=g, device=dev).to(dtype)

    n = len(kinds)
    q = [rnd((wl.B, 1, wl.H, wl.D)) for _ in range(n)]
    iq = [rnd((wl.B, 1, wl.HI, wl.dI)) for _ in range(n)]
    w = [rnd((wl.B, 1, wl.HI), torch.float32) for _ in range(n)]
    sinks = [rnd((wl.H,), torch.float32) for _ in range(n)]
    new_kv = rnd((n, wl.B, wl.D))
    new_ik = rnd((n, wl.B, wl.dI))
    new_g = rnd((n, wl.B))
    t = wl.L - 1
    pos = torch.full((wl.B, 1), t, dtype=torch.int32, device=dev)

    def step():
        for l in range(n):
            stack.append(l, t, new_kv[l], new_ik[l], new_g[l])
        stack.step(t, q, iq, w, sinks, pos)

    torch.cuda.synchronize()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    hattn.check_status()
    K = args.steps
    stream = torch.cuda.Stream(device=dev)
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream, capture_error_mode="relaxed"):
        ev[0].record()
        for _ in range(K):
            step()
        ev[1].record()
    torch.cuda.synchronize()
    gr.replay()
    torch.cuda.synchronize()
    hattn.check_status()
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.perf_counter() + args.soak_ms / 1e3
    while time.perf_counter() < t_end:
        gr.replay()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    gr.replay()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    hattn.check_status()
    value, total_ms = job_throughput(world, wl.B * K, ev[0].elapsed_time(ev[1]))
    ms_step = total_ms / K
    hbm, _, src = peaks()
    sb = stack_bytes(wl, kinds)
    achieved = sb / (ms_step / 1e3) / 1e9
    counts = {kd: kinds.count(kd) for kd in ("swa", "csa", "hca")}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(wl, workload=f"attention_stack_{len(kinds)}_layers_1m",
                              l2=f"per-step input {sb / 1e9:.1f} GB > 126 MB L2 (no flush)",
                              layers=counts, ring_tokens=stack.ring,
                              caches="compressed caches drawn directly (seeded N(0,1) bf16) "
                                     "for a built 1M context",
                              parallelism=f"replicas x{world}" if world > 1 else "1 GPU"),
        "roofline": {"bound": "hbm", "kernel": "whole step (all layers)", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes_per_step": sb},
        "clocks": clocks, "gpu_launches": stack.launches_per_step(t) * K,
        "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_cache_build(args, world, rank, local):
    """The cache build of one sequence from hidden states: the CSA entries
    (with indexer keys) and the HCA entries of L tokens in one call,
    hattn_compress_hidden_pair (one read of the hidden states: pool each
    window, project once per entry on the tensor cores, norm and rope).
    Hidden states and weights are seeded N(0,1) bf16 (weights scaled by
    1/sqrt(d_model))."""
    import torch
    from sparse_attention_26_b300 import hattn

    hattn.lib()
    dev = torch.device("cuda", local)
    L = args.context or (1 << 20)
    dm, D, dI, r = 7168, 512, 128, 64
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    x = torch.empty((1, L, dm), dtype=torch.bfloat16, device=dev)
    for c in range(0, L, 16384):
        x[:, c:c + 16384].copy_(torch.randn((1, min(16384, L - c), dm), generator=g, device=dev))
    W_c = (torch.randn((dm, D + dI), generator=g, device=dev) / math.sqrt(dm)).to(torch.bfloat16)
    W_h = (torch.randn((dm, D), generator=g, device=dev) / math.sqrt(dm)).to(torch.bfloat16)
    g_c = torch.randn((1, L), generator=g, device=dev).to(torch.bfloat16)
    g_h = torch.randn((1, L), generator=g, device=dev).to(torch.bfloat16)
    kv_c = torch.empty((1, L // 4, D), dtype=torch.bfloat16, device=dev)
    ik_c = torch.empty((1, L // 4, dI), dtype=torch.bfloat16, device=dev)
    kv_h = torch.empty((1, L // 128, D), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(hattn.lib().hattn_compress_hidden_pair_workspace_bytes(1, L, L // 4, L // 128,
                                                                           dm),
                     dtype=torch.uint8, device=dev)

    def build():
        hattn.compress_hidden_pair(x, W_c, g_c, W_h, g_h, D=D, r=r, kv_c=kv_c, ik_c=ik_c,
                                   kv_h=kv_h, workspace=ws)

    for _ in range(args.warmup):
        build()
    torch.cuda.synchronize()
    hattn.check_status()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    sampler = ClockSampler(local)
    sampler.start()
    ev[0].record()
    for _ in range(args.steps):
        build()
    ev[1].record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    hattn.check_status()
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    hbm, _, src = peaks()
    x_bytes = L * dm * 2
    n_c, n_h = L // 4, L // 128
    # one read of the hidden states (the overlapping CSA windows and the HCA
    # window of a block re-read rows just read), the two gate rows, the entries
    alg_bytes = x_bytes + n_c * (D + dI) * 2 + n_h * D * 2 + 2 * L * 2
    # the projections: pooled rows (two bf16 parts each) times W
    flops = 2 * 2.0 * dm * (n_c * (D + dI) + n_h * D)
    achieved = alg_bytes / (ms / 1e3) / 1e9
    line = {
        "metric": "cache build tokens/s from hidden states (1 B300)", "value": L / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "cache_build_1m_from_hidden", "context_tokens": L, "d_model": dm,
                   "head_dim": D, "indexer_dim": dI, "csa_entries": n_c, "hca_entries": n_h},
        "roofline": {"bound": "hbm", "kernel": "whole build (pool both caches, project, norm)",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": None, "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes": alg_bytes, "projection_flops": flops,
                     "projection_tflops": flops / (ms / 1e3) / 1e12},
        "clocks": clocks, "e2e": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_quantize_keys(args, world, rank, local):
    """Quantising a bf16 indexer key cache in place of building it in the
    low-precision format: B x L/4 rows of 128 (8 x 262,144 for the 1M-token
    decode workload, 537 MB, larger than L2), to E4M3 codes with a row scale
    (hattn_quantize_e4m3) or to MXFP4 codes with E8M0 block scales
    (hattn_quantize_mxfp4).  Keys are seeded N(0,1) bf16."""
    import torch
    from sparse_attention_26_b300 import hattn

    hattn.lib()
    dev = torch.device("cuda", local)
    B = args.batch or 8
    N = (args.context or (1 << 20)) // 4
    dI = 128
    g = torch.Generator(device=dev)
    g.manual_seed(12)
    ik = torch.randn((B, N, dI), generator=g, device=dev).to(torch.bfloat16)
    if args.quantize_keys == "mxfp4":
        codes = torch.empty((B, N, dI // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty((B, N, dI // 32), dtype=torch.uint8, device=dev)
        out_bytes = dI // 2 + dI // 32

        def run():
            hattn.quantize_mxfp4(ik, codes=codes, scales=scales)
    else:
        codes = torch.empty((B, N, dI), dtype=torch.uint8, device=dev)
        scales = torch.empty((B, N), dtype=torch.float32, device=dev)
        out_bytes = dI + 4

        def run():
            hattn.quantize_e4m3(ik, codes=codes, scales=scales)

    for _ in range(max(args.warmup, 3)):
        run()
    torch.cuda.synchronize()
    hattn.check_status()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.perf_counter() + args.soak_ms / 1e3  # clocks under the same load
    while time.perf_counter() < t_end:
        run()
        torch.cuda.synchronize()
    ev[0].record()
    for _ in range(args.steps):
        run()
    ev[1].record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    clocks["window"] = "soak launches of the same kernel immediately before and during the timed region"
    hattn.check_status()
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    hbm, _, src = peaks()
    rows = B * N
    alg_bytes = rows * (dI * 2 + out_bytes)
    achieved = alg_bytes / (ms / 1e3) / 1e9
    kernel = ("quantize_mxfp4_kernel<128>" if args.quantize_keys == "mxfp4"
              else "quantize_e4m3_rows128_kernel")
    line = {
        "metric": "indexer key rows quantised per second (1 B300)", "value": rows / (ms / 1e3),
        "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u8" if args.quantize_keys == "mxfp4" else "u8+f32", "data": "synthetic",
        "config": {"workload": f"quantize_indexer_keys_{args.quantize_keys}", "batch": B,
                   "rows_per_sequence": N, "indexer_dim": dI, "l2": "inputs larger than L2"},
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)",
                     "algorithmic_bytes": alg_bytes,
                     "bytes_per_row": dI * 2 + out_bytes},
        "clocks": clocks, "e2e": None, "gpu_launches": args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, world, layer, inp, wl, t_new, stream, side):
    """The same steps with every step's inputs coming from pinned host memory
    and its result going back, inside the timed region.  A step's inputs (q,
    iq, w, pos and the new tokens' raw KV, indexer keys and gate logits) are
    packed in one pinned buffer and moved by one host-to-device copy; the
    new tokens' rows are then placed in the caches on the device, and out and lse
    (adjacent in one device buffer) come back by one device-to-host copy.
    Inputs and results are double-buffered so these copies overlap the
    compute of the neighbouring steps, as a serving loop would run them."""
    import torch
    K = args.steps
    dev = inp["q"].device
    raw = layer.raw
    new = slice(t_new - wl.T + 1, t_new + 1)  # the step's new tokens
    parts = [("q", inp["q"]), ("iq", inp["iq"]), ("w", inp["w"]), ("pos", inp["pos"]),
             ("kv", inp["kv_raw"][:, new]), ("ik", inp["ik_raw"][:, new]),
             ("gc", inp["gate_csa"][:, new]), ("gh", inp["gate_hca"][:, new])]
    offs, total = {}, 0
    for name, t in parts:
        nbytes = t.numel() * t.element_size()
        offs[name] = (total, nbytes, t.dtype, tuple(t.shape))
        total += (nbytes + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    for name, t in parts:
        o, n, _, _ = offs[name]
        host[o:o + n].copy_(t.contiguous().view(torch.uint8).reshape(-1).cpu())
    # two device copies of the inputs and of the result, so that the copies
    # of one step overlap the compute of its neighbours (a copy stream moves
    # step i+1's inputs in and step i-1's result out while step i runs)
    dbufs = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

    def view(buf, name):
        o, n, dt, shape = offs[name]
        return buf[o:o + n].view(dt).view(shape)

    res = layer.result_buffer(wl.T)  # out and lse, adjacent
    stage = [torch.empty(res.numel(), dtype=torch.uint8, device=dev) for _ in range(2)]
    out_h = [torch.empty(res.numel(), dtype=torch.uint8).pin_memory() for _ in range(2)]
    copy = torch.cuda.Stream(device=dev)
    mk = lambda: torch.cuda.Event(external=True)  # noqa: E731
    in_ready = [mk() for _ in range(K)]
    done = [mk() for _ in range(K)]
    out_done = [mk() for _ in range(K)]
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        ev[0].record()
        copy.wait_stream(stream)

        def fetch(i):  # on the copy stream: step i's inputs into buffer i % 2
            with torch.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(done[i - 2])  # step i-2 has finished reading that buffer
                dbufs[i % 2].copy_(host, non_blocking=True)
                in_ready[i].record(copy)

        fetch(0)
        if K > 1:
            fetch(1)
        for i in range(K):
            buf, st = dbufs[i % 2], stage[i % 2]
            stream.wait_event(in_ready[i])
            for name, cache in [("kv", "kv_raw"), ("ik", "ik_raw"), ("gc", "gate_csa"),
                                ("gh", "gate_hca")]:
                raw[cache][:, new].copy_(view(buf, name))
            layer.step(view(buf, "q"), view(buf, "iq"), view(buf, "w"), view(buf, "pos"),
                       inp["sink"], t_new=t_new, side_stream=side)
            if i >= 2:
                stream.wait_event(out_done[i - 2])  # that result copy has left the stage buffer
            st.copy_(res)
            done[i].record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(done[i])
                out_h[i % 2].copy_(st, non_blocking=True)
                out_done[i].record(copy)
            if i + 2 < K:
                fetch(i + 2)
        stream.wait_stream(copy)
        ev[1].record()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    barrier(world)
    e2e_value, ms = job_throughput(world, wl.B * wl.T * K, ev[0].elapsed_time(ev[1]))
    h2d = sum(n for _, n, _, _ in offs.values())
    out, lse = layer.buffers(wl.T)["out"], layer.buffers(wl.T)["lse"]
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
    return {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / K,
            "copies_per_step": {"h2d": 1, "d2h": 1, "d2d_token_rows": 4, "d2d_result": 1},
            "overlap": "double-buffered: step i+1's inputs and step i-1's result move on a "
                       "copy stream while step i computes"}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.stack:
        run_stack(args, world, rank, local)
    elif args.cache_build:
        run_cache_build(args, world, rank, local)
    elif args.quantize_keys:
        run_quantize_keys(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
