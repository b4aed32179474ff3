"""Benchmark of the sparse MLA prefill forward on one node (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config h128] [--e2e-steps E] [--cpu-seconds S]
                    [--per-workload all|none|name,name,...] [--pw-steps P]

A step is one forward call over the whole workload (all tokens of the
configuration; default the T=4096 H=128 topk=512 workload the headline metric
is quoted on).  Inputs are synthetic and seeded (window + causally visible
compressed-pool index lists, bf16 N(0,1) q/kv, fp32 N(0,1) sink).  The L2 is
flushed (a 512 MB write) before every timed step; each step is timed with CUDA
events on the stream the kernels run on; the reported time is the sum over the
K steps, max over ranks.

Under torchrun (N > 1) every rank runs its own seeded batch of the workload on
its own GPU (weak scaling, no collective on the data path); ``value`` is the
FLOPs of all ranks over the slowest rank's time.

Besides the headline workload, the JSON line carries ``per_workload``: every
other workload (the small-head workload, the H=8 top-k sweep with the sink on
and off, the long H=128 workload, the GLM-shaped top-k 2048 call, the tiny
workload and decode-sized calls of 1-16 tokens), each timed the same way (L2
flushed before every timed call, CUDA events on the launching stream), with
its roofline fractions and the fp64 oracle timed on a bounded token sample;
``fp8_small_head`` / ``fp8_sweep_k640``: the same workloads on an fp8 KV
cache; and ``bwd_h128`` / ``bwd_h128_k1024`` / ``bwd_h128_t8192``: the training
backward on the page's three measured shapes (T=4096 topk=512, T=4096 topk=1024,
T=8192 topk=512; H=128).

``--impl reference`` times the fp64 CPU oracle (the only reference this op
has) on bounded token samples of the same workload, on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_mla_attention_token_gb300 import dist as sdist  # noqa: E402
from sparse_mla_attention_token_gb300 import roofline, synth  # noqa: E402

METRIC = "sparse-MLA fwd ms/call & TFLOP/s (T=4096 H=128 topk=512); % of roofline"
L2_FLUSH_BYTES = 512 << 20
KERNEL_NAMES = {0: "smallh_fwd_kernel", 1: "h128_fwd_kernel"}
KERNEL_SOURCES = {0: "smla_smallh.cu", 1: "smla_h128.cu"}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while it runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.rows: list[list[str]] = []
        self.proc = None
        self.gpu_index = gpu_index
        self.period_ms = period_ms
        self._t = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.period_ms), "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")] + [time.time()])

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = self.rows
        if self.window is not None:
            a, b = self.window
            inside = [r for r in rows if a <= r[-1] <= b + 0.05]
            rows = inside if inside else rows[-3:]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- oracle (CPU baseline)
def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return len(os.sched_getaffinity(0))


def oracle_rate(x: dict, cfg, seconds: float, start_token: int = 0) -> dict:
    """Time the fp64 oracle, as it stands, on ~``seconds`` worth of consecutive tokens.

    A short calibration call sizes the sample; the timed call then runs the
    oracle once over that many tokens.
    """
    from oracle import oracle as orc
    valid = ((x["idx"] >= 0) & (x["idx"] < cfg.num_kv)).sum(axis=1)
    cal = [(start_token + i) % cfg.T for i in range(4)]
    t0 = time.perf_counter()
    orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], tokens=cal)
    per_tok = (time.perf_counter() - t0) / len(cal)
    n = int(max(4, min(cfg.T, seconds / max(per_tok, 1e-6))))
    toks = [(start_token + i) % cfg.T for i in range(n)]
    t0 = time.perf_counter()
    orc.sparse_mla_fwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], tokens=toks)
    el = time.perf_counter() - t0
    flops = 4.0 * cfg.H * 512 * float(valid[toks].sum())
    return {"tokens": n, "seconds": el, "flops": flops, "tflops": flops / el / 1e12,
            "first_token": start_token}


# ----------------------------------------------------------------- ncu traffic
def kernel_source_sha(family: int) -> str:
    p = os.path.join(ROOT, "sparse_mla_attention_token_gb300", "csrc", KERNEL_SOURCES[family])
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def committed_traffic(family: int, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on this kernel source."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None, "no profiles/"
    sha = kernel_source_sha(family)
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as f:
            txt = f.read()
        for m in re.finditer(r"traffic_per_launch: kernel=(\S+) workload=(\S+) "
                             r"source_sha=(\S+) dram_bytes=(\d+)", txt):
            if m.group(1) == KERNEL_NAMES[family] and m.group(2) == workload:
                if m.group(3) == sha:
                    return int(m.group(4)), f"profiles/{fn}"
                return None, f"profiles/{fn} was taken on another source ({m.group(3)} != {sha})"
    return None, "no ncu summary for this kernel/workload"


# ----------------------------------------------------------------- workload
def workload_desc(cfg) -> str:
    return (f"{cfg.name}: T={cfg.T} H={cfg.H} D=512 num_kv={cfg.num_kv} "
            f"({cfg.T} token rows + {cfg.pool} pool rows, ratio {cfg.ratio}) topk={cfg.topk} "
            f"(window {cfg.window} + {cfg.topk - cfg.window} pool) {cfg.index_dtype}, "
            f"sink {'on' if cfg.sink else 'off'}"
            + (f", kv at a {cfg.kv_offset_bytes}-byte offset" if cfg.kv_offset_bytes else ""))


def config_dict(cfg, counts, extra=None) -> dict:
    d = {"workload": workload_desc(cfg), "T": cfg.T, "H": cfg.H, "D": 512,
         "num_kv": cfg.num_kv, "topk": cfg.topk, "index_dtype": cfg.index_dtype,
         "sink": cfg.sink, "valid_slots": counts.valid, "unique_rows": counts.unique_rows,
         "gflop_valid": round(counts.flops / 1e9, 3),
         "gflop_all_slots": round(counts.flops_all_slots / 1e9, 3),
         "l2": "flushed before every timed step (512 MB write, outside the timed events)"}
    if extra:
        d.update(extra)
    return d


def _physical_gpu(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


def _device_inputs(x, cfg, dev):
    import torch
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).to(dev)
    n = cfg.num_kv
    if cfg.kv_offset_bytes:
        start = cfg.kv_offset_bytes // 2
        keep = torch.zeros(start + n * 512, dtype=torch.int16, device=dev)
        keep[start:] = torch.from_numpy(x["kv"].view(np.int16).reshape(-1)).to(dev)
        kv = keep[start:].view(n, 512).view(torch.bfloat16)
    else:
        keep = None
        kv = torch.from_numpy(x["kv"].view(np.int16)).view(torch.bfloat16).to(dev)
    idx = torch.from_numpy(x["idx"]).to(dev)
    sink = torch.from_numpy(x["sink"]).to(dev) if x["sink"] is not None else None
    return q, kv, idx, sink, keep


# Workloads reported beside the headline, in this order.
PER_WORKLOAD = ["small_head", "sweep_k32", "sweep_k32_nosink", "sweep_k128", "sweep_k128_nosink",
                "sweep_k256", "sweep_k256_nosink", "sweep_k640", "sweep_k640_nosink", "h128_long",
                "glm_k2048", "tiny", "decode_h8_t1", "decode_h8_t4", "decode_h8_t16",
                "decode_h16_t1", "decode_h16_t4", "decode_h16_t16", "decode_h128_t1",
                "decode_h128_t4", "decode_h128_t16"]


def time_calls(fn, steps: int, warmup: int, flush, stream) -> list:
    """Per-call device times (ms) of ``fn``: L2 flushed before every call, CUDA
    events recorded on ``stream`` around the call only."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def measure_workload(name: str, args, dev, flush, stream, peaks: dict) -> dict:
    """One per-workload entry: device time per call, roofline, oracle baseline."""
    import torch
    from sparse_mla_attention_token_gb300 import binding as B
    cfg = synth.CONFIGS[name]
    x = synth.make_inputs(cfg)
    counts = roofline.count(x["idx"], cfg.num_kv, cfg.H, cfg.sink)
    q, kv, idx, sink, keep = _device_inputs(x, cfg, dev)
    out = torch.empty_like(q)
    lse = torch.empty((cfg.T, cfg.H), dtype=torch.float32, device=dev)
    family, splits, launches = B.sparse_mla_plan(cfg.T, cfg.H, cfg.topk)

    def step():
        B.sparse_mla_fwd(q, kv, idx, sink, x["scale"], out=out, lse=lse)

    ms = time_calls(step, args.pw_steps, 3, flush, stream)
    if B.sparse_mla_device_status() != 0:
        raise RuntimeError(f"device status not OK after {name}")
    med = statistics.median(ms)
    t = roofline.terms(counts, med * 1e-3, peaks)
    e = {"workload": workload_desc(cfg), "kernel": KERNEL_NAMES[family],
         "kernel_family": family, "splits": splits, "launches_per_call": launches,
         "ms_per_call": med, "ms_min": min(ms), "ms_max": max(ms), "steps": len(ms),
         "tflops": counts.flops / (med * 1e-3) / 1e12,
         "valid_slots": counts.valid, "unique_rows": counts.unique_rows,
         "bound": "tensor" if t["flop"]["time_s"] >= t["gathered"]["time_s"] else "hbm",
         "frac_of_roofline_gathered": t["frac_of_roofline_gathered"],
         "frac_of_roofline_unique": t["frac_of_roofline_unique"],
         "tensor_frac": t["flop"]["frac"],
         "roofline_gathered_ms": t["roofline_gathered_s"] * 1e3,
         "roofline_unique_ms": t["roofline_unique_s"] * 1e3,
         "gpu_launches": len(ms) * launches}
    if cfg.T <= 16:
        # decode-sized calls are latency-bound: the device time of one tiny kernel
        # launch (a 1-element fill, same events, same stream) is their floor
        one = flush[:1]
        floor = time_calls(lambda: one.zero_(), args.pw_steps, 3, flush, stream)
        e["launch_floor_ms"] = statistics.median(floor)
    if args.cpu_seconds > 0:
        r = oracle_rate(x, cfg, min(args.cpu_seconds, 2.0))
        e["cpu_baseline"] = {
            "value": r["tflops"], "unit": "TFLOP/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"tokens {r['first_token']}..{r['first_token'] + r['tokens'] - 1} "
                      f"({r['tokens']} tokens, {r['seconds']:.2f} s, fp64 numpy oracle)"}
    del q, kv, idx, sink, keep, out, lse
    return e


def measure_fp8(name: str, args, dev, flush, stream, peaks: dict) -> dict:
    """The forward on an fp8 KV cache of the workload's kv (e4m3 codes + one fp32
    scale per 128 columns): device time per call and the roofline with 528
    gathered bytes per valid slot (512 codes + 16 scale bytes)."""
    import torch
    from sparse_mla_attention_token_gb300 import binding as B
    cfg = synth.CONFIGS[name]
    x = synth.make_inputs(cfg)
    kv8, sc = synth.fp8_cache(x["kv"])
    counts = roofline.count(x["idx"], cfg.num_kv, cfg.H, cfg.sink)
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).to(dev)
    k8 = torch.from_numpy(kv8).to(dev)
    s8 = torch.from_numpy(sc).to(dev)
    idx = torch.from_numpy(x["idx"]).to(dev)
    sink = torch.from_numpy(x["sink"]).to(dev) if x["sink"] is not None else None
    out = torch.empty_like(q)
    lse = torch.empty((cfg.T, cfg.H), dtype=torch.float32, device=dev)

    def step():
        B.sparse_mla_fwd_fp8kv(q, k8, s8, idx, sink, x["scale"], out=out, lse=lse)

    ms = time_calls(step, args.pw_steps, 3, flush, stream)
    if B.sparse_mla_device_status() != 0:
        raise RuntimeError(f"device status not OK after fp8 {name}")
    med = statistics.median(ms)
    fixed = counts.fixed_bytes
    gathered = fixed + 528.0 * counts.valid
    t_flop = counts.flops / (peaks["bf16_tflops"] * 1e12)
    t_mem = gathered / (peaks["hbm_gbs"] * 1e9)
    family, splits, launches = B.sparse_mla_plan(cfg.T, cfg.H, cfg.topk)
    e = {"workload": workload_desc(cfg) + " (fp8 e4m3 cache, one fp32 scale per 128 columns)",
         "kernel": "smallh_fwd_kernel (fp8 cache)", "ms_per_call": med, "ms_min": min(ms),
         "ms_max": max(ms), "steps": len(ms), "tflops": counts.flops / (med * 1e-3) / 1e12,
         "bound": "tensor" if t_flop >= t_mem else "hbm",
         "frac_of_roofline_gathered": max(t_flop, t_mem) / (med * 1e-3),
         "roofline_gathered_ms": max(t_flop, t_mem) * 1e3,
         "bytes_counted": "Q+O+lse+indices+sink + 528 B (codes + scales) per valid slot",
         "splits": splits, "gpu_launches": len(ms) * launches}
    if args.cpu_seconds > 0:
        from oracle import fp8kv
        import time as _time
        n = 4
        t0 = _time.perf_counter()
        fp8kv.sparse_mla_fwd_fp8kv(x["q"], kv8, sc, x["idx"], x["sink"], x["scale"],
                                   tokens=range(cfg.T - n, cfg.T))
        per = (_time.perf_counter() - t0) / n
        n = int(max(4, min(cfg.T, min(args.cpu_seconds, 2.0) / max(per, 1e-6))))
        toks = list(range(cfg.T - n, cfg.T))
        t0 = _time.perf_counter()
        fp8kv.sparse_mla_fwd_fp8kv(x["q"], kv8, sc, x["idx"], x["sink"], x["scale"], tokens=toks)
        el = _time.perf_counter() - t0
        valid = ((x["idx"][toks] >= 0) & (x["idx"][toks] < cfg.num_kv)).sum()
        e["cpu_baseline"] = {"value": 4.0 * cfg.H * 512 * float(valid) / el / 1e12,
                             "unit": "TFLOP/s", "cores": _blas_threads(), "kind": "oracle",
                             "sample": f"tokens {toks[0]}..{toks[-1]} ({n} tokens, {el:.2f} s, "
                                       f"fp64 numpy fp8-cache oracle)"}
    del q, k8, s8, idx, sink, out, lse
    return e


def measure_backward(name: str, args, dev, flush, stream, peaks: dict) -> dict:
    """The training backward on one workload: the forward's O / lse (CUDA) and a
    seeded dO feed ``sparse_mla_bwd``; device time per call, roofline, oracle."""
    import torch
    from sparse_mla_attention_token_gb300 import binding as B
    cfg = synth.CONFIGS[name]
    x = synth.make_inputs(cfg)
    counts = roofline.count(x["idx"], cfg.num_kv, cfg.H, cfg.sink)
    q, kv, idx, sink, keep = _device_inputs(x, cfg, dev)
    out, lse = B.sparse_mla_fwd(q, kv, idx, sink, x["scale"])
    dbits = synth.make_dout(cfg)
    dout = torch.from_numpy(dbits.view(np.int16)).view(torch.bfloat16).to(dev)
    dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    dkv = torch.empty(kv.shape, dtype=torch.float32, device=dev)
    dsink = torch.empty(cfg.H, dtype=torch.float32, device=dev) if sink is not None else None
    ws = torch.empty(B.sparse_mla_bwd_workspace(cfg.T, cfg.H, cfg.topk, cfg.num_kv),
                     dtype=torch.uint8, device=dev)

    def step():
        B.sparse_mla_bwd(q, kv, idx, out, lse, dout, sink, x["scale"], dq=dq, dkv=dkv,
                         dsink=dsink, workspace=ws)

    ms = time_calls(step, args.pw_steps, 3, flush, stream)
    torch.cuda.synchronize()
    med = statistics.median(ms)
    flops = 10.0 * cfg.H * 512 * counts.valid            # S, dP, dq and the two dkv terms
    flops_all = 10.0 * cfg.T * cfg.H * cfg.topk * 512     # the page's all-slot count
    TH = cfg.T * cfg.H
    # algorithmic bytes: q, O, dO in (bf16), lse, indices, one gathered kv row per
    # valid slot, dq out (fp32), dkv out (fp32, every row)
    nbytes = (3.0 * TH * 1024 + 4.0 * TH + cfg.T * cfg.topk * x["idx"].dtype.itemsize +
              counts.valid * 1024.0 + TH * 2048.0 + cfg.num_kv * 2048.0)
    t_flop = flops / (peaks["bf16_tflops"] * 1e12)
    t_mem = nbytes / (peaks["hbm_gbs"] * 1e9)
    e = {"workload": workload_desc(cfg) + " (backward: dq, dkv, dsink)",
         "kernels": "bwd_delta, bwd_compact, bwd_sdp_tc / bwd_dq_tc / bwd_interm_tc (tcgen05; "
                    "bwd_dq / bwd_interm on mma.sync when H < 128), inverted index (count, scan, "
                    "fill), bwd_gather, bwd_dsink",
         "ms_per_call": med, "ms_min": min(ms), "ms_max": max(ms), "steps": len(ms),
         "tflops": flops / (med * 1e-3) / 1e12,
         "tflops_all_slots": flops_all / (med * 1e-3) / 1e12,
         "bound": "tensor" if t_flop >= t_mem else "hbm",
         "frac_of_roofline": max(t_flop, t_mem) / (med * 1e-3),
         "tensor_frac": t_flop / (med * 1e-3), "roofline_ms": max(t_flop, t_mem) * 1e3,
         "workspace_bytes": int(ws.numel())}
    if args.cpu_seconds > 0:
        from oracle import backward as obwd
        import time as _time
        toks = list(range(cfg.T - 4, cfg.T))    # calibrate on full-length lists
        t0 = _time.perf_counter()
        obwd.sparse_mla_bwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], dbits, tokens=toks)
        per = (_time.perf_counter() - t0) / len(toks)
        n = int(max(4, min(cfg.T, min(args.cpu_seconds, 2.0) / max(per, 1e-6))))
        toks = list(range(cfg.T - n, cfg.T))     # the last tokens: full-length lists
        t0 = _time.perf_counter()
        obwd.sparse_mla_bwd(x["q"], x["kv"], x["idx"], x["sink"], x["scale"], dbits, tokens=toks)
        el = _time.perf_counter() - t0
        valid = ((x["idx"][toks] >= 0) & (x["idx"][toks] < cfg.num_kv)).sum()
        e["cpu_baseline"] = {"value": 10.0 * cfg.H * 512 * float(valid) / el / 1e12,
                             "unit": "TFLOP/s", "cores": _blas_threads(), "kind": "oracle",
                             "sample": f"tokens {toks[0]}..{toks[-1]} ({n} tokens, {el:.2f} s, "
                                       f"fp64 numpy backward oracle)"}
    del q, kv, idx, sink, keep, out, lse, dout, dq, dkv, dsink, ws
    return e


# ----------------------------------------------------------------- our arm
def run_ours(args, cfg) -> None:
    import torch
    from sparse_mla_attention_token_gb300 import binding as B

    rank, local_rank, world = sdist.env_world()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    sdist.init("nccl")
    B.lib()

    rcfg = cfg.with_(seed=sdist.rank_seed(cfg.seed, rank))
    x = synth.make_inputs(rcfg)
    counts = roofline.count(x["idx"], cfg.num_kv, cfg.H, cfg.sink)
    q, kv, idx, sink, _keep = _device_inputs(x, cfg, dev)
    out = torch.empty_like(q)
    lse = torch.empty((cfg.T, cfg.H), dtype=torch.float32, device=dev)
    family, splits, launches = B.sparse_mla_plan(cfg.T, cfg.H, cfg.topk)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        B.sparse_mla_fwd(q, kv, idx, sink, x["scale"], out=out, lse=lse)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if B.sparse_mla_device_status() != 0:
        raise RuntimeError("device status not OK after warm-up")

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sampler = ClockSampler(_physical_gpu(local_rank))
    sampler.start()
    sdist.barrier(dev)
    torch.cuda.synchronize()
    w0 = time.time()
    for k in range(K):
        flush.zero_()                       # L2 flush, outside the events
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    sdist.barrier(dev)
    w1 = time.time()
    sampler.mark(w0, w1)
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if B.sparse_mla_device_status() != 0:
        raise RuntimeError("device status not OK after the timed steps")
    total_ms = sum(step_ms)
    max_total_ms = sdist.max_over_ranks(total_ms, dev)
    # warm-L2 reference (not the headline): the same call back to back without the flush
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(min(K, 20))]
    for a, b in wev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    warm_ms = [a.elapsed_time(b) for a, b in wev]
    all_flops = sdist.sum_over_ranks(counts.flops, dev)
    value = all_flops * K / (max_total_ms * 1e-3) / 1e12

    geom = B.sparse_mla_launch_config(cfg.T, cfg.H, cfg.topk, cfg.num_kv)

    # end to end through the public host-buffer call: pinned host inputs in,
    # results out, every step (the library overlaps the copies with the compute)
    E = args.e2e_steps
    hq = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hkv = torch.from_numpy(x["kv"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hidx = torch.from_numpy(x["idx"]).pin_memory()
    hsink = torch.from_numpy(x["sink"]).pin_memory() if sink is not None else None
    ho = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    idt = B.SMLA_IDX_INT64 if cfg.index_dtype == "int64" else B.SMLA_IDX_INT32
    ws = torch.empty(B.sparse_mla_fwd_host_workspace(cfg.T, cfg.H, cfg.topk, cfg.num_kv, idt,
                                                     sink is not None),
                     dtype=torch.uint8, device=dev) if E > 0 else None

    def e2e_step():
        B.sparse_mla_fwd_host(hq, hkv, hidx, ho, hl, hsink, ws, x["scale"], stream)

    h2d = (hq.numel() * 2 + hkv.numel() * 2 + hidx.numel() * hidx.element_size() +
           (hsink.numel() * 4 if hsink is not None else 0))
    d2h = ho.numel() * 2 + hl.numel() * 4
    e2e = None
    if E > 0:
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(E)]
        sdist.barrier(dev)
        for k in range(E):
            flush.zero_()
            eev[k][0].record(stream)
            e2e_step()
            eev[k][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = sdist.max_over_ranks(sum(a.elapsed_time(b) for a, b in eev), dev)
        e2e = {"value": all_flops * E / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms / E, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "steps": E,
               "path": "binding.sparse_mla_fwd_host (C ABI, host buffers, copies overlapped "
                       "with the compute in token chunks)"}

    # roofline of the dominant kernel (one launch per step when splits == 1)
    peaks, psrc = roofline.load_peaks(ROOT)
    launch_s = (total_ms / K / launches) * 1e-3
    t = roofline.terms(counts, launch_s * launches, peaks)
    flop_bound = t["flop"]["time_s"] >= t["gathered"]["time_s"]
    traffic, tsrc = committed_traffic(family, cfg.name)
    dom = t["flop"] if flop_bound else t["gathered"]
    roof = {"bound": "tensor" if flop_bound else "hbm", "achieved": dom["achieved"],
            "peak": dom["peak"], "unit": dom["unit"], "frac": dom["frac"], "traffic": traffic,
            "traffic_source": tsrc, "kernel": KERNEL_NAMES[family],
            "launch_ms": launch_s * 1e3,
            "peak_source": f"{psrc} (MEASURED_PEAKS.json, burst)" if psrc == "measured"
            else "fallback",
            "bytes_counted": "gathered: Q+O+lse+indices+sink + 1 KB per valid slot"}

    line = {"metric": METRIC, "impl": "ours", "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": max_total_ms / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; window + causally visible pool top-k; bf16 N(0,1))",
            "config": config_dict(cfg, counts, {"kernel_family": family, "splits": splits,
                                                "launch": geom,
                                                "parallelism": f"replicas x{world} (own batch per rank)"}),
            "e2e": e2e, "gpu_launches": K * launches, "clocks": clocks, "roofline": roof,
            "roofline_terms": t,
            "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms),
                        "max": max(step_ms),
                        "warm_l2_median": statistics.median(warm_ms) if warm_ms else None}}
    if args.per_workload != "none" and world == 1:
        names = PER_WORKLOAD if args.per_workload == "all" else args.per_workload.split(",")
        pw = {}
        pw_sampler = ClockSampler(_physical_gpu(local_rank))
        pw_sampler.start()
        p0 = time.time()
        if args.per_workload == "all":
            names = names + ["fp8_small_head", "fp8_sweep_k640", "bwd_h128", "bwd_h128_k1024",
                             "bwd_h128_t8192"]
        for n in names:
            if n == cfg.name:
                continue
            # fp8_<config>: the fp8-cache forward; bwd_<config>: the training backward
            if n.startswith("fp8_"):
                pw[n] = measure_fp8(n[4:], args, dev, flush, stream, peaks)
            elif n.startswith("bwd_"):
                pw[n] = measure_backward(n[4:], args, dev, flush, stream, peaks)
            else:
                pw[n] = measure_workload(n, args, dev, flush, stream, peaks)
            torch.cuda.empty_cache()
        pw_sampler.mark(p0, time.time())
        line["per_workload"] = pw
        line["per_workload_clocks"] = pw_sampler.stop()
    if world == 1 and rank == 0 and args.cpu_seconds > 0:
        r = oracle_rate(x, cfg, args.cpu_seconds)
        line["cpu_baseline"] = {
            "value": r["tflops"], "unit": "TFLOP/s", "cores": _blas_threads(), "kind": "oracle",
            "sample": f"tokens {r['first_token']}..{r['first_token'] + r['tokens'] - 1} of the "
                      f"{cfg.name} workload ({r['tokens']} tokens, {r['seconds']:.1f} s, fp64 "
                      f"numpy oracle)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if sdist.env_world()[2] > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------- reference arm (the oracle)
def run_reference(args, cfg) -> None:
    rank, _, world = sdist.env_world()
    if rank != 0:
        return
    x = synth.make_inputs(cfg)
    counts = roofline.count(x["idx"], cfg.num_kv, cfg.H, cfg.sink)
    per_step = max(0.5, min(20.0, args.reference_budget / max(1, args.steps + args.warmup)))
    tok = 0
    for _ in range(args.warmup):
        r = oracle_rate(x, cfg, per_step, tok)
        tok += r["tokens"]
    flops = secs = 0.0
    ntok = 0
    first = tok
    for _ in range(args.steps):
        r = oracle_rate(x, cfg, per_step, tok)
        tok += r["tokens"]
        ntok += r["tokens"]
        flops += r["flops"]
        secs += r["seconds"]
    value = flops / secs / 1e12
    sample = (f"{args.steps} steps of {secs / args.steps:.3g} s, {ntok} tokens in all "
              f"({ntok // args.steps} per step, consecutive from token {first % cfg.T}, "
              f"wrapping at {cfg.T}) of the {cfg.name} workload (fp64 numpy oracle)")
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3,
            "ms_per_call_extrapolated": counts.flops / (value * 1e12) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; window + causally visible pool top-k; bf16 N(0,1))",
            "config": config_dict(cfg, counts),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _blas_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=synth.BENCH_CONFIG, choices=sorted(synth.CONFIGS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--per-workload", default="all",
                    help="other workloads to report: all, none, or a comma-separated list "
                         "(fp8_<config>: fp8-cache forward; bwd_<config>: training backward)")
    ap.add_argument("--pw-steps", type=int, default=20,
                    help="timed calls per workload in per_workload")
    ap.add_argument("--reference-budget", type=float, default=120.0,
                    help="total seconds of oracle work for --impl reference")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = synth.CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)
    return 0


if __name__ == "__main__":
    sys.exit(main())
