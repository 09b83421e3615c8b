#!/usr/bin/env python
"""Benchmark of the fused attention forward on GB300.

One step = one ``attn_fwd`` call (the whole bf16 prefill path: Q/K/V tile
loads, S = Q K^T, mask, online softmax, O correction, O += P V, epilogue) over
the dense workload B=1 H=32 N=8192 D=128, inputs resident in HBM, L2 flushed
before every step (a 256 MiB write), each step timed with CUDA events on the
launching stream.  ``value`` is attention-forward TFLOP/s counted as
4*B*Hq*Nq*Nk*D (halved for causal).  The one JSON line printed on stdout is
kept short (every figure rounded to four significant digits) and carries:

* ``roofline``: achieved TFLOP/s of the kernel against the measured dense bf16
  peak, plus the DRAM traffic of one ncu capture of the same kernel;
* ``decode``: the split-KV decode (B=64 Hq=32 Hkv=8, Nk_b ~ U[512, 32768],
  chunk 512) in HBM GB/s against the measured copy bandwidth, for the whole
  step and for the partial-step kernel alone;
* ``causal``: the causal GQA prefill (B=4 Hq=32 Hkv=8 N=4096) in TFLOP/s;
* ``e2e``: the same metric through the C ABI with the inputs copied from pinned
  host memory and O / LSE copied back inside every timed step;
* ``cpu_baseline``: the fp64 CPU oracle timed on this host on whole heads of
  the dense workload, on one thread and on every core;
* ``w``: every other workload as ``[value, fraction of its roofline]``;
* ``fp32``: the fp32 configurations (B=2 H=4 N=64 D=32 and the B=2 H=8 sweep
  over N x D) in TFLOP/s against the derived FP32 SIMT peak;
* ``clocks``: SM clocks and throttle reasons sampled during the timed region.

``--details PATH`` also writes every workload's full record (descriptions,
step times, peaks) as JSON to PATH.  ``--impl reference`` times the CPU oracle
instead (rank 0 only).  Under torchrun every rank runs its own replica of the
workload (weak scaling, no collective on the data path); timing is the maximum
over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn-fwd TFLOP/s & % of BF16 tensor peak; split-KV decode HBM GB/s"
MAIN = dict(B=1, Hq=32, Hkv=32, N=8192, D=128, causal=False)
CAUSAL = dict(B=4, Hq=32, Hkv=8, N=4096, D=128, causal=True)
DECODE = dict(B=64, Hq=32, Hkv=8, D=128, nk_lo=512, nk_hi=32768, chunk=512)
DECODE_NAMES = ("decode", "paged", "decode_fp8", "decode_mqa", "decode_d64")
# widened decode workloads: multi-query (32 query heads on one KV head) and head dimension 64
DECODE_MQA = dict(DECODE, B=128, Hkv=1)
DECODE_D64 = dict(DECODE, D=64)
FP32 = dict(B=2, Hq=8, Hkv=8, N=4096, D=128, causal=False)
# widened prefill workloads: sliding window, chunked prefill (Nq < Nk), head dim 64
WINDOW = dict(B=1, Hq=32, Hkv=8, Nq=16384, Nk=16384, D=128, causal=True, window=4096)
CHUNKED = dict(B=1, Hq=32, Hkv=8, Nq=2048, Nk=16384, D=128, causal=True, window=0)
DENSE64 = dict(B=1, Hq=32, Hkv=32, N=8192, D=64, causal=False)
VARLEN = dict(B=32, Hq=32, Hkv=8, D=128, n_lo=512, n_hi=8192, causal=True)
# fp32 configurations: B=2 H=4 N=64 D=32, then the B=2 H=8 sweep over N x D
FP32_POINTS = [(2, 4, 64, 32)] + [(2, 8, n, d) for n in (64, 256, 1024, 4096) for d in (32, 64, 128)]
SHORT = {"paged": "paged_dec", "decode_fp8": "fp8kv_dec", "decode_mqa": "mqa_dec", "decode_d64": "d64_dec", "window": "window4k", "chunked": "chunked",
         "d64": "d64", "fp16": "fp16", "varlen": "varlen", "softcap": "softcap", "bwd": "bwd", "bwd_d64": "bwd_d64",
         "fp32": "fp32", "dense": "dense", "fp8": "fp8"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP32_SIMT_FLOP_PER_CLK_SM = 256.0   # 128 FP32 lanes x 2 (fused multiply-add)
GB300_SMS = 152
FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_bf16_dense_B1_H32_N8192.md")
KERNEL_SRC = os.path.join(ROOT, "softmax_attention_attn_gb300", "csrc", "attn_fwd_bf16.cu")


def flops(B, Hq, N, D, causal, **_):
    f = 4.0 * B * Hq * N * N * D
    return f / 2 if causal else f


def visible_pairs(Nq, Nk, causal, window):
    """Number of (query, key) pairs the mask leaves visible (bottom-right aligned)."""
    import numpy as np
    i = np.arange(Nq, dtype=np.int64)
    hi = np.minimum(Nk - 1, i + (Nk - Nq)) if causal else np.full(Nq, Nk - 1)
    lo = np.maximum(0, i + (Nk - Nq) - window + 1) if window > 0 else np.zeros(Nq, dtype=np.int64)
    return int(np.maximum(0, hi - lo + 1).sum())


def masked_flops(B, Hq, Nq, Nk, D, causal, window, **_):
    """4*D per visible (query, key) pair: the exact count for window / chunked workloads."""
    return 4.0 * B * Hq * D * visible_pairs(Nq, Nk, causal, window)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=["dense", "causal", "decode", "fp32", "window", "chunked", "d64",
                                           "paged", "fp16", "varlen", "decode_fp8", "softcap", "bwd",
                                           "decode_mqa", "decode_d64", "bwd_d64", "fp8"],
                    default="dense",
                    help="workload of the timed loop (default: the dense bf16 prefill)")
    ap.add_argument("--no-extras", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-oracle sample budget")
    ap.add_argument("--details", default=None, help="also write every workload's full record to this JSON file")
    ap.add_argument("--cpu-worker", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="sequences in the decode workload (smaller for profiler captures)")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it matches the kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    src_hash = hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()[:16]
    fields = {}
    for line in open(TRAFFIC_FILE):
        if ": " in line and line.startswith("- "):
            k, v = line[2:].split(": ", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel source sha256[:16]") != src_hash:
        return None
    try:
        return float(fields["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        load = [r for r in rows if r[2] > 0.3 * max(x[2] for x in rows)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows), "samples": len(load), "reasons": reasons}


# ------------------------------------------------------------------ timing helpers
def time_steps(torch, fn, steps, warmup, flush, stream):
    """Per-step device time (ms) with an L2 flush before every step (not timed)."""
    for _ in range(warmup):
        flush.zero_()
        fn()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


MAIN_CONFIG = {"workload": "bf16 dense prefill B=1 H=32 N=8192 D=128 (non-causal)", "global_batch": 1,
               "seq_len": MAIN["N"], "parallelism": "single"}


def host_cores():
    return len(os.sched_getaffinity(0))


def cpu_oracle_heads(threads, budget_s, seed=0):
    """Whole heads of the dense workload through the fp64 oracle on ``threads`` threads.

    Heads are handed out one at a time until ``budget_s`` has elapsed (heads in
    flight finish).  Input generation is not timed.  Returns (heads, seconds).
    Run in a process whose BLAS is limited to one thread (``--cpu-worker``), so
    that ``threads`` is the number of cores actually used.
    """
    import threading
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    from softmax_attention_attn_gb300 import inputs
    q, k, v = inputs.prefill_inputs(1, MAIN["Hq"], MAIN["Hkv"], MAIN["N"], MAIN["N"], MAIN["D"], "bf16", seed)
    scale = 1 / math.sqrt(MAIN["D"])
    lock = threading.Lock()
    state = {"next": 0, "done": 0}
    t0 = time.perf_counter()

    def worker():
        while True:
            with lock:
                h = state["next"]
                if h >= MAIN["Hq"] or time.perf_counter() - t0 >= budget_s:
                    return
                state["next"] = h + 1
            oracle.attention_forward(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], scale)
            with lock:
                state["done"] += 1

    with ThreadPoolExecutor(threads) as ex:
        for f in [ex.submit(worker) for _ in range(threads)]:
            f.result()
    return state["done"], time.perf_counter() - t0


def cpu_worker_main(threads, budget_s):
    """``bench.py --cpu-worker N``: print one JSON object with the oracle's heads and seconds."""
    heads, dt = cpu_oracle_heads(threads, budget_s)
    print(json.dumps({"threads": threads, "heads": heads, "seconds": dt}), flush=True)


def cpu_oracle_run(threads, budget_s):
    """The oracle on ``threads`` threads in a child process with one BLAS thread per call."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    for key in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(key, None)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", str(threads),
                        "--cpu-seconds", str(budget_s)], capture_output=True, text=True, env=env,
                       timeout=budget_s * 6 + 300)
    if r.returncode != 0:
        raise RuntimeError(f"CPU oracle worker failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(budget_s):
    """fp64 oracle on whole heads of the dense workload: one thread, then every core."""
    f_head = flops(1, 1, MAIN["N"], MAIN["D"], False)
    n = host_cores()
    one = cpu_oracle_run(1, budget_s)
    alln = cpu_oracle_run(n, budget_s)
    v1 = one["heads"] * f_head / one["seconds"] / 1e12
    vn = alln["heads"] * f_head / alln["seconds"] / 1e12
    return {"value": sig(vn), "unit": "TFLOP/s", "cores": n, "kind": "oracle", "value_1_core": sig(v1),
            "sample": f"fp64 oracle, whole heads of the dense workload: {alln['heads']} heads in "
                      f"{alln['seconds']:.1f} s on {n} threads, {one['heads']} in {one['seconds']:.1f} s on 1"}


def sig(x, n=4):
    """``x`` rounded to ``n`` significant digits (None stays None)."""
    if x is None or not math.isfinite(x) or x == 0:
        return x
    return round(x, n - 1 - int(math.floor(math.log10(abs(x)))))


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    """The CPU oracle, as it stands, on a bounded sample of the dense workload per step.

    A step is R query rows (against all 8192 keys) of one head, split over every
    core in blocks of 256 rows; R is set from one calibration step so that the
    whole run takes about a minute.
    """
    if rank != 0:
        return
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    from softmax_attention_attn_gb300 import inputs
    q, k, v = inputs.prefill_inputs(1, MAIN["Hq"], MAIN["Hkv"], MAIN["N"], MAIN["N"], MAIN["D"], "bf16", 0)
    scale = 1 / math.sqrt(MAIN["D"])
    n = host_cores()
    blk = 256
    rng = np.random.default_rng(0)
    ex = ThreadPoolExecutor(n)

    def step(rows):
        h = int(rng.integers(MAIN["Hq"]))
        i0 = int(rng.integers(0, MAIN["N"] - rows + 1))
        parts = [(i, min(i + blk, i0 + rows)) for i in range(i0, i0 + rows, blk)]
        list(ex.map(lambda p: oracle.attention_forward(q[:, h:h + 1, p[0]:p[1]], k[:, h:h + 1],
                                                       v[:, h:h + 1], scale), parts))

    t0 = time.perf_counter()
    step(n * blk)
    per_row = (time.perf_counter() - t0) / (n * blk)
    target = min(2.0, 60.0 / (args.steps + args.warmup))
    rows = int(max(blk, min(MAIN["N"], target / per_row)) // blk * blk)
    for _ in range(args.warmup):
        step(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(rows)
    dt = time.perf_counter() - t0
    ex.shutdown()
    f = 4.0 * rows * MAIN["N"] * MAIN["D"] * args.steps
    value = sig(f / dt / 1e12)
    sample = (f"{rows} query rows x all 8192 keys of one head of the dense workload per step, fp64 oracle "
              f"on {n} threads (blocks of {blk} rows, one BLAS thread each)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sig(dt / args.steps * 1e3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": dict(MAIN_CONFIG),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": n, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GB300 arm
WORKLOAD_NAMES = {
    "dense": "bf16 dense prefill B=1 H=32 N=8192 D=128 (non-causal)",
    "causal": "bf16 causal GQA prefill B=4 Hq=32 Hkv=8 N=4096 D=128",
    "decode": "bf16 split-KV decode B=64 Hq=32 Hkv=8 D=128, Nk_b~U[512,32768], chunk 512",
    "fp32": "fp32 dense prefill B=2 H=8 N=4096 D=128",
    "window": "bf16 causal sliding-window (4096) prefill B=1 Hq=32 Hkv=8 N=16384 D=128",
    "chunked": "bf16 chunked prefill (causal, bottom-right) B=1 Hq=32 Hkv=8 Nq=2048 Nk=16384 D=128",
    "d64": "bf16 dense prefill B=1 H=32 N=8192 D=64 (non-causal)",
    "fp16": "fp16 dense prefill B=1 H=32 N=8192 D=128 (non-causal)",
    "varlen": "bf16 ragged causal prefill, 32 sequences of U[512,8192] tokens, Hq=32 Hkv=8 D=128",
    "paged": "bf16 split-KV decode on a paged cache (page 256) B=64 Hq=32 Hkv=8 D=128, Nk_b~U[512,32768], chunk 512",
    "decode_fp8": "split-KV decode on an fp8 E4M3 KV cache (bf16 Q) B=64 Hq=32 Hkv=8 D=128, Nk_b~U[512,32768], "
                  "chunk 512",
    "softcap": "bf16 dense prefill B=1 H=32 N=8192 D=128 with softcap 50 and per-head attention sinks",
    "decode_mqa": "bf16 multi-query split-KV decode B=128 Hq=32 Hkv=1 D=128, Nk_b~U[512,32768], chunk 512",
    "decode_d64": "bf16 split-KV decode B=64 Hq=32 Hkv=8 D=64, Nk_b~U[512,32768], chunk 512",
    "bwd": "bf16 backward (dQ, dK, dV) B=1 H=32 N=8192 D=128 (non-causal); FLOPs = 2.5 x forward",
    "bwd_d64": "bf16 backward (dQ, dK, dV) B=1 H=32 N=8192 D=64 (non-causal); FLOPs = 2.5 x forward",
    "fp8": "fp8 E4M3 Q/K/V dense prefill B=1 H=32 N=8192 D=128 (non-causal): Q K^T on E4M3 tensor cores, "
           "P V in bf16 after V is widened (2 launches)",
}


def make_workload(name, dev, seed, peaks, peak_src, sm_max_mhz, decode_batch=None):
    """Inputs resident on ``dev`` plus the step function and its roofline terms."""
    import torch
    from softmax_attention_attn_gb300 import binding, inputs
    w = {"name": name, "desc": WORKLOAD_NAMES[name]}
    if name in ("bwd", "bwd_d64"):
        c = MAIN if name == "bwd" else DENSE64
        host = inputs.prefill_inputs(c["B"], c["Hq"], c["Hkv"], c["N"], c["N"], c["D"], "bf16", seed)
        q, k, v = (x.to(dev) for x in host)
        do = torch.randn(c["B"], c["Hq"], c["N"], c["D"], generator=torch.Generator("cpu").manual_seed(seed + 9))
        do = do.to(torch.bfloat16).to(dev)
        o, lse = binding.attn_fwd(q, k, v)
        dq = torch.empty(q.shape, device=dev, dtype=torch.float32)
        dk, dv = torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(binding.lib().attn_bwd_workspace_size(c["B"], c["Hq"], c["N"]), device=dev,
                         dtype=torch.uint8)
        w["fn"] = lambda: binding.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws)
        w["work"] = 2.5 * flops(**c)
        w["unit"], w["launches"], w["dtype"] = "TFLOP/s", 2, "bf16"
        w["seq_len"], w["batch"] = c["N"], c["B"]
        w["bound"], w["peak"] = "tensor", peaks["bf16_tflops"]
        w["peak_source"] = f"{peak_src} dense bf16 (burst)"
        w["e2e_in"] = [(x, t) for x, t in zip(host, (q, k, v))]
        w["e2e_out"] = [dq, dk, dv]
    elif name == "fp8":
        c = MAIN
        host = inputs.prefill_inputs_fp8(c["B"], c["Hq"], c["Hkv"], c["N"], c["N"], c["D"], seed)
        q, k, v = (x.to(dev) for x in host)
        o = torch.empty(q.shape, device=dev, dtype=torch.bfloat16)
        lse = torch.empty(c["B"], c["Hq"], c["N"], device=dev, dtype=torch.float32)
        ws = torch.empty(binding.attn_fwd_fp8_workspace_size(c["B"], c["Hkv"], c["N"], c["D"]), device=dev,
                         dtype=torch.uint8)
        w["fn"] = lambda: binding.attn_fwd_fp8(q, k, v, 1.0, 1.0, 1.0, o, lse, ws)
        w["make_fn"] = lambda ins, outs: (lambda: binding.attn_fwd_fp8(ins[0], ins[1], ins[2], 1.0, 1.0, 1.0,
                                                                       outs[0], outs[1], ws))
        w["work"] = flops(**c)
        w["unit"], w["launches"], w["dtype"] = "TFLOP/s", 2, "e4m3"
        w["seq_len"], w["batch"] = c["N"], c["B"]
        # half the FLOPs (Q K^T) at the fp8 rate (twice bf16: the nominal 4.5 / 2.25 PFLOP/s
        # ratio), half (P V) at the bf16 rate: 1 / (0.5 / 2P + 0.5 / P) = 4P / 3
        w["bound"], w["peak"] = "tensor", peaks["bf16_tflops"] * 4.0 / 3.0
        w["peak_source"] = f"4/3 x {peak_src} dense bf16 (burst): Q K^T at 2x (fp8), P V at 1x (bf16)"
        w["e2e_in"] = [(x, t) for x, t in zip(host, (q, k, v))]
        w["e2e_out"] = [o, lse]
    elif name == "varlen":
        c = VARLEN
        g = torch.Generator("cpu").manual_seed(seed + 11)
        lens = torch.randint(c["n_lo"], c["n_hi"] + 1, (c["B"],), generator=g).tolist()
        host = inputs.varlen_inputs(lens, lens, c["Hq"], c["Hkv"], c["D"], "bf16", seed)
        q, k, v, cq, ck = (x.to(dev) for x in host)
        o = torch.empty_like(q)
        lse = torch.empty(c["Hq"], q.shape[0], device=dev, dtype=torch.float32)
        w["fn"] = lambda: binding.attn_fwd_varlen(q, k, v, cq, ck, max(lens), o, lse, causal=True)
        w["work"] = sum(masked_flops(1, c["Hq"], n, n, c["D"], True, 0) for n in lens)
        w["unit"], w["launches"], w["dtype"] = "TFLOP/s", 1, "bf16"
        w["seq_len"], w["batch"] = max(lens), c["B"]
        w["bound"], w["peak"] = "tensor", peaks["bf16_tflops"]
        w["peak_source"] = f"{peak_src} dense bf16 (burst)"
        w["e2e_in"] = [(x, t) for x, t in zip(host, (q, k, v, cq, ck))]
        w["e2e_out"] = [o, lse]
    elif name in ("dense", "causal", "fp32", "window", "chunked", "d64", "fp16", "softcap"):
        c = {"dense": MAIN, "causal": CAUSAL, "fp32": FP32, "window": WINDOW, "chunked": CHUNKED,
             "d64": DENSE64, "fp16": MAIN, "softcap": MAIN}[name]
        Nq, Nk = c.get("Nq", c.get("N")), c.get("Nk", c.get("N"))
        dt = {"fp32": "fp32", "fp16": "fp16"}.get(name, "bf16")
        host = inputs.prefill_inputs(c["B"], c["Hq"], c["Hkv"], Nq, Nk, c["D"], dt, seed)
        q, k, v = (x.to(dev) for x in host)
        o = torch.empty_like(q)
        lse = torch.empty(c["B"], c["Hq"], Nq, device=dev, dtype=torch.float32)
        call = {"fp32": binding.attn_fwd_fp32, "fp16": binding.attn_fwd_fp16}.get(name, binding.attn_fwd)
        wnd = c.get("window", 0)
        w["fn"] = lambda: call(q, k, v, o, lse, causal=c["causal"], window=wnd)
        # the same step on other buffers (the pipelined end-to-end loop alternates two sets)
        w["make_fn"] = lambda ins, outs: (lambda: call(ins[0], ins[1], ins[2], outs[0], outs[1],
                                                       causal=c["causal"], window=wnd))
        if name == "softcap":
            sinks = torch.randn(c["Hq"], generator=torch.Generator("cpu").manual_seed(seed + 5)).float().to(dev)
            w["fn"] = lambda: binding.attn_fwd_softcap_sink(q, k, v, o, lse, causal=c["causal"], softcap=50.0,
                                                            sinks=sinks)
            w["make_fn"] = lambda ins, outs: (lambda: binding.attn_fwd_softcap_sink(
                ins[0], ins[1], ins[2], outs[0], outs[1], causal=c["causal"], softcap=50.0, sinks=sinks))
        w["work"] = masked_flops(c["B"], c["Hq"], Nq, Nk, c["D"], c["causal"], wnd) if "Nq" in c else flops(**c)
        w["unit"] = "TFLOP/s"
        w["launches"] = 1
        w["dtype"] = dt
        w["seq_len"], w["batch"] = Nk, c["B"]
        if name == "fp32":
            w["bound"] = "alu"
            w["peak"] = GB300_SMS * FP32_SIMT_FLOP_PER_CLK_SM * sm_max_mhz * 1e6 / 1e12
            w["peak_source"] = f"152 SMs x 256 FP32 FLOP/clk x {sm_max_mhz:.0f} MHz"
        else:
            w["bound"] = "tensor"
            w["peak"] = peaks["bf16_tflops"]
            w["peak_source"] = f"{peak_src} dense bf16 (burst)" + (" = fp16 dense rate" if name == "fp16" else "")
        w["e2e_in"] = [(x, t) for x, t in zip(host, (q, k, v))]
        w["e2e_out"] = [o, lse]
    else:
        base = {"decode_mqa": DECODE_MQA, "decode_d64": DECODE_D64}.get(name, DECODE)
        d = dict(base, B=decode_batch) if decode_batch else dict(base)
        w["desc"] = WORKLOAD_NAMES[name].replace(f"B={base['B']}", f"B={d['B']}")
        ws = torch.empty(binding.attn_decode_workspace_size(d["B"], d["Hq"], d["D"], d["nk_hi"], d["chunk"]),
                         device=dev, dtype=torch.uint8)
        o = torch.empty(d["B"], d["Hq"], d["D"], device=dev, dtype=torch.bfloat16)
        lse = torch.empty(d["B"], d["Hq"], device=dev)
        if name in ("decode", "decode_mqa", "decode_d64"):
            qh, kc, vc, sl = inputs.decode_inputs(d["B"], d["Hq"], d["Hkv"], d["D"], d["nk_lo"], d["nk_hi"],
                                                  seed=seed, device=dev)
            q, sl_d = qh.to(dev), sl.to(dev)
            w["fn"] = lambda: binding.attn_decode(q, kc, vc, sl_d, ws, o, lse, chunk=d["chunk"])
            w["split_fn"] = lambda: binding.attn_decode_splitkv(q, kc, vc, sl_d, ws, chunk=d["chunk"])
            extra_in = [(sl, sl_d), (None, kc), (None, vc)]
        elif name == "decode_fp8":
            qh, kc, vc, sl = inputs.decode_inputs(d["B"], d["Hq"], d["Hkv"], d["D"], d["nk_lo"], d["nk_hi"],
                                                  seed=seed, device=dev, kv_dtype="e4m3")
            q, sl_d = qh.to(dev), sl.to(dev)
            w["fn"] = lambda: binding.attn_decode_fp8(q, kc, vc, sl_d, 1.0, 1.0, ws, o, lse, chunk=d["chunk"])
            lib = binding.lib()

            def split_fp8():
                rc = lib.attn_decode_splitkv_fp8(
                    binding._ptr(q), binding._ptr(kc), binding._ptr(vc), 1.0, 1.0, binding._ptr(sl_d),
                    binding._ptr(ws), d["B"], d["Hq"], d["Hkv"], d["nk_hi"], d["D"], 1 / math.sqrt(d["D"]),
                    d["chunk"], binding._stream(None))
                assert rc == 0
            w["split_fn"] = split_fp8
            extra_in = [(sl, sl_d), (None, kc), (None, vc)]
        else:
            qh, kc, vc, bt, sl = inputs.paged_decode_inputs(d["B"], d["Hq"], d["Hkv"], d["D"], d["nk_lo"],
                                                            d["nk_hi"], 256, seed=seed, device=dev)
            q, sl_d, bt_d = qh.to(dev), sl.to(dev), bt.to(dev)
            w["fn"] = lambda: binding.attn_decode_paged(q, kc, vc, bt_d, sl_d, ws, o, lse, chunk=d["chunk"])
            lib = binding.lib()

            def split_paged():
                rc = lib.attn_decode_splitkv_paged(
                    binding._ptr(q), binding._ptr(kc), binding._ptr(vc), binding._ptr(bt_d), binding._ptr(sl_d),
                    binding._ptr(ws), d["B"], d["Hq"], d["Hkv"], kc.shape[0], 256, bt.shape[1], d["D"],
                    1 / math.sqrt(d["D"]), d["chunk"], binding._stream(None))
                assert rc == 0
            w["split_fn"] = split_paged
            extra_in = [(sl, sl_d), (bt, bt_d), (None, kc), (None, vc)]
        kv_elem = 1 if name == "decode_fp8" else 2
        kv_bytes = int(sl.sum()) * d["Hkv"] * d["D"] * kv_elem * 2
        w["kv_bytes"] = kv_bytes
        w["work"] = kv_bytes + q.numel() * 2 + o.numel() * 2 + lse.numel() * 4
        w["unit"] = "GB/s"
        w["launches"] = 2
        w["dtype"] = "e4m3" if name == "decode_fp8" else "bf16"
        w["seq_len"], w["batch"] = d["nk_hi"], d["B"]
        w["bound"] = "hbm"
        w["peak"] = peaks["hbm_gbs"]
        w["peak_source"] = f"{peak_src} copy bandwidth"
        w["e2e_in"] = [(qh, q)] + extra_in
        w["e2e_out"] = [o, lse]
    return w


def make_fp32_point(dev, seed, B, H, N, D, sm_max_mhz):
    """One fp32 configuration (dense, non-causal, Hq = Hkv = H) resident on ``dev``."""
    import torch
    from softmax_attention_attn_gb300 import binding, inputs
    q, k, v = (x.to(dev) for x in inputs.prefill_inputs(B, H, H, N, N, D, "fp32", seed))
    o = torch.empty_like(q)
    lse = torch.empty(B, H, N, device=dev, dtype=torch.float32)
    return {"desc": f"fp32 dense prefill B={B} H={H} N={N} D={D}",
            "fn": lambda: binding.attn_fwd_fp32(q, k, v, o, lse), "work": flops(B, H, N, D, False),
            "unit": "TFLOP/s", "peak": GB300_SMS * FP32_SIMT_FLOP_PER_CLK_SM * sm_max_mhz * 1e6 / 1e12,
            "peak_source": f"152 SMs x 256 FP32 FLOP/clk x {sm_max_mhz:.0f} MHz"}


def max_over_ranks_of(x, world, device):
    """Maximum of a per-rank float over all ranks (the step time of the slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rate(w, ms):
    scale = 1e12 if w["unit"] == "TFLOP/s" else 1e9
    return w["work"] / (ms * 1e-3) / scale


def build_line(args, world, main, main_work_desc, value, ms_step, ms_median, ms_min, achieved, traffic, e2e,
               clocks, workloads, cpu, launch_floor, wall_s):
    """The short stdout JSON line and the full details record of a GB300-arm run."""
    details = {
        "main": {"workload": main_work_desc, "ms_per_step": ms_step, "ms_per_step_median": ms_median,
                 "ms_per_step_min": ms_min, "peak_source": main["peak_source"]},
        "wall_s_timed_region": wall_s, "launch_floor": launch_floor, "e2e": e2e, "workloads": workloads,
        "cpu_baseline": cpu, "clocks": clocks,
    }
    line = {
        "metric": METRIC, "value": sig(value), "unit": main["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sig(ms_step), "ms_med": sig(ms_median), "ms_min": sig(ms_min),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": main["dtype"],
        "data": "synthetic", "gpu_launches": args.steps * main["launches"],
        "config": dict(MAIN_CONFIG, global_batch=world * main["batch"],
                       parallelism="replicas" if world > 1 else "single")
        if main["name"] == "dense" else {"workload": main_work_desc, "global_batch": world * main["batch"],
                                         "seq_len": main["seq_len"],
                                         "parallelism": "replicas" if world > 1 else "single"},
        "timing": "CUDA events per step; L2 flushed (256 MiB write) before every step",
        "roofline": {"bound": main["bound"], "achieved": sig(achieved), "peak": main["peak"], "unit": main["unit"],
                     "frac": sig(achieved / main["peak"]), "traffic": traffic,
                     "peak_source": main["peak_source"]},
    }
    if "decode" in workloads:
        d = workloads["decode"]
        line["decode"] = {"GB/s": sig(d["value"]), "frac": sig(d["frac"]), "split_GB/s": sig(d["splitkv_kernel_gbs"]),
                          "split_frac": sig(d["splitkv_frac"]), "peak_GB/s": d["peak"],
                          "workload": "bf16 split-KV decode B=64 Hq=32 Hkv=8 D=128 Nk~U[512,32768] chunk 512"}
    if "causal" in workloads:
        c = workloads["causal"]
        line["causal"] = {"TFLOP/s": sig(c["value"]), "frac": sig(c["frac"]),
                          "workload": "bf16 causal GQA B=4 Hq=32 Hkv=8 N=4096 D=128"}
    if e2e is not None:
        line["e2e"] = {"value": sig(e2e["value"]), "unit": e2e["unit"], "h2d_bytes_per_step": e2e["h2d_bytes_per_step"],
                       "d2h_bytes_per_step": e2e["d2h_bytes_per_step"], "ms_per_step": sig(e2e["ms_per_step"]),
                       "pipelined": e2e["pipelined"]}
        if "serial_value" in e2e:
            line["e2e"]["serial_value"] = sig(e2e["serial_value"])
    line["clocks"] = None if clocks is None else {k: (sig(v) if isinstance(v, float) else v) for k, v in clocks.items()}
    line["cpu_baseline"] = cpu
    line["w"] = {SHORT.get(n, n): [sig(e["value"]), sig(e["frac"])] for n, e in workloads.items()
                 if n not in ("decode", "causal") and not n.startswith("fp32_B")}
    for n in ("paged", "decode_fp8", "decode_mqa", "decode_d64"):
        if n in workloads:
            line["w"][SHORT[n]].append(sig(workloads[n]["splitkv_frac"]))
    fp32 = {n[5:].replace("_", ""): [sig(e["value"]), sig(e["frac"])] for n, e in workloads.items()
            if n.startswith("fp32_B")}
    if fp32:
        line["fp32"] = fp32
    line["keys"] = "w/fp32: [value, frac of roofline(, split-kernel frac)]; units: TFLOP/s, decode GB/s"
    return details, line


def run_gb300(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from softmax_attention_attn_gb300 import binding, build

    build.build()
    binding.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()
    sm_max = float(peaks.get("sm_max_mhz", 2070.0))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def max_over_ranks(x):
        return max_over_ranks_of(x, world, dev)

    def barrier():
        if world > 1:
            dist.barrier()

    # ---------------- the timed workload
    w = make_workload(args.workload, dev, rank, peaks, peak_src, sm_max, args.decode_batch)
    for _ in range(args.warmup):
        flush.zero_()
        w["fn"]()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        ms = time_steps(torch, w["fn"], args.steps, 0, flush, stream)
        torch.cuda.synchronize()
        barrier()
        wall1 = time.perf_counter()
    clocks = clk.summary()
    ms_step = max_over_ranks(sum(ms) / len(ms))
    ms_median = max_over_ranks(statistics.median(ms))
    ms_min = max_over_ranks(min(ms))
    value = world * rate(w, ms_step)
    if w["name"] in DECODE_NAMES:   # roofline of the dominant kernel: the split-KV partial step
        ms_k = max_over_ranks(statistics.mean(time_steps(torch, w["split_fn"], min(args.steps, 50), 3, flush, stream)))
        achieved = w["kv_bytes"] / (ms_k * 1e-3) / 1e9
        traffic = None
    else:
        achieved = rate(w, ms_step)
        traffic = kernel_traffic() if w["name"] == "dense" else None
    rc = binding.get_device_error()
    if rc != 0:
        raise RuntimeError(f"device error word {rc} after the timed region")

    # ---------------- launch floor: the smallest valid forward call (one 128-query tile), timed
    # back to back, against which the timed steps above are long enough to ignore launch costs
    lq = torch.randn(1, 1, 128, 128, device=dev).to(torch.bfloat16)
    lo = torch.empty_like(lq)
    ll = torch.empty(1, 1, 128, device=dev)
    for _ in range(10):
        binding.attn_fwd(lq, lq, lq, lo, ll)
    torch.cuda.synchronize()
    n_floor = 200
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    ev0.record(stream)
    for _ in range(n_floor):
        binding.attn_fwd(lq, lq, lq, lo, ll)
    ev1.record(stream)
    torch.cuda.synchronize()
    launch_floor = {"us_per_call_device": ev0.elapsed_time(ev1) * 1e3 / n_floor,
                    "us_per_call_host": (time.perf_counter() - t0) * 1e6 / n_floor,
                    "call": "attn_fwd B=1 H=1 N=128 D=128 bf16, 200 calls back to back"}
    del lq, lo, ll

    # ---------------- end to end: pinned host inputs copied in, results copied out, every step
    e2e = None
    if not args.no_e2e:
        pins = [(x.pin_memory() if x is not None else torch.empty(t.shape, dtype=t.dtype).pin_memory(), t)
                for x, t in w["e2e_in"]]
        outs = [(torch.empty(t.shape, dtype=t.dtype).pin_memory(), t) for t in w["e2e_out"]]
        if w["name"] in DECODE_NAMES:   # the host copy of the caches is the device draw
            for (x, t), (hp, _) in zip(w["e2e_in"], pins):
                if x is None:
                    hp.copy_(t)
        e2e_steps = max(5, min(args.steps, 100 if w["name"] not in DECODE_NAMES else 10))

        def e2e_step():
            for hp, t in pins:
                t.copy_(hp, non_blocking=True)
            w["fn"]()
            for hp, t in outs:
                hp.copy_(t, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier()
        t0 = time.perf_counter()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(max(ev0.elapsed_time(ev1), (time.perf_counter() - t0) * 1e3) / e2e_steps)
        e2e = {"value": world * rate(w, e2e_ms), "unit": w["unit"],
               "h2d_bytes_per_step": sum(hp.numel() * hp.element_size() for hp, _ in pins),
               "d2h_bytes_per_step": sum(hp.numel() * hp.element_size() for hp, _ in outs),
               "ms_per_step": e2e_ms, "pipelined": False}
        if "make_fn" in w:
            # Pipelined: the same steps (each copies its inputs in from pinned host memory and
            # its results out to pinned host memory) with step i+1's copy in and step i-1's
            # copy out running on their own streams while step i computes.  Two sets of device
            # buffers alternate so that no copy touches a buffer a kernel still uses.
            sets_in = [[t for _, t in pins], [torch.empty_like(t) for _, t in pins]]
            sets_out = [[t for _, t in outs], [torch.empty_like(t) for _, t in outs]]
            host_out = [[hp for hp, _ in outs], [torch.empty(t.shape, dtype=t.dtype).pin_memory() for _, t in outs]]
            fns = [w["make_fn"](sets_in[j], sets_out[j]) for j in range(2)]
            s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
            ev_in = [torch.cuda.Event() for _ in range(2)]
            ev_comp = [torch.cuda.Event() for _ in range(2)]
            ev_out = [torch.cuda.Event() for _ in range(2)]

            def pipelined(n):
                s_in.wait_stream(stream)
                s_out.wait_stream(stream)
                for i in range(n):
                    j = i % 2
                    with torch.cuda.stream(s_in):
                        if i >= 2:
                            s_in.wait_event(ev_comp[j])      # step i-2's kernel has read set j
                        for (hp, _), t in zip(pins, sets_in[j]):
                            t.copy_(hp, non_blocking=True)
                        ev_in[j].record(s_in)
                    stream.wait_event(ev_in[j])
                    if i >= 2:
                        stream.wait_event(ev_out[j])         # step i-2's results are out
                    fns[j]()
                    ev_comp[j].record(stream)
                    with torch.cuda.stream(s_out):
                        s_out.wait_event(ev_comp[j])
                        for hp, t in zip(host_out[j], sets_out[j]):
                            hp.copy_(t, non_blocking=True)
                        ev_out[j].record(s_out)
                stream.wait_stream(s_out)

            pipelined(3)
            torch.cuda.synchronize()
            barrier()
            t0 = time.perf_counter()
            ev0.record(stream)
            pipelined(e2e_steps)
            ev1.record(stream)
            torch.cuda.synchronize()
            barrier()
            p_ms = max_over_ranks(max(ev0.elapsed_time(ev1), (time.perf_counter() - t0) * 1e3) / e2e_steps)
            e2e.update({"serial_value": e2e["value"], "serial_ms_per_step": e2e_ms,
                        "value": world * rate(w, p_ms), "ms_per_step": p_ms, "pipelined": True,
                        "pipelining": "step i+1's copy in and step i-1's copy out overlap step i "
                                      "(two device buffer sets, three streams)"})
            del sets_in, sets_out, host_out, fns
        del pins, outs
    main_work_desc = w["desc"]
    main = {k: w[k] for k in ("name", "unit", "bound", "peak", "peak_source", "dtype", "seq_len", "batch", "launches")}
    del w
    torch.cuda.empty_cache()

    # ---------------- the other workloads, shorter loops
    workloads = {}
    if not args.no_extras:
        xs = max(5, min(args.steps // 10, 50))
        for name in ("dense", "causal", "decode", "paged", "decode_fp8", "decode_mqa", "decode_d64", "window",
                     "chunked", "d64", "fp16", "varlen", "softcap", "bwd", "bwd_d64", "fp8"):
            if name == args.workload:
                continue
            x = make_workload(name, dev, rank, peaks, peak_src, sm_max, args.decode_batch)
            mx = max_over_ranks(statistics.mean(time_steps(torch, x["fn"], xs, 3, flush, stream)))
            r = rate(x, mx)
            entry = {"workload": x["desc"], "value": world * r, "unit": x["unit"], "ms_per_step": mx,
                     "bound": x["bound"], "frac": r / x["peak"], "peak": x["peak"], "peak_source": x["peak_source"]}
            if name in DECODE_NAMES:
                mk = max_over_ranks(statistics.mean(time_steps(torch, x["split_fn"], xs, 3, flush, stream)))
                entry["splitkv_kernel_ms"] = mk
                entry["splitkv_kernel_gbs"] = x["kv_bytes"] / (mk * 1e-3) / 1e9
                entry["splitkv_frac"] = entry["splitkv_kernel_gbs"] / x["peak"]
            workloads[name] = entry
            del x
            torch.cuda.empty_cache()
        # the fp32 configurations: B=2 H=4 N=64 D=32 and the B=2 H=8 sweep over N x D
        for (B, H, N, D) in FP32_POINTS:
            x = make_fp32_point(dev, rank, B, H, N, D, sm_max)
            mx = max_over_ranks(statistics.mean(time_steps(torch, x["fn"], xs, 3, flush, stream)))
            r = rate(x, mx)
            workloads[f"fp32_B{B}_H{H}_N{N}_D{D}"] = {
                "workload": x["desc"], "value": world * r, "unit": "TFLOP/s", "ms_per_step": mx, "bound": "alu",
                "frac": r / x["peak"], "peak": x["peak"], "peak_source": x["peak_source"]}
            del x
        torch.cuda.empty_cache()
        if binding.get_device_error() != 0:
            raise RuntimeError("device error word set by a secondary workload")

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        cpu = cpu_baseline(args.cpu_seconds)

    details, line = build_line(args, world, main, main_work_desc, value, ms_step, ms_median, ms_min,
                               achieved, traffic, e2e, clocks, workloads, cpu, launch_floor, wall1 - wall0)
    if args.details:
        with open(args.details, "w") as f:
            json.dump({"line": line, "details": details}, f, indent=1)
    if rank == 0:
        print(json.dumps(line, separators=(",", ":")), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.cpu_worker > 0:      # child process of cpu_baseline(): the oracle on N threads
        cpu_worker_main(args.cpu_worker, args.cpu_seconds)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
