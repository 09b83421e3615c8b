#!/usr/bin/env python
"""Benchmark of the fused attention forward on GB300.

One step = one ``attn_fwd`` call (the whole bf16 prefill path: Q/K/V tile
loads, S = Q K^T, mask, online softmax, O correction, O += P V, epilogue) over
the dense workload B=1 H=32 N=8192 D=128, inputs resident in HBM, L2 flushed
before every step (a 256 MiB write), each step timed with CUDA events on the
launching stream.  ``value`` is attention-forward TFLOP/s counted as
4*B*Hq*Nq*Nk*D (halved for causal).  The same JSON line also carries:

* ``e2e``: the same metric through the C ABI with the inputs copied from pinned
  host memory and O / LSE copied back inside every timed step;
* ``roofline``: achieved TFLOP/s of the kernel against the measured dense bf16
  peak, plus the DRAM traffic of one ncu capture of the same kernel;
* ``workloads``: the causal GQA prefill (B=4 Hq=32 Hkv=8 N=4096), the split-KV
  decode (B=64 Hq=32 Hkv=8, Nk_b ~ U[512, 32768], chunk 512, HBM GB/s against
  the measured copy bandwidth) and the fp32 prefill (B=2 H=8 N=4096 D=128);
* ``cpu_baseline``: the fp64 CPU oracle timed on this host on a bounded
  sample of the same workload;
* ``clocks``: SM clocks and throttle reasons sampled during the timed region.

``--impl reference`` times the CPU oracle instead (rank 0 only).  Under
torchrun every rank runs its own replica of the workload (weak scaling, no
collective on the data path); timing is the maximum over ranks.
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
FP32 = dict(B=2, Hq=8, Hkv=8, N=4096, D=128, causal=False)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP32_SIMT_FLOP_PER_CLK_SM = 256.0   # 128 FP32 lanes x 2 (fused multiply-add)
GB300_SMS = 152
FLUSH_BYTES = 256 << 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_bf16_dense_B1_H32_N8192.md")
KERNEL_SRC = os.path.join(ROOT, "softmax_attention_attn_gb300", "csrc", "attn_fwd_bf16.cu")


def flops(B, Hq, N, D, causal, **_):
    f = 4.0 * B * Hq * N * N * D
    return f / 2 if causal else f


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-extras", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-oracle sample budget")
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
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
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


def cpu_oracle_sample(budget_s, seed=0):
    """fp64 oracle on whole heads of the dense workload until ``budget_s`` elapses."""
    import numpy as np  # noqa: F401
    import oracle
    from softmax_attention_attn_gb300 import inputs
    q, k, v = inputs.prefill_inputs(1, MAIN["Hq"], MAIN["Hkv"], MAIN["N"], MAIN["N"], MAIN["D"], "bf16", seed)
    scale = 1 / math.sqrt(MAIN["D"])
    heads, t0 = 0, time.perf_counter()
    while heads < MAIN["Hq"] and (time.perf_counter() - t0) < budget_s:
        h = heads
        oracle.attention_forward(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], scale)
        heads += 1
    dt = time.perf_counter() - t0
    f = flops(1, heads, MAIN["N"], MAIN["D"], False)
    return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle",
            "sample": f"{heads} of 32 heads of the dense workload (B=1 N=8192 D=128), fp64 numpy, "
                      f"{dt:.1f} s; matmul on numpy's BLAS threads, the rest single-threaded"}


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from softmax_attention_attn_gb300 import inputs
    q, k, v = inputs.prefill_inputs(1, MAIN["Hq"], MAIN["Hkv"], MAIN["N"], MAIN["N"], MAIN["D"], "bf16", 0)
    scale = 1 / math.sqrt(MAIN["D"])
    rows_per_step = 64
    import numpy as np
    rng = np.random.default_rng(0)

    def step(i):
        h = int(rng.integers(MAIN["Hq"]))
        i0 = int(rng.integers(0, MAIN["N"] - rows_per_step))
        rows = [(0, h, i) for i in range(i0, i0 + rows_per_step)]
        oracle.attention_rows(q, k, v, scale, rows)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    f = 4.0 * rows_per_step * MAIN["N"] * MAIN["D"] * args.steps
    value = f / dt / 1e12
    sample = (f"{rows_per_step} query rows of one head of the dense workload (B=1 H=32 N=8192 D=128) "
              "per step, fp64 numpy oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "bf16 dense prefill B=1 H=32 N=8192 D=128 (oracle on sampled rows)",
                       "global_batch": 1, "seq_len": MAIN["N"], "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GB300 arm
def run_gb300(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from softmax_attention_attn_gb300 import binding, build, inputs

    build.build()
    binding.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def max_over_ranks(x):
        if world == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    def barrier():
        if world > 1:
            dist.barrier()

    # ---------------- main workload: dense bf16 prefill
    c = MAIN
    qh, kh, vh = inputs.prefill_inputs(c["B"], c["Hq"], c["Hkv"], c["N"], c["N"], c["D"], "bf16", seed=rank)
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(c["B"], c["Hq"], c["N"], device=dev, dtype=torch.float32)
    fwd = lambda: binding.attn_fwd(q, k, v, o, lse, causal=False)  # noqa: E731
    for _ in range(args.warmup):
        flush.zero_()
        fwd()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        ms = time_steps(torch, fwd, args.steps, 0, flush, stream)
        torch.cuda.synchronize()
        barrier()
        wall1 = time.perf_counter()
    clocks = clk.summary()
    ms_step = max_over_ranks(sum(ms) / len(ms))
    f_main = flops(**c)
    value = world * f_main / (ms_step * 1e-3) / 1e12
    achieved = f_main / (ms_step * 1e-3) / 1e12
    rc = binding.get_device_error()
    if rc != 0:
        raise RuntimeError(f"device error word {rc} after the timed region")

    # ---------------- end to end: pinned host buffers, copies inside every step
    qp, kp, vp = (x.pin_memory() for x in (qh, kh, vh))
    op = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lp = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e2e_steps = max(5, min(args.steps, 100))

    def e2e_step():
        q.copy_(qp, non_blocking=True)
        k.copy_(kp, non_blocking=True)
        v.copy_(vp, non_blocking=True)
        fwd()
        op.copy_(o, non_blocking=True)
        lp.copy_(lse, non_blocking=True)

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
    h2d = sum(x.numel() * x.element_size() for x in (qp, kp, vp))
    d2h = op.numel() * op.element_size() + lp.numel() * lp.element_size()
    del qp, kp, vp, op, lp

    # ---------------- secondary workloads
    workloads = {}
    if not args.no_extras:
        xs = max(5, min(args.steps // 10, 50))
        # causal GQA prefill
        c4 = CAUSAL
        q4, k4, v4 = (x.to(dev) for x in inputs.prefill_inputs(c4["B"], c4["Hq"], c4["Hkv"], c4["N"], c4["N"],
                                                               c4["D"], "bf16", seed=rank))
        o4 = torch.empty_like(q4)
        l4 = torch.empty(c4["B"], c4["Hq"], c4["N"], device=dev)
        t4 = time_steps(torch, lambda: binding.attn_fwd(q4, k4, v4, o4, l4, causal=True), xs, 3, flush, stream)
        m4 = max_over_ranks(statistics.mean(t4))
        a4 = flops(**c4) / (m4 * 1e-3) / 1e12
        workloads["bf16_causal_gqa_B4_Hq32_Hkv8_N4096"] = {
            "value": world * a4, "unit": "TFLOP/s", "ms_per_step": m4,
            "frac_of_bf16_peak": a4 / peaks["bf16_tflops"], "peak": f"{peaks['bf16_tflops']} ({peak_src})"}
        del q4, k4, v4, o4, l4
        # split-KV decode
        d = DECODE
        qd, kc, vc, sl = inputs.decode_inputs(d["B"], d["Hq"], d["Hkv"], d["D"], d["nk_lo"], d["nk_hi"],
                                              seed=rank, device=dev)
        qd, sl_d = qd.to(dev), sl.to(dev)
        ws = torch.empty(binding.attn_decode_workspace_size(d["B"], d["Hq"], d["D"], d["nk_hi"], d["chunk"]),
                         device=dev, dtype=torch.uint8)
        od = torch.empty(d["B"], d["Hq"], d["D"], device=dev, dtype=torch.bfloat16)
        ld = torch.empty(d["B"], d["Hq"], device=dev)
        kv_bytes = int(sl.sum()) * d["Hkv"] * d["D"] * 2 * 2
        alg_bytes = kv_bytes + qd.numel() * 2 + od.numel() * 2 + ld.numel() * 4
        ts = time_steps(torch, lambda: binding.attn_decode_splitkv(qd, kc, vc, sl_d, ws, chunk=d["chunk"]),
                        xs, 3, flush, stream)
        tt = time_steps(torch, lambda: binding.attn_decode(qd, kc, vc, sl_d, ws, od, ld, chunk=d["chunk"]),
                        xs, 3, flush, stream)
        ms_s, ms_t = max_over_ranks(statistics.mean(ts)), max_over_ranks(statistics.mean(tt))
        workloads["bf16_splitkv_decode_B64_Hq32_Hkv8_chunk512"] = {
            "value": world * alg_bytes / (ms_t * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_t,
            "frac_of_hbm_peak": alg_bytes / (ms_t * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "splitkv_kernel_gbs": kv_bytes / (ms_s * 1e-3) / 1e9, "splitkv_kernel_ms": ms_s,
            "splitkv_frac_of_hbm_peak": kv_bytes / (ms_s * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "algorithmic_bytes": alg_bytes, "peak": f"{peaks['hbm_gbs']} GB/s ({peak_src})"}
        del qd, kc, vc, ws, od, ld
        torch.cuda.empty_cache()
        # fp32 prefill
        c2 = FP32
        q2, k2, v2 = (x.to(dev) for x in inputs.prefill_inputs(c2["B"], c2["Hq"], c2["Hkv"], c2["N"], c2["N"],
                                                               c2["D"], "fp32", seed=rank))
        t2 = time_steps(torch, lambda: binding.attn_fwd_fp32(q2, k2, v2), xs, 3, flush, stream)
        m2 = max_over_ranks(statistics.mean(t2))
        a2 = flops(**c2) / (m2 * 1e-3) / 1e12
        sm_mhz = (clocks or {}).get("sm_max_mhz") or peaks.get("sm_max_mhz", 2070.0)
        fp32_peak = GB300_SMS * FP32_SIMT_FLOP_PER_CLK_SM * sm_mhz * 1e6 / 1e12
        workloads["fp32_B2_H8_N4096_D128"] = {
            "value": world * a2, "unit": "TFLOP/s", "ms_per_step": m2, "frac_of_fp32_simt_peak": a2 / fp32_peak,
            "peak": f"{fp32_peak:.1f} TFLOP/s (152 SMs x 256 FLOP/clk x max SM clock)"}
        del q2, k2, v2
        if binding.get_device_error() != 0:
            raise RuntimeError("device error word set by a secondary workload")

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        cpu = cpu_oracle_sample(args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "bf16 dense prefill B=1 H=32 N=8192 D=128 (non-causal)", "global_batch": world,
                   "seq_len": c["N"], "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed (256 MiB write) before every step", "timing": "CUDA events per step"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": kernel_traffic(),
                     "peak_source": f"{peak_src} dense bf16 (burst)"},
        "e2e": {"value": world * f_main / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps,
        "wall_s_timed_region": wall1 - wall0,
        "clocks": clocks,
        "workloads": workloads,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
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
