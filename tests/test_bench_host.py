"""Host-side checks of bench.py (CPU only): the multi-rank aggregation over
gloo with two ranks, the FLOP convention, and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 1.5 + rank                       # rank 1 is the slowest
        out[rank] = bench.max_over_ranks_of(local_ms, world, torch.device("cpu"))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_single_rank_max_is_identity():
    assert bench.max_over_ranks_of(3.25, 1, None) == 3.25


def test_flop_convention():
    # 4*B*Hq*Nq*Nk*D, halved for causal
    assert bench.flops(**bench.MAIN) == 4 * 1 * 32 * 8192 * 8192 * 128
    assert bench.flops(**bench.CAUSAL) == 4 * 4 * 32 * 4096 * 4096 * 128 / 2


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["steps"] == 3 and line["warmup"] == 3 and line["higher_is_better"] is True


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_below_three_is_rejected():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "2"], capture_output=True, text=True, timeout=600)
    assert r.returncode != 0


def test_visible_pairs_matches_enumeration():
    for Nq, Nk, causal, window in [(5, 5, True, 0), (3, 7, True, 0), (7, 3, True, 0), (6, 6, True, 2),
                                   (5, 4, False, 3), (4, 4, False, 0)]:
        brute = sum(1 for i in range(Nq) for j in range(Nk)
                    if (not causal or j <= i + Nk - Nq) and (window <= 0 or j > i + Nk - Nq - window))
        assert bench.visible_pairs(Nq, Nk, causal, window) == brute


def test_kernel_traffic_reads_summary_only_for_matching_source(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu summary only while the kernel source
    it was captured from is unchanged (the field name itself contains a colon)."""
    import hashlib
    src = tmp_path / "kernel.cu"
    src.write_text("__global__ void k() {}\n")
    h = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    summary = tmp_path / "summary.md"
    summary.write_text(f"# k\n\n- kernel source sha256[:16]: `{h}`\n- dram bytes per launch: `1234`\n")
    monkeypatch.setattr(bench, "KERNEL_SRC", str(src))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(summary))
    assert bench.kernel_traffic() == 1234.0
    src.write_text("__global__ void k() { }\n")
    assert bench.kernel_traffic() is None



def _fake_run():
    """Workload records of a full run with plausible magnitudes (no GPU involved)."""
    wl = {}
    for name in ("causal", "decode", "paged", "decode_fp8", "decode_mqa", "decode_d64", "window", "chunked",
                 "d64", "fp16", "varlen", "softcap", "bwd", "bwd_d64", "fp8"):
        dec = name in bench.DECODE_NAMES
        e = {"workload": bench.WORKLOAD_NAMES[name], "value": 6543.21987 if dec else 1234.56789,
             "unit": "GB/s" if dec else "TFLOP/s", "ms_per_step": 0.61234567, "bound": "hbm" if dec else "tensor",
             "frac": 0.9634567891, "peak": 6791.0 if dec else 1898.5, "peak_source": "measured"}
        if dec:
            e.update(splitkv_kernel_ms=0.6012345, splitkv_kernel_gbs=6612.345678, splitkv_frac=0.97345678)
        wl[name] = e
    for (B, H, N, D) in bench.FP32_POINTS:
        wl[f"fp32_B{B}_H{H}_N{N}_D{D}"] = {"workload": "x", "value": 38.123456789, "unit": "TFLOP/s",
                                           "ms_per_step": 3.6123, "bound": "alu", "frac": 0.4712345678,
                                           "peak": 80.54784, "peak_source": "derived"}
    main = {"name": "dense", "unit": "TFLOP/s", "bound": "tensor", "peak": 1898.5,
            "peak_source": "measured dense bf16 (burst)", "dtype": "bf16", "seq_len": 8192, "batch": 1,
            "launches": 1}
    e2e = {"value": 1010.88529, "unit": "TFLOP/s", "h2d_bytes_per_step": 201326592, "d2h_bytes_per_step": 68157440,
           "ms_per_step": 1.08767200006, "pipelined": True, "serial_value": 562.521911, "serial_ms_per_step": 1.95}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "power_w_max": 1171.51, "samples": 33,
              "reasons": ["sw_power_cap"]}
    cpu = {"value": 0.7012, "unit": "TFLOP/s", "cores": 16, "kind": "oracle", "value_1_core": 0.04512,
           "sample": "fp64 oracle, whole heads of the dense workload: 32 heads in 10.3 s on 16 threads, "
                     "3 in 10.9 s on 1"}
    args = type("A", (), {"steps": 1000, "warmup": 10})()
    return bench.build_line(args, 1, main, bench.WORKLOAD_NAMES["dense"], 1743.68449, 0.63056799, 0.6301, 0.6289,
                            1743.68449, 245076224.0, e2e, clocks, wl, cpu, {"us": 5.0}, 0.63)


def test_bench_line_fits_the_recorded_tail():
    """The stdout line carries the decode and causal figures at top level and stays short
    enough (< 2800 characters) that a 3000-character tail of the output holds all of it."""
    details, line = _fake_run()
    text = json.dumps(line, separators=(",", ":"))
    assert len(text) < 2800, len(text)
    back = json.loads(text)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches",
                "cpu_baseline", "clocks", "decode", "causal", "w", "fp32"):
        assert key in back, key
    assert back["decode"]["GB/s"] == 6543.0 and back["decode"]["split_frac"] == 0.9735
    assert back["causal"]["frac"] == 0.9635
    assert len(back["fp32"]) == 13
    assert back["config"] == dict(bench.MAIN_CONFIG)
    assert back["cpu_baseline"]["cores"] == 16 and back["cpu_baseline"]["value_1_core"] > 0
    assert details["workloads"]["decode"]["splitkv_kernel_gbs"] == 6612.345678


def test_sig_rounds_to_four_digits():
    assert bench.sig(1743.68449) == 1744.0 and bench.sig(0.0451234) == 0.04512
    assert bench.sig(None) is None and bench.sig(0.0) == 0.0


def test_cpu_worker_reports_heads_and_seconds():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-worker", "2", "--cpu-seconds",
                        "0.01"], capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OPENBLAS_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["threads"] == 2 and out["heads"] >= 1 and out["seconds"] > 0
