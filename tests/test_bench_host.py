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

