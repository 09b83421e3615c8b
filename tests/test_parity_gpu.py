"""GPU parity: the CUDA kernels (through the C ABI) against the fp64 oracle.

Tolerances (fixed by the attention-forward target):
  * fp32 inputs: max-abs error <= 1e-4 on O and on LSE;
  * bf16 inputs (fp32 accumulation): max-abs error <= 2e-2 on O and
    |dLSE| <= 1e-2 * max(1, |LSE|) on LSE.
Rows that see no key must give O = 0 and LSE = -inf on both sides.
Small and ragged shapes are compared element by element; the full benchmark
workloads are compared on sampled rows that the oracle computes one by one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from softmax_attention_attn_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

FP32_TOL = 1e-4
BF16_O_TOL = 2e-2
BF16_LSE_REL = 1e-2


@pytest.fixture(scope="module")
def dev(cuda_lib):
    return torch.device("cuda:0")


def check(o_gpu, lse_gpu, O, L, o_tol, lse_tol, lse_relative):
    o = o_gpu.float().cpu().numpy().reshape(O.shape)
    l = lse_gpu.float().cpu().numpy().reshape(L.shape)
    assert np.isfinite(o).all(), "non-finite output"
    err_o = float(np.abs(o - O).max()) if O.size else 0.0
    fin = np.isfinite(L)
    fin_ok = np.array_equal(np.isfinite(l), fin) and bool(np.all(l[~fin] == -np.inf))
    err_l = 0.0
    if fin.any() and fin_ok:
        d = np.abs(l[fin] - L[fin])
        if lse_relative:
            d = d / np.maximum(1.0, np.abs(L[fin]))
        err_l = float(d.max())
    msg = f"O max-abs err {err_o:.3e} (tol {o_tol}), LSE err {err_l:.3e} (tol {lse_tol}), finiteness ok {fin_ok}"
    assert fin_ok and err_o <= o_tol and err_l <= lse_tol, msg
    return err_o


def sample_rows(B, H, N, n, seed, tile=128):
    rng = np.random.default_rng(seed)
    rows = {(int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(N))) for _ in range(n)}
    for i in (0, 1, tile - 1, tile, 2 * tile - 1, 2 * tile, N - 2, N - 1):
        if 0 <= i < N:
            rows.add((int(rng.integers(B)), int(rng.integers(H)), i))
    return sorted(rows)


# ---------------------------------------------------------------- fp32 path
def run_fp32(dev, B, Hq, Hkv, Nq, Nk, D, causal=False, window=0, seed=0):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, D, "fp32", seed)
    o, lse = binding.attn_fwd_fp32(q.to(dev), k.to(dev), v.to(dev), causal=causal, window=window)
    return q, k, v, o, lse


def test_fp32_small_config(dev):
    """fp32 dense non-causal, B=2 H=4 N=64 D=32."""
    q, k, v, o, lse = run_fp32(dev, 2, 4, 4, 64, 64, 32)
    O, L = oracle.attention_forward(q, k, v, 1 / math.sqrt(32))
    check(o, lse, O, L, FP32_TOL, FP32_TOL, False)


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("N", [64, 256, 1024, 4096])
def test_fp32_sweep(dev, N, D):
    """fp32 dense non-causal sweep, B=2 H=8."""
    q, k, v, o, lse = run_fp32(dev, 2, 8, 8, N, N, D, seed=N + D)
    if N <= 1024:
        O, L = oracle.attention_forward(q, k, v, 1 / math.sqrt(D))
        check(o, lse, O, L, FP32_TOL, FP32_TOL, False)
    else:
        rows = sample_rows(2, 8, N, 48, seed=N, tile=64)
        O, L = oracle.attention_rows(q, k, v, 1 / math.sqrt(D), rows)
        idx = tuple(np.array(rows).T)
        check(o.cpu()[idx], lse.cpu()[idx], O, L, FP32_TOL, FP32_TOL, False)


FP32_EDGE = [  # (B, Hq, Hkv, Nq, Nk, D, causal, window)
    (1, 2, 2, 100, 77, 64, False, 0),
    (1, 4, 2, 130, 130, 32, True, 0),
    (2, 2, 1, 65, 200, 128, True, 0),     # Nq < Nk: bottom-right causal
    (1, 2, 1, 200, 65, 64, True, 0),      # Nq > Nk: fully masked rows
    (1, 2, 2, 150, 150, 32, True, 40),    # causal + window
    (1, 2, 2, 150, 150, 64, False, 33),   # window only
    (1, 2, 2, 1, 1, 32, False, 0),
    (1, 1, 1, 3, 1000, 128, False, 0),
]


@pytest.mark.parametrize("case", FP32_EDGE, ids=str)
def test_fp32_edge_cases(dev, case):
    B, Hq, Hkv, Nq, Nk, D, causal, window = case
    q, k, v, o, lse = run_fp32(dev, B, Hq, Hkv, Nq, Nk, D, causal, window, seed=7)
    O, L = oracle.attention_forward(q, k, v, 1 / math.sqrt(D), causal, window)
    check(o, lse, O, L, FP32_TOL, FP32_TOL, False)


# ---------------------------------------------------------------- bf16 path
def run_bf16(dev, B, Hq, Hkv, Nq, Nk, causal=False, window=0, seed=0, D=128):
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, D, "bf16", seed)
    o, lse = binding.attn_fwd(q.to(dev), k.to(dev), v.to(dev), causal=causal, window=window)
    return q, k, v, o, lse


BF16_CASES = [  # (B, Hq, Hkv, Nq, Nk, causal, window)
    (1, 2, 2, 128, 128, False, 0),        # one tile
    (1, 2, 2, 300, 300, False, 0),        # ragged tail, two Q tiles
    (2, 4, 2, 513, 513, True, 0),         # GQA, causal, ragged
    (1, 2, 1, 256, 1000, True, 0),        # Nq < Nk
    (1, 2, 2, 700, 300, True, 0),         # Nq > Nk: fully masked rows
    (1, 2, 2, 1000, 1000, True, 100),     # causal + window
    (1, 2, 2, 600, 600, False, 64),       # window only
    (1, 1, 1, 1, 1, False, 0),
    (1, 2, 2, 5, 3000, False, 0),
    (1, 3, 1, 257, 129, False, 0),
    (1, 4, 4, 1024, 1024, False, 0),      # several full K/V tiles
]


@pytest.mark.parametrize("case", BF16_CASES, ids=str)
def test_bf16_cases(dev, case):
    B, Hq, Hkv, Nq, Nk, causal, window = case
    q, k, v, o, lse = run_bf16(dev, B, Hq, Hkv, Nq, Nk, causal, window, seed=11)
    O, L = oracle.attention_forward(q, k, v, 1 / math.sqrt(128), causal, window)
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)


BF16_D64_CASES = [  # (B, Hq, Hkv, Nq, Nk, causal, window)
    (1, 2, 2, 128, 128, False, 0),
    (1, 2, 2, 300, 300, False, 0),
    (2, 4, 2, 513, 513, True, 0),
    (1, 2, 1, 256, 1000, True, 0),
    (1, 2, 2, 700, 300, True, 0),
    (1, 2, 2, 1000, 1000, True, 100),
    (1, 4, 4, 2048, 2048, False, 0),
]


@pytest.mark.parametrize("case", BF16_D64_CASES, ids=str)
def test_bf16_head_dim_64(dev, case):
    B, Hq, Hkv, Nq, Nk, causal, window = case
    q, k, v, o, lse = run_bf16(dev, B, Hq, Hkv, Nq, Nk, causal, window, seed=13, D=64)
    O, L = oracle.attention_forward(q, k, v, 1 / math.sqrt(64), causal, window)
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)


FP16_CASES = [  # (B, Hq, Hkv, Nq, Nk, D, causal, window)
    (1, 2, 2, 300, 300, 128, False, 0),
    (2, 4, 2, 513, 513, 128, True, 0),
    (1, 2, 1, 256, 1000, 128, True, 0),
    (1, 2, 2, 1000, 1000, 64, True, 100),
    (1, 4, 4, 1024, 1024, 64, False, 0),
]


@pytest.mark.parametrize("case", FP16_CASES, ids=str)
def test_fp16_forward(dev, case):
    B, Hq, Hkv, Nq, Nk, D, causal, window = case
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, D, "fp16", seed=17)
    o, lse = binding.attn_fwd_fp16(q.to(dev), k.to(dev), v.to(dev), causal=causal, window=window)
    O, L = oracle.attention_forward(q, k, v, 1 / math.sqrt(D), causal, window)
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)


def test_fp16_dense_workload_sampled(dev):
    q, k, v = inputs.prefill_inputs(1, 32, 32, 8192, 8192, 128, "fp16", seed=0)
    o, lse = binding.attn_fwd_fp16(q.to(dev), k.to(dev), v.to(dev))
    rows = sample_rows(1, 32, 8192, 64, seed=4)
    O, L = oracle.attention_rows(q, k, v, 1 / math.sqrt(128), rows)
    idx = tuple(np.array(rows).T)
    check(o.cpu()[idx], lse.cpu()[idx], O, L, BF16_O_TOL, BF16_LSE_REL, True)


VARLEN_CASES = [  # (lens_q, lens_k, Hq, Hkv, D, causal, window)
    ([1, 300, 0, 1000, 129], [1, 300, 0, 1000, 129], 4, 2, 128, True, 0),
    ([1, 300, 0, 1000, 129], [1, 300, 0, 1000, 129], 4, 2, 128, False, 0),
    ([64, 200, 513], [700, 200, 1100], 4, 4, 128, True, 0),     # chunked prefill per sequence
    ([257, 5, 800], [257, 0, 800], 2, 1, 64, True, 100),        # a sequence without keys
]


@pytest.mark.parametrize("case", VARLEN_CASES, ids=str)
def test_bf16_varlen(dev, case):
    lens_q, lens_k, Hq, Hkv, D, causal, window = case
    q, k, v, cq, ck = inputs.varlen_inputs(lens_q, lens_k, Hq, Hkv, D, "bf16", seed=19)
    o, lse = binding.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), max(lens_q),
                                     causal=causal, window=window)
    O, L = oracle.attention_varlen(q, k, v, cq, ck, 1 / math.sqrt(D), causal, window)
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    assert binding.get_device_error() == 0


def test_bf16_varlen_benchmark_workload_sampled(dev):
    """The benchmark's ragged batch (32 causal sequences, lengths ~U[512, 8192], Hq=32 Hkv=8,
    the bench's draws and launch): sampled rows of every sequence, including its first and
    last, against the oracle on that sequence alone."""
    Hq, Hkv, D = 32, 8, 128
    lens = torch.randint(512, 8192 + 1, (32,), generator=torch.Generator("cpu").manual_seed(11)).tolist()
    q, k, v, cq, ck = inputs.varlen_inputs(lens, lens, Hq, Hkv, D, "bf16", 0)
    o, lse = binding.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), max(lens),
                                     causal=True)
    o, lse = o.cpu(), lse.cpu()
    assert binding.get_device_error() == 0
    rng = np.random.default_rng(3)
    for b, n in enumerate(lens):
        t0 = int(cq[b])
        seq = lambda x: x[t0:t0 + n].permute(1, 0, 2).unsqueeze(0)  # noqa: E731  [1, H, n, D]
        rows = sorted({(0, int(rng.integers(Hq)), i)
                       for i in (0, n - 1, int(rng.integers(n)), int(rng.integers(n)), int(rng.integers(n)))})
        O, L = oracle.attention_rows(seq(q), seq(k), seq(v), 1 / math.sqrt(D), rows, True)
        hs = [h for _, h, _ in rows]
        ts = [t0 + i for _, _, i in rows]
        check(o[ts, hs], lse[hs, ts], O, L, BF16_O_TOL, BF16_LSE_REL, True)


@pytest.mark.parametrize("name,B,Hq,Hkv,Nq,Nk,D,causal,window", [
    ("sliding_window_4096_B1_H32_KV8_N16384", 1, 32, 8, 16384, 16384, 128, True, 4096),
    ("chunked_prefill_B1_H32_KV8_Nq2048_Nk16384", 1, 32, 8, 2048, 16384, 128, True, 0),
    ("dense_d64_B1_H32_N8192", 1, 32, 32, 8192, 8192, 64, False, 0),
])
def test_bf16_widened_workloads_sampled(dev, name, B, Hq, Hkv, Nq, Nk, D, causal, window):
    """Sliding window, chunked prefill (Nq < Nk, bottom-right causal) and D=64 at full size."""
    q, k, v, o, lse = run_bf16(dev, B, Hq, Hkv, Nq, Nk, causal, window, seed=1, D=D)
    assert torch.isfinite(o.float()).all().item() and torch.isfinite(lse).all().item()
    rows = sample_rows(B, Hq, Nq, 64, seed=9)
    O, L = oracle.attention_rows(q, k, v, 1 / math.sqrt(D), rows, causal, window)
    idx = tuple(np.array(rows).T)
    check(o.cpu()[idx], lse.cpu()[idx], O, L, BF16_O_TOL, BF16_LSE_REL, True)


@pytest.mark.parametrize("name,B,Hq,Hkv,N,causal", [
    ("dense_B1_H32_N8192", 1, 32, 32, 8192, False),
    ("causal_gqa_B4_H32_KV8_N4096", 4, 32, 8, 4096, True),
])
def test_bf16_benchmark_workloads_sampled(dev, name, B, Hq, Hkv, N, causal):
    """The benchmark's prefill workloads, checked on sampled rows."""
    q, k, v, o, lse = run_bf16(dev, B, Hq, Hkv, N, N, causal, 0, seed=0)
    assert torch.isfinite(o.float()).all().item() and torch.isfinite(lse).all().item()
    rows = sample_rows(B, Hq, N, 96, seed=5)
    O, L = oracle.attention_rows(q, k, v, 1 / math.sqrt(128), rows, causal)
    idx = tuple(np.array(rows).T)
    check(o.cpu()[idx], lse.cpu()[idx], O, L, BF16_O_TOL, BF16_LSE_REL, True)


# ---------------------------------------------------------------- decode
def run_decode(dev, B, Hq, Hkv, lens, nk_max, chunk, seed=0):
    _, q = inputs.decode_seqlens_and_q(B, Hq, 128, 1, 2, seed)
    seqlens = torch.tensor(lens, dtype=torch.int32)
    kc = torch.full((B, nk_max, Hkv, 128), inputs.K_SENTINEL, dtype=torch.bfloat16)
    vc = torch.full((B, nk_max, Hkv, 128), inputs.V_SENTINEL, dtype=torch.bfloat16)
    for b, n in enumerate(lens):
        kb, vb = inputs.decode_kv_rows(seed, b, n, Hkv, 128)
        kc[b, :n], vc[b, :n] = kb, vb
    ws = torch.empty(binding.attn_decode_workspace_size(B, Hq, 128, nk_max, chunk), device=dev,
                     dtype=torch.uint8)
    o, lse = binding.attn_decode(q.to(dev), kc.to(dev), vc.to(dev), seqlens.to(dev), ws, chunk=chunk)
    return q, kc, vc, seqlens, ws, o, lse


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("chunk", [64, 512, 1024])
def test_decode_small(dev, G, chunk):
    lens = [1, 64, 511, 512, 513, 1500, 2048]
    B, Hkv = len(lens), 2
    Hq = G * Hkv
    q, kc, vc, seqlens, ws, o, lse = run_decode(dev, B, Hq, Hkv, lens, 2048, chunk, seed=G + chunk)
    scale = 1 / math.sqrt(128)
    O, L = oracle.decode_forward(q, kc, vc, seqlens, scale)
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    # the partial step on its own, valid chunks only
    Op, Lp, ns = oracle.decode_split_partials(q, kc, vc, seqlens, scale, chunk)
    S_max = Op.shape[2]
    wsf = ws.view(torch.float32).cpu().numpy()
    go = wsf[: B * Hq * S_max * 128].reshape(B, Hq, S_max, 128)
    gl = wsf[B * Hq * S_max * 128: B * Hq * S_max * 129].reshape(B, Hq, S_max)
    for b in range(B):
        n = int(ns[b])
        assert np.abs(go[b, :, :n] - Op[b, :, :n]).max() <= BF16_O_TOL
        assert (np.abs(gl[b, :, :n] - Lp[b, :, :n]) / np.maximum(1, np.abs(Lp[b, :, :n]))).max() <= BF16_LSE_REL
    assert binding.get_device_error() == 0


def test_decode_benchmark_workload_sampled(dev):
    """B=64 Hq=32 Hkv=8, Nk_b ~ U[512, 32768], chunk 512: sampled sequences.

    The 8.6 GB cache is drawn on the device; the sampled sequences' rows are
    copied back for the oracle.
    """
    q, kc, vc, seqlens = inputs.decode_inputs(64, 32, 8, 128, 512, 32768, seed=0, device=dev)
    o, lse = binding.attn_decode(q.to(dev), kc, vc, seqlens.to(dev), chunk=512)
    lens = seqlens.numpy()
    batches = sorted({int(lens.argmax()), int(lens.argmin()), 0, 17, 40, 63})
    O = np.zeros((len(batches), 32, 128))
    L = np.zeros((len(batches), 32))
    for n, b in enumerate(batches):
        nk = int(lens[b])
        Ob, Lb = oracle.decode_forward(q[b:b + 1], kc[b:b + 1, :nk].cpu(), vc[b:b + 1, :nk].cpu(),
                                       [nk], 1 / math.sqrt(128))
        O[n], L[n] = Ob[0], Lb[0]
    check(o.cpu()[batches], lse.cpu()[batches], O, L, BF16_O_TOL, BF16_LSE_REL, True)
    assert binding.get_device_error() == 0


@pytest.mark.parametrize("page_size,chunk,G", [(64, 512, 4), (256, 512, 4), (128, 64, 2), (512, 1024, 8)])
def test_decode_paged_small(dev, page_size, chunk, G):
    """Paged cache with sequences scattered over the pool (and spare pages)."""
    B, Hkv = 7, 2
    Hq = G * Hkv
    q, kp, vp, bt, sl = inputs.paged_decode_inputs(B, Hq, Hkv, 128, 1, 3000, page_size, seed=page_size + G,
                                                   spare_pages=5)
    o, lse = binding.attn_decode_paged(q.to(dev), kp.to(dev), vp.to(dev), bt.to(dev), sl.to(dev), chunk=chunk)
    O, L = oracle.decode_forward_paged(q, kp, vp, bt, sl, 1 / math.sqrt(128))
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    assert binding.get_device_error() == 0


def test_decode_paged_benchmark_workload_sampled(dev):
    """B=64 Hq=32 Hkv=8, Nk_b ~ U[512, 32768], page 256, chunk 512: sampled sequences."""
    q, kp, vp, bt, sl = inputs.paged_decode_inputs(64, 32, 8, 128, 512, 32768, 256, seed=0, device=dev)
    o, lse = binding.attn_decode_paged(q.to(dev), kp, vp, bt.to(dev), sl.to(dev), chunk=512)
    lens = sl.numpy()
    batches = sorted({int(lens.argmax()), int(lens.argmin()), 3, 31, 50})
    O = np.zeros((len(batches), 32, 128))
    L = np.zeros((len(batches), 32))
    for n, b in enumerate(batches):
        pages = bt[b, : -(-int(lens[b]) // 256)].long()
        kb, vb = kp[pages.to(dev)].cpu(), vp[pages.to(dev)].cpu()   # this sequence's pages, in order
        Ob, Lb = oracle.decode_forward_paged(q[b:b + 1], kb, vb, [list(range(len(pages)))], [int(lens[b])],
                                             1 / math.sqrt(128))
        O[n], L[n] = Ob[0], Lb[0]
    check(o.cpu()[batches], lse.cpu()[batches], O, L, BF16_O_TOL, BF16_LSE_REL, True)
    assert binding.get_device_error() == 0


def test_decode_nan_in_unused_cache_rows_does_not_leak(dev):
    """Rows past a sequence's end may hold anything, NaN included."""
    lens = [5, 700, 1]
    B, Hq, Hkv, nk_max = 3, 8, 2, 1024
    _, q = inputs.decode_seqlens_and_q(B, Hq, 128, 1, 2, 6)
    kc = torch.full((B, nk_max, Hkv, 128), float("nan"), dtype=torch.bfloat16)
    vc = torch.full((B, nk_max, Hkv, 128), float("nan"), dtype=torch.bfloat16)
    for b, n in enumerate(lens):
        kb, vb = inputs.decode_kv_rows(6, b, n, Hkv, 128)
        kc[b, :n], vc[b, :n] = kb, vb
    o, lse = binding.attn_decode(q.to(dev), kc.to(dev), vc.to(dev), torch.tensor(lens, dtype=torch.int32).to(dev))
    O, L = oracle.decode_forward(q, kc, vc, lens, 1 / math.sqrt(128))
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)


def test_decode_bad_seqlen_reported(dev):
    """A sequence length outside [1, Nk_max] is skipped and reported; others stay correct."""
    B, Hq, Hkv, nk_max = 3, 8, 2, 1024
    _, q = inputs.decode_seqlens_and_q(B, Hq, 128, 1, 2, 4)
    kc = torch.zeros(B, nk_max, Hkv, 128, dtype=torch.bfloat16)
    vc = torch.zeros(B, nk_max, Hkv, 128, dtype=torch.bfloat16)
    kb, vb = inputs.decode_kv_rows(4, 1, 700, Hkv, 128)
    kc[1, :700], vc[1, :700] = kb, vb
    seqlens = torch.tensor([0, 700, nk_max + 5], dtype=torch.int32)
    assert binding.get_device_error() == 0
    o, lse = binding.attn_decode(q.to(dev), kc.to(dev), vc.to(dev), seqlens.to(dev), chunk=512)
    assert binding.get_device_error() == -10  # ATTN_ERR_SEQLEN
    O, L = oracle.decode_forward(q, kc, vc, [1, 700, 1], 1 / math.sqrt(128), batches=[1])
    check(o.cpu()[1:2], lse.cpu()[1:2], O[1:2], L[1:2], BF16_O_TOL, BF16_LSE_REL, True)
    assert torch.all(o.cpu()[[0, 2]].float() == 0) and torch.all(lse.cpu()[[0, 2]] == -math.inf)
    assert binding.get_device_error() == 0


# ---------------------------------------------------------------- fp8 (E4M3) KV cache
FP8_SCALES = (0.37, 1.9)   # k_scale, v_scale: values are code * scale


@pytest.mark.parametrize("G,chunk", [(1, 512), (4, 512), (8, 64), (2, 1024)])
def test_decode_fp8_small(dev, G, chunk):
    """fp8 E4M3 cache: ragged lengths around the chunk and tile sizes."""
    lens = [1, 63, 64, 511, 513, 1500, 2048]
    B, Hkv = len(lens), 2
    Hq = G * Hkv
    ks, vs = FP8_SCALES
    q, kc, vc, _ = inputs.decode_inputs(B, Hq, Hkv, 128, 1, 2, seed=G + chunk, nk_max=2048, kv_dtype="e4m3")
    sl = torch.tensor(lens, dtype=torch.int32)
    # regenerate rows for the chosen lengths (the drawn lengths are ignored)
    for b, n in enumerate(lens):
        kb, vb = inputs.decode_kv_rows(G + chunk, b, n, Hkv, 128, kv_dtype="e4m3")
        kc[b, :n], vc[b, :n] = kb, vb
    o, lse = binding.attn_decode_fp8(q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), ks, vs, chunk=chunk)
    O, L = oracle.decode_forward_fp8(q, kc.numpy(), vc.numpy(), ks, vs, lens, 1 / math.sqrt(128))
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    assert binding.get_device_error() == 0


@pytest.mark.parametrize("page_size,chunk,G", [(64, 512, 4), (256, 512, 8), (128, 64, 2)])
def test_decode_fp8_paged_small(dev, page_size, chunk, G):
    """Paged fp8 cache, sequences scattered over the pool (and spare pages)."""
    B, Hkv = 6, 2
    Hq = G * Hkv
    ks, vs = FP8_SCALES
    q, kp, vp, bt, sl = inputs.paged_decode_inputs(B, Hq, Hkv, 128, 1, 3000, page_size, seed=page_size + G,
                                                   spare_pages=5, kv_dtype="e4m3")
    o, lse = binding.attn_decode_paged_fp8(q.to(dev), kp.to(dev), vp.to(dev), bt.to(dev), sl.to(dev), ks, vs,
                                           chunk=chunk)
    O, L = oracle.decode_forward_paged_fp8(q, kp.numpy(), vp.numpy(), ks, vs, bt, sl, 1 / math.sqrt(128))
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    assert binding.get_device_error() == 0


def test_decode_fp8_benchmark_workload_sampled(dev):
    """B=64 Hq=32 Hkv=8, Nk_b ~ U[512, 32768], chunk 512, fp8 cache: sampled sequences."""
    ks, vs = FP8_SCALES
    q, kc, vc, seqlens = inputs.decode_inputs(64, 32, 8, 128, 512, 32768, seed=0, device=dev, kv_dtype="e4m3")
    o, lse = binding.attn_decode_fp8(q.to(dev), kc, vc, seqlens.to(dev), ks, vs, chunk=512)
    lens = seqlens.numpy()
    batches = sorted({int(lens.argmax()), int(lens.argmin()), 0, 21, 63})
    O = np.zeros((len(batches), 32, 128))
    L = np.zeros((len(batches), 32))
    for n, b in enumerate(batches):
        nk = int(lens[b])
        Ob, Lb = oracle.decode_forward_fp8(q[b:b + 1], kc[b:b + 1, :nk].cpu().numpy(),
                                           vc[b:b + 1, :nk].cpu().numpy(), ks, vs, [nk], 1 / math.sqrt(128))
        O[n], L[n] = Ob[0], Lb[0]
    check(o.cpu()[batches], lse.cpu()[batches], O, L, BF16_O_TOL, BF16_LSE_REL, True)
    assert binding.get_device_error() == 0


def test_decode_fp8_nan_codes_in_unused_rows_do_not_leak(dev):
    """Rows past a sequence's end hold NaN codes (0x7F, 0xFF): never weighted."""
    lens = [5, 700, 1]
    B, Hq, Hkv, nk_max = 3, 8, 2, 1024
    _, q = inputs.decode_seqlens_and_q(B, Hq, 128, 1, 2, 6)
    kc = torch.full((B, nk_max, Hkv, 128), 0x7F, dtype=torch.uint8)
    vc = torch.full((B, nk_max, Hkv, 128), 0xFF, dtype=torch.uint8)
    for b, n in enumerate(lens):
        kb, vb = inputs.decode_kv_rows(6, b, n, Hkv, 128, kv_dtype="e4m3")
        kc[b, :n], vc[b, :n] = kb, vb
    o, lse = binding.attn_decode_fp8(q.to(dev), kc.to(dev), vc.to(dev), torch.tensor(lens, dtype=torch.int32).to(dev),
                                     1.0, 1.0)
    O, L = oracle.decode_forward_fp8(q, kc.numpy(), vc.numpy(), 1.0, 1.0, lens, 1 / math.sqrt(128))
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)


# ---------------------------------------------------------------- softcap and attention sinks
def _sinks(Hq, kind, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    if kind is None:
        return None
    s = torch.randn(Hq, generator=g) * 2.0
    if kind == "extreme":          # one head never attends (sink dominates), one has no sink
        s[0] = 30.0
        s[-1] = -math.inf
    return s.float()


SOFTCAP_CASES = [
    # B, Hq, Hkv, Nq, Nk, D, causal, window, cap, sinks
    (1, 4, 4, 300, 300, 128, False, 0, 20.0, "normal"),
    (2, 8, 2, 257, 257, 128, True, 0, 5.0, "extreme"),
    (1, 4, 2, 300, 130, 128, True, 0, 10.0, "normal"),    # rows 0..169 see no key
    (1, 4, 1, 384, 384, 128, True, 64, 0.0, "normal"),    # sinks only
    (2, 4, 2, 200, 333, 64, False, 0, 30.0, None),        # cap only, D = 64
    (1, 8, 8, 129, 1000, 128, True, 0, 50.0, "extreme"),  # chunked-prefill shape
]


@pytest.mark.parametrize("case", SOFTCAP_CASES, ids=lambda c: "-".join(map(str, c)))
def test_softcap_sink(dev, case):
    B, Hq, Hkv, Nq, Nk, D, causal, window, cap, kind = case
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, D, "bf16", seed=Nq + Nk)
    sinks = _sinks(Hq, kind, Nq)
    o, lse = binding.attn_fwd_softcap_sink(q.to(dev), k.to(dev), v.to(dev), causal=causal, window=window,
                                           softcap=cap, sinks=None if sinks is None else sinks.to(dev))
    O, L = oracle.attention_forward_ext(q, k, v, 1 / math.sqrt(D), causal, window, cap,
                                        None if sinks is None else sinks.numpy())
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    if causal and Nq > Nk and sinks is not None:   # rows with no visible key: O = 0, LSE = sink
        lo = lse.cpu()[:, :, : Nq - Nk]
        assert torch.all(o.cpu()[:, :, : Nq - Nk].float() == 0)
        assert torch.equal(lo, sinks.view(1, Hq, 1).expand_as(lo))
    assert binding.get_device_error() == 0


def test_softcap_sink_full_size_sampled(dev):
    """Dense B=1 H=32 N=8192 D=128, softcap 50 and per-head sinks: sampled rows."""
    q, k, v = inputs.prefill_inputs(1, 32, 32, 8192, 8192, 128, "bf16", seed=0)
    sinks = _sinks(32, "extreme", 9)
    o, lse = binding.attn_fwd_softcap_sink(q.to(dev), k.to(dev), v.to(dev), softcap=50.0, sinks=sinks.to(dev))
    rows = sample_rows(1, 32, 8192, 24, seed=3)
    O, L = oracle.attention_rows_ext(q, k, v, 1 / math.sqrt(128), rows, False, 0, 50.0, sinks.numpy())
    og = torch.stack([o[b, h, i] for b, h, i in rows]).cpu()
    lg = torch.stack([lse[b, h, i] for b, h, i in rows]).cpu()
    check(og, lg, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    assert binding.get_device_error() == 0


# ---------------------------------------------------------------- backward
BWD_CASES = [
    # B, Hq, Hkv, Nq, Nk, causal
    (1, 2, 2, 200, 200, False),
    (2, 4, 2, 257, 257, True),      # GQA, ragged tiles
    (1, 4, 1, 130, 300, True),      # bottom-right causal, Nq < Nk
    (1, 2, 2, 300, 130, True),      # Nq > Nk: rows 0..169 see no key
    (1, 2, 1, 64, 1000, False),     # one query tile, many key tiles
    (1, 4, 2, 384, 384, True),      # whole tiles only, two query heads per KV head
    (2, 2, 1, 5, 37, True),         # fewer queries than one 32-row dQ box
]


def _bwd_check(got, want, name):
    """Each gradient against 2 % of its tensor's largest magnitude (P, dS and O are
    rounded to bf16, relative 2^-9, before the fp32 sums)."""
    g = got.float().cpu().numpy()
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    err = float(np.abs(g - want).max())
    tol = 2e-2 * max(1.0, float(np.abs(want).max()))
    assert err <= tol, f"{name}: max-abs err {err:.3e} (tol {tol:.3e})"
    return err


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward(dev, case):
    B, Hq, Hkv, Nq, Nk, causal = case
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, 128, "bf16", seed=Nq * 7 + Nk)
    g = torch.Generator("cpu").manual_seed(Nq + 3)
    do = torch.randn(B, Hq, Nq, 128, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = binding.attn_fwd(qd, kd, vd, causal=causal)
    dq, dk, dv = binding.attn_bwd(qd, kd, vd, o, dod, lse, causal=causal)
    dQ, dK, dV = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(128), causal, 0)
    _bwd_check(dq, dQ, "dQ")
    _bwd_check(dk, dK, "dK")
    _bwd_check(dv, dV, "dV")
    assert binding.get_device_error() == 0


def test_backward_full_size_two_heads(dev):
    """The benchmarked backward (B=1 H=32 N=8192 D=128, non-causal, the bench's inputs and dO
    draw and the same launch): every dQ, dK and dV row of heads 0 and 17 against the oracle,
    whose per-head fp64 backward fits this size (about 86 GFLOP and 2.6 GB per head)."""
    B, H, N, D, seed = 1, 32, 8192, 128, 0
    q, k, v = inputs.prefill_inputs(B, H, H, N, N, D, "bf16", seed)
    do = torch.randn(B, H, N, D, generator=torch.Generator("cpu").manual_seed(seed + 9)).to(torch.bfloat16)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = binding.attn_fwd(qd, kd, vd)
    dq, dk, dv = binding.attn_bwd(qd, kd, vd, o, dod, lse)
    torch.cuda.synchronize()
    assert binding.get_device_error() == 0
    for h in (0, 17):
        sl = slice(h, h + 1)
        dQ, dK, dV = oracle.attention_backward(q[:, sl], k[:, sl], v[:, sl], do[:, sl], 1 / math.sqrt(D), False, 0)
        _bwd_check(dq[:, sl], dQ, f"dQ head {h}")
        _bwd_check(dk[:, sl], dK, f"dK head {h}")
        _bwd_check(dv[:, sl], dV, f"dV head {h}")


def test_backward_multi_tile(dev):
    """B=1 Hq=4 Hkv=2 N=2048 causal: 16 key tiles x 32 query tiles per head."""
    q, k, v = inputs.prefill_inputs(1, 4, 2, 2048, 2048, 128, "bf16", seed=5)
    do = torch.randn(1, 4, 2048, 128, generator=torch.Generator("cpu").manual_seed(6)).to(torch.bfloat16)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = binding.attn_fwd(qd, kd, vd, causal=True)
    dq, dk, dv = binding.attn_bwd(qd, kd, vd, o, dod, lse, causal=True)
    dQ, dK, dV = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(128), True, 0)
    _bwd_check(dq, dQ, "dQ")
    _bwd_check(dk, dK, "dK")
    _bwd_check(dv, dV, "dV")
    assert binding.get_device_error() == 0
