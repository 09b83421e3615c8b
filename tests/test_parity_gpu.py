"""GPU parity: the CUDA kernels (through the C ABI) against the fp64 oracle.

Tolerances (fixed by the attention-forward target):
  * fp32 inputs: max-abs error <= 1e-4 on O and on LSE;
  * bf16 inputs (fp32 accumulation): max-abs error <= 2e-2 on O and
    |dLSE| <= 1e-2 * max(1, |LSE|) on LSE.
Rows that see no key must give O = 0 and LSE = -inf on both sides.
Small and ragged shapes are compared element by element.  The benchmark's
dense, causal GQA and split-KV decode workloads are compared element by element
on every output (the oracle runs over (batch, head) slices on every host core);
the other full-size workloads on sampled rows that the oracle computes one by one.
Every output and workspace the library writes sits between canary-filled guard
regions (``helpers.Guarded``) that are checked after the call.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import check_guards, compare_rows, guarded, parallel_map
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
    go, gl = guarded(q.shape, torch.float32, dev), guarded((B, Hq, Nq), torch.float32, dev)
    o, lse = binding.attn_fwd_fp32(q.to(dev), k.to(dev), v.to(dev), go.t, gl.t, causal=causal, window=window)
    check_guards(go, gl)
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
    go, gl = guarded(q.shape, torch.bfloat16, dev), guarded((B, Hq, Nq), torch.float32, dev)
    o, lse = binding.attn_fwd(q.to(dev), k.to(dev), v.to(dev), go.t, gl.t, causal=causal, window=window)
    check_guards(go, gl)
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


@pytest.mark.parametrize("D", [64, 128])
def test_bf16_output_only_16_byte_aligned(dev, D):
    """O at an address that is 16- but not 32-byte aligned takes the 16-byte store path of
    the epilogue; the result must equal the 32-byte-aligned call bit for bit."""
    B, Hq, Hkv, N = 1, 2, 2, 300
    q, k, v = (x.to(dev) for x in inputs.prefill_inputs(B, Hq, Hkv, N, N, D, "bf16", seed=21))
    o_ref, lse_ref = binding.attn_fwd(q, k, v, causal=True)
    n = B * Hq * N * D * 2
    buf = torch.full((n + 16 + 4096,), 0xA5, dtype=torch.uint8, device=dev)
    o16 = buf[16:16 + n].view(torch.bfloat16).view(B, Hq, N, D)
    assert o16.data_ptr() % 32 == 16
    binding.attn_fwd(q, k, v, o16, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o16, o_ref)
    assert int((buf[:16] != 0xA5).sum()) == 0 and int((buf[16 + n:] != 0xA5).sum()) == 0


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
    go, gl = guarded(q.shape, torch.float16, dev), guarded((B, Hq, Nq), torch.float32, dev)
    o, lse = binding.attn_fwd_fp16(q.to(dev), k.to(dev), v.to(dev), go.t, gl.t, causal=causal, window=window)
    check_guards(go, gl)
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
    go, gl = guarded(q.shape, torch.bfloat16, dev), guarded((Hq, q.shape[0]), torch.float32, dev)
    o, lse = binding.attn_fwd_varlen(q.to(dev), k.to(dev), v.to(dev), cq.to(dev), ck.to(dev), max(lens_q),
                                     go.t, gl.t, causal=causal, window=window)
    check_guards(go, gl)
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
def test_bf16_benchmark_workloads_full(dev, name, B, Hq, Hkv, N, causal):
    """The benchmark's prefill workloads (its draws and launch), every O and LSE element
    against the oracle, one (batch, head) slice per task on every host core."""
    q, k, v, o, lse = run_bf16(dev, B, Hq, Hkv, N, N, causal, 0, seed=0)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    g = Hq // Hkv

    def one(bh):
        b, h = divmod(bh, Hq)
        O, L = oracle.attention_forward(q[b:b + 1, h:h + 1], k[b:b + 1, h // g:h // g + 1],
                                        v[b:b + 1, h // g:h // g + 1], 1 / math.sqrt(128), causal)
        return compare_rows(o[b, h], lse[b, h], O[0, 0], L[0, 0])

    res = parallel_map(one, range(B * Hq))
    err_o = max(r[0] for r in res)
    err_l = max(r[1] for r in res)
    print(f"[achieved] {name} full: O err {err_o:.3e}, LSE err {err_l:.3e}")
    assert all(r[2] for r in res), "non-finite output or LSE finiteness mismatch"
    assert err_o <= BF16_O_TOL and err_l <= BF16_LSE_REL, f"O err {err_o:.3e}, LSE err {err_l:.3e}"


# ---------------------------------------------------------------- fp8 (E4M3) Q/K/V prefill
def run_fp8(dev, B, Hq, Hkv, Nq, Nk, causal=False, window=0, seed=0, scales=(1.0, 1.0, 1.0)):
    q, k, v = inputs.prefill_inputs_fp8(B, Hq, Hkv, Nq, Nk, 128, seed)
    gw = guarded((binding.attn_fwd_fp8_workspace_size(B, Hkv, Nk, 128),), torch.uint8, dev)
    go, gl = guarded((B, Hq, Nq, 128), torch.bfloat16, dev), guarded((B, Hq, Nq), torch.float32, dev)
    o, lse = binding.attn_fwd_fp8(q.to(dev), k.to(dev), v.to(dev), *scales, go.t, gl.t, gw.t,
                                  causal=causal, window=window)
    check_guards(gw, go, gl)
    return q.numpy(), k.numpy(), v.numpy(), o, lse


FP8_CASES = [  # (B, Hq, Hkv, Nq, Nk, causal, window, (q_scale, k_scale, v_scale))
    (1, 2, 2, 128, 128, False, 0, (1.0, 1.0, 1.0)),      # one tile
    (1, 2, 2, 300, 300, False, 0, (2.0, 0.5, 0.75)),     # ragged tail, scales folded
    (2, 4, 2, 513, 513, True, 0, (1.0, 1.0, 1.0)),       # GQA, causal, ragged
    (1, 2, 1, 256, 1000, True, 0, (0.25, 4.0, 3.0)),     # Nq < Nk
    (1, 2, 2, 700, 300, True, 0, (1.0, 1.0, 1.0)),       # Nq > Nk: fully masked rows
    (1, 2, 2, 1000, 1000, True, 100, (1.0, 1.0, 1.0)),   # causal + window
    (1, 2, 2, 600, 600, False, 64, (1.0, 1.0, 1.0)),     # window only
    (1, 1, 1, 1, 1, False, 0, (1.0, 1.0, 1.0)),
    (1, 3, 1, 257, 129, False, 0, (1.0, 1.0, 1.0)),
    (1, 4, 4, 1024, 1024, False, 0, (0.5, 0.5, 1.0)),    # several full K/V tiles
]


@pytest.mark.parametrize("case", FP8_CASES, ids=str)
def test_fp8_prefill_cases(dev, case):
    B, Hq, Hkv, Nq, Nk, causal, window, scales = case
    q, k, v, o, lse = run_fp8(dev, B, Hq, Hkv, Nq, Nk, causal, window, seed=23, scales=scales)
    O, L = oracle.attention_forward_fp8(q, k, v, *scales, 1 / math.sqrt(128), causal, window)
    err = check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    print(f"[achieved] fp8 prefill {case}: O err {err:.3e}")
    assert binding.get_device_error() == 0


def test_fp8_prefill_benchmark_workload_full(dev):
    """The benchmark's fp8 prefill workload (B=1 H=32 N=8192 D=128 dense, its draws and
    launch): every O and LSE element against the oracle, one head per task."""
    B, H, N = 1, 32, 8192
    q, k, v, o, lse = run_fp8(dev, B, H, H, N, N, seed=0)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()

    def one(h):
        O, L = oracle.attention_forward_fp8(q[:, h:h + 1], k[:, h:h + 1], v[:, h:h + 1], 1.0, 1.0, 1.0,
                                            1 / math.sqrt(128))
        return compare_rows(o[0, h], lse[0, h], O[0, 0], L[0, 0])

    res = parallel_map(one, range(H))
    err_o = max(r[0] for r in res)
    err_l = max(r[1] for r in res)
    print(f"[achieved] fp8 prefill B1 H32 N8192 full: O err {err_o:.3e}, LSE err {err_l:.3e}")
    assert all(r[2] for r in res), "non-finite output or LSE finiteness mismatch"
    assert err_o <= BF16_O_TOL and err_l <= BF16_LSE_REL, f"O err {err_o:.3e}, LSE err {err_l:.3e}"


def test_fp8_prefill_extreme_codes(dev):
    """Q and K at the largest E4M3 magnitude (448) and V with subnormal and maximal codes,
    with scales that keep the scaled scores moderate: the fp32 accumulation of 448^2
    products and the exact widening of every V code."""
    B, H, N = 1, 2, 384
    g = torch.Generator("cpu").manual_seed(29)
    q = torch.randint(0, 256, (B, H, N, 128), generator=g, dtype=torch.uint8)
    k = torch.randint(0, 256, (B, H, N, 128), generator=g, dtype=torch.uint8)
    v = torch.randint(0, 256, (B, H, N, 128), generator=g, dtype=torch.uint8)
    for t in (q, k, v):
        t[(t & 0x7F) == 0x7F] = 0x7E         # +-448 instead of NaN
    q[0, 0, :64] = 0x7E                      # rows of +448
    k[0, 0, 5::7] = 0x7E
    v[0, 1, ::3] = 0x01                      # smallest subnormal
    scales = (1.0 / 448, 1.0 / 448, 0.01)
    gw = guarded((binding.attn_fwd_fp8_workspace_size(B, H, N, 128),), torch.uint8, dev)
    go, gl = guarded((B, H, N, 128), torch.bfloat16, dev), guarded((B, H, N), torch.float32, dev)
    o, lse = binding.attn_fwd_fp8(q.to(dev), k.to(dev), v.to(dev), *scales, go.t, gl.t, gw.t, causal=True)
    check_guards(gw, go, gl)
    O, L = oracle.attention_forward_fp8(q.numpy(), k.numpy(), v.numpy(), *scales, 1 / math.sqrt(128), True)
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    # the widened V in the workspace is the exact bf16 value of every code
    wide = gw.t.view(torch.bfloat16).view(B, H, N, 128).float().cpu().numpy()
    assert np.array_equal(wide, oracle.e4m3_to_float(v.numpy()).astype(np.float32))


# ---------------------------------------------------------------- decode
def run_decode(dev, B, Hq, Hkv, lens, nk_max, chunk, seed=0, D=128, fill=None):
    _, q = inputs.decode_seqlens_and_q(B, Hq, D, 1, 2, seed)
    seqlens = torch.tensor(lens, dtype=torch.int32)
    kfill, vfill = (inputs.K_SENTINEL, inputs.V_SENTINEL) if fill is None else (fill, fill)
    kc = torch.full((B, nk_max, Hkv, D), kfill, dtype=torch.bfloat16)
    vc = torch.full((B, nk_max, Hkv, D), vfill, dtype=torch.bfloat16)
    for b, n in enumerate(lens):
        kb, vb = inputs.decode_kv_rows(seed, b, n, Hkv, D)
        kc[b, :n], vc[b, :n] = kb, vb
    gw = guarded((binding.attn_decode_workspace_size(B, Hq, D, nk_max, chunk),), torch.uint8, dev)
    go, gl = guarded((B, Hq, D), torch.bfloat16, dev), guarded((B, Hq), torch.float32, dev)
    ws = gw.t
    o, lse = binding.attn_decode(q.to(dev), kc.to(dev), vc.to(dev), seqlens.to(dev), ws, go.t, gl.t, chunk=chunk)
    check_guards(gw, go, gl)
    return q, kc, vc, seqlens, ws, o, lse


@pytest.mark.parametrize("D,G", [(128, 1), (128, 2), (128, 4), (128, 8), (128, 16), (128, 32),
                                 (64, 1), (64, 4), (64, 8), (64, 32)])
@pytest.mark.parametrize("chunk", [64, 512, 1024])
def test_decode_small(dev, D, G, chunk):
    """bf16 cache: D = 128 with up to 8 query heads per KV head runs the SIMT consumer,
    16 or 32 heads (MQA with Hkv = 1) and D = 64 the tensor-core consumer."""
    lens = [1, 64, 511, 512, 513, 1500, 2048]
    B = len(lens)
    Hkv = 2 if G < 32 else 1
    Hq = G * Hkv
    q, kc, vc, seqlens, ws, o, lse = run_decode(dev, B, Hq, Hkv, lens, 2048, chunk, seed=G + chunk, D=D)
    scale = 1 / math.sqrt(D)
    O, L = oracle.decode_forward(q, kc, vc, seqlens, scale)
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
    # the partial step on its own, valid chunks only
    Op, Lp, ns = oracle.decode_split_partials(q, kc, vc, seqlens, scale, chunk)
    S_max = Op.shape[2]
    wsf = ws.view(torch.float32).cpu().numpy()
    go = wsf[: B * Hq * S_max * D].reshape(B, Hq, S_max, D)
    gl = wsf[B * Hq * S_max * D: B * Hq * S_max * (D + 1)].reshape(B, Hq, S_max)
    for b in range(B):
        n = int(ns[b])
        assert np.abs(go[b, :, :n] - Op[b, :, :n]).max() <= BF16_O_TOL
        assert (np.abs(gl[b, :, :n] - Lp[b, :, :n]) / np.maximum(1, np.abs(Lp[b, :, :n]))).max() <= BF16_LSE_REL
    assert binding.get_device_error() == 0


def test_decode_benchmark_workload_full(dev):
    """B=64 Hq=32 Hkv=8, Nk_b ~ U[512, 32768], chunk 512 (the benchmark's draws and launch):
    every O and LSE element of every sequence against the oracle.

    The 8.6 GB cache is drawn on the device; each sequence's rows are copied back
    for the oracle, which runs one sequence per task on every host core.
    """
    q, kc, vc, seqlens = inputs.decode_inputs(64, 32, 8, 128, 512, 32768, seed=0, device=dev)
    B, Hq = 64, 32
    gw = guarded((binding.attn_decode_workspace_size(B, Hq, 128, 32768, 512),), torch.uint8, dev)
    go, gl = guarded((B, Hq, 128), torch.bfloat16, dev), guarded((B, Hq), torch.float32, dev)
    o, lse = binding.attn_decode(q.to(dev), kc, vc, seqlens.to(dev), gw.t, go.t, gl.t, chunk=512)
    check_guards(gw, go, gl)
    assert binding.get_device_error() == 0
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    lens = seqlens.numpy()

    def one(b):
        nk = int(lens[b])
        Ob, Lb = oracle.decode_forward(q[b:b + 1], kc[b:b + 1, :nk].cpu(), vc[b:b + 1, :nk].cpu(), [nk],
                                       1 / math.sqrt(128))
        return compare_rows(o[b], lse[b], Ob[0], Lb[0])

    res = parallel_map(one, range(B), threads=8)   # at most 8 sequences' fp64 caches in memory
    err_o = max(r[0] for r in res)
    err_l = max(r[1] for r in res)
    print(f"[achieved] decode B=64 full: O err {err_o:.3e}, LSE err {err_l:.3e}")
    assert all(r[2] for r in res), "non-finite output or LSE finiteness mismatch"
    assert err_o <= BF16_O_TOL and err_l <= BF16_LSE_REL, f"O err {err_o:.3e}, LSE err {err_l:.3e}"


@pytest.mark.parametrize("name,B,Hq,Hkv,D", [
    ("mqa_B128_Hq32_Hkv1_D128", 128, 32, 1, 128),
    ("d64_B64_Hq32_Hkv8", 64, 32, 8, 64),
])
def test_decode_widened_workloads_full(dev, name, B, Hq, Hkv, D):
    """Multi-query decode and head dimension 64 (the benchmark's draws: Nk_b ~ U[512, 32768],
    chunk 512): every O and LSE element against the oracle."""
    q, kc, vc, seqlens = inputs.decode_inputs(B, Hq, Hkv, D, 512, 32768, seed=0, device=dev)
    gw = guarded((binding.attn_decode_workspace_size(B, Hq, D, 32768, 512),), torch.uint8, dev)
    go, gl = guarded((B, Hq, D), torch.bfloat16, dev), guarded((B, Hq), torch.float32, dev)
    o, lse = binding.attn_decode(q.to(dev), kc, vc, seqlens.to(dev), gw.t, go.t, gl.t, chunk=512)
    check_guards(gw, go, gl)
    assert binding.get_device_error() == 0
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    lens = seqlens.numpy()

    def one(b):
        nk = int(lens[b])
        Ob, Lb = oracle.decode_forward(q[b:b + 1], kc[b:b + 1, :nk].cpu(), vc[b:b + 1, :nk].cpu(), [nk],
                                       1 / math.sqrt(D))
        return compare_rows(o[b], lse[b], Ob[0], Lb[0])

    res = parallel_map(one, range(B), threads=8)
    err_o = max(r[0] for r in res)
    err_l = max(r[1] for r in res)
    print(f"[achieved] decode {name} full: O err {err_o:.3e}, LSE err {err_l:.3e}")
    assert all(r[2] for r in res), "non-finite output or LSE finiteness mismatch"
    assert err_o <= BF16_O_TOL and err_l <= BF16_LSE_REL, f"O err {err_o:.3e}, LSE err {err_l:.3e}"


@pytest.mark.parametrize("page_size,chunk,G,D", [(64, 512, 4, 128), (256, 512, 4, 128), (128, 64, 2, 128),
                                                 (512, 1024, 8, 128), (64, 512, 16, 128), (128, 512, 4, 64)])
def test_decode_paged_small(dev, page_size, chunk, G, D):
    """Paged cache with sequences scattered over the pool (and spare pages)."""
    B, Hkv = 7, 2
    Hq = G * Hkv
    q, kp, vp, bt, sl = inputs.paged_decode_inputs(B, Hq, Hkv, D, 1, 3000, page_size, seed=page_size + G,
                                                   spare_pages=5)
    gw = guarded((binding.attn_decode_workspace_size(B, Hq, D, bt.shape[1] * page_size, chunk),), torch.uint8, dev)
    go, gl = guarded((B, Hq, D), torch.bfloat16, dev), guarded((B, Hq), torch.float32, dev)
    o, lse = binding.attn_decode_paged(q.to(dev), kp.to(dev), vp.to(dev), bt.to(dev), sl.to(dev), gw.t, go.t, gl.t,
                                       chunk=chunk)
    check_guards(gw, go, gl)
    O, L = oracle.decode_forward_paged(q, kp, vp, bt, sl, 1 / math.sqrt(D))
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


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 8, 2), (128, 32, 2), (64, 8, 2), (128, 32, 1)])
def test_decode_nan_in_unused_cache_rows_does_not_leak(dev, D, Hq, Hkv):
    """Rows past a sequence's end may hold anything, NaN included (SIMT and tensor-core consumers)."""
    lens = [5, 700, 1]
    q, kc, vc, seqlens, ws, o, lse = run_decode(dev, 3, Hq, Hkv, lens, 1024, 512, seed=6, D=D, fill=float("nan"))
    O, L = oracle.decode_forward(q, kc, vc, lens, 1 / math.sqrt(D))
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


@pytest.mark.parametrize("G,chunk,D", [(1, 512, 128), (4, 512, 128), (8, 64, 128), (2, 1024, 128),
                                       (16, 512, 128), (32, 512, 128), (4, 512, 64), (32, 64, 64)])
def test_decode_fp8_small(dev, G, chunk, D):
    """fp8 E4M3 cache: ragged lengths around the chunk and tile sizes."""
    lens = [1, 63, 64, 511, 513, 1500, 2048]
    B = len(lens)
    Hkv = 2 if G < 32 else 1
    Hq = G * Hkv
    ks, vs = FP8_SCALES
    q, kc, vc, _ = inputs.decode_inputs(B, Hq, Hkv, D, 1, 2, seed=G + chunk, nk_max=2048, kv_dtype="e4m3")
    sl = torch.tensor(lens, dtype=torch.int32)
    # regenerate rows for the chosen lengths (the drawn lengths are ignored)
    for b, n in enumerate(lens):
        kb, vb = inputs.decode_kv_rows(G + chunk, b, n, Hkv, D, kv_dtype="e4m3")
        kc[b, :n], vc[b, :n] = kb, vb
    gw = guarded((binding.attn_decode_workspace_size(B, Hq, D, 2048, chunk),), torch.uint8, dev)
    go, gl = guarded((B, Hq, D), torch.bfloat16, dev), guarded((B, Hq), torch.float32, dev)
    o, lse = binding.attn_decode_fp8(q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), ks, vs, gw.t, go.t, gl.t,
                                     chunk=chunk)
    check_guards(gw, go, gl)
    O, L = oracle.decode_forward_fp8(q, kc.numpy(), vc.numpy(), ks, vs, lens, 1 / math.sqrt(D))
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
    gw = guarded((binding.attn_decode_workspace_size(B, Hq, 128, bt.shape[1] * page_size, chunk),), torch.uint8, dev)
    go, gl = guarded((B, Hq, 128), torch.bfloat16, dev), guarded((B, Hq), torch.float32, dev)
    o, lse = binding.attn_decode_paged_fp8(q.to(dev), kp.to(dev), vp.to(dev), bt.to(dev), sl.to(dev), ks, vs,
                                           gw.t, go.t, gl.t, chunk=chunk)
    check_guards(gw, go, gl)
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


def test_decode_fp8_query_magnitudes_outside_f16_range(dev):
    """The fp8 consumer runs its MMAs on f16 operands: each query head is scaled by a power of two
    into f16 range first.  A head with |q| up to about 1e5 (beyond f16's 65504), one near 1e-6
    (f16 subnormal range) and a zero head must still match the oracle."""
    lens = [700, 1500, 64]
    B, Hq, Hkv = 3, 8, 2
    q, kc, vc, _ = inputs.decode_inputs(B, Hq, Hkv, 128, 1, 2, seed=41, nk_max=2048, kv_dtype="e4m3")
    for b, n in enumerate(lens):
        kb, vb = inputs.decode_kv_rows(41, b, n, Hkv, 128, kv_dtype="e4m3")
        kc[b, :n], vc[b, :n] = kb, vb
    q = q.float()
    q[:, 1] *= 3e4                # |q| up to ~1e5, beyond f16's 65504; softmax close to one-hot
    q[:, 2] *= 1e-6
    q[:, 5] = 0.0
    q = q.to(torch.bfloat16)
    sl = torch.tensor(lens, dtype=torch.int32)
    o, lse = binding.attn_decode_fp8(q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), 1.0, 1.0)
    O, L = oracle.decode_forward_fp8(q, kc.numpy(), vc.numpy(), 1.0, 1.0, lens, 1 / math.sqrt(128))
    check(o, lse, O, L, BF16_O_TOL, BF16_LSE_REL, True)
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
    # Q scaled by 3 (scaled scores ~ N(0, 9)) against cap 5: in one launch some warps'
    # tiles stay within the polynomial range |score / cap| <= 1 and others leave it
    (1, 4, 4, 384, 1024, 128, False, 0, 5.0, "normal", 3.0),
    (1, 4, 2, 256, 2048, 64, False, 0, 50.0, None, 1.0),  # every tile on the polynomial path, D = 64
    (2, 4, 1, 640, 640, 128, True, 0, 2.0, "normal", 1.5),  # causal, cap 2: unmasked tiles on both paths
    # per-head Q scales 0.3 / 0.7 / 1.3 against cap 4: the largest |score / cap| of a warp's tile
    # is about 0.3 / 0.7 / 1.4, so warps of one launch take the short polynomial (|y| <= 0.5),
    # the long one (|y| <= 1) and the exponential identity
    (1, 8, 8, 512, 2048, 128, False, 0, 4.0, "normal", (0.3, 0.3, 0.7, 0.7, 1.3, 1.3, 1.3, 1.3)),
]


@pytest.mark.parametrize("case", SOFTCAP_CASES, ids=lambda c: "-".join(map(str, c)))
def test_softcap_sink(dev, case):
    B, Hq, Hkv, Nq, Nk, D, causal, window, cap, kind = case[:10]
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, D, "bf16", seed=Nq + Nk)
    if len(case) > 10:
        mul = torch.tensor(case[10], dtype=torch.float32).view(1, -1, 1, 1) if isinstance(case[10], tuple) \
            else case[10]
        q = (q.float() * mul).to(torch.bfloat16)
    sinks = _sinks(Hq, kind, Nq)
    go, gl = guarded(q.shape, torch.bfloat16, dev), guarded((B, Hq, Nq), torch.float32, dev)
    o, lse = binding.attn_fwd_softcap_sink(q.to(dev), k.to(dev), v.to(dev), go.t, gl.t, causal=causal,
                                           window=window, softcap=cap,
                                           sinks=None if sinks is None else sinks.to(dev))
    check_guards(go, gl)
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
    # B, Hq, Hkv, Nq, Nk, causal, window
    (1, 2, 2, 200, 200, False, 0),
    (2, 4, 2, 257, 257, True, 0),       # GQA, ragged tiles
    (1, 4, 1, 130, 300, True, 0),       # bottom-right causal, Nq < Nk
    (1, 2, 2, 300, 130, True, 0),       # Nq > Nk: rows 0..169 see no key
    (1, 2, 1, 64, 1000, False, 0),      # one query tile, many key tiles
    (1, 4, 2, 384, 384, True, 0),       # whole tiles only, two query heads per KV head
    (2, 2, 1, 5, 37, True, 0),          # fewer queries than one 32-row dQ box
    (1, 2, 2, 300, 300, True, 64),      # causal sliding window
    (1, 4, 2, 257, 257, False, 100),    # window without causal
    (1, 2, 1, 130, 700, True, 50),      # chunked prefill + window: key tiles no query sees (dK = dV = 0)
    (1, 2, 2, 512, 512, True, 128),     # window of exactly one tile, whole tiles
    (1, 4, 2, 300, 300, False, 0),      # key-tile pairs, odd tile count (a CTA past the last key)
    (2, 4, 2, 257, 520, False, 0),      # key-tile pairs, GQA, ragged query and key tiles
    # head dimension 64
    (1, 2, 1, 130, 300, False, 0, 64),  # key-tile pairs, odd tile count
    (1, 2, 2, 200, 200, False, 0, 64),
    (2, 4, 2, 257, 257, True, 0, 64),
    (1, 4, 1, 130, 300, True, 0, 64),
    (1, 2, 1, 130, 700, True, 50, 64),
    (1, 4, 2, 384, 384, True, 0, 64),
]


def _bwd_check(got, want, name):
    """Each gradient against 2 % of its tensor's largest magnitude (P, dS and O are
    rounded to bf16, relative 2^-9, before the fp32 sums)."""
    g = got.float().cpu().numpy()
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    err = float(np.abs(g - want).max())
    tol = 2e-2 * max(1.0, float(np.abs(want).max()))
    print(f"[achieved] backward {name}: max-abs err {err:.3e}, tol {tol:.3e}, max |grad| {np.abs(want).max():.3e}")
    assert err <= tol, f"{name}: max-abs err {err:.3e} (tol {tol:.3e})"
    return err


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "-".join(map(str, c)))
def test_backward(dev, case):
    B, Hq, Hkv, Nq, Nk, causal, window = case[:7]
    D = case[7] if len(case) > 7 else 128
    q, k, v = inputs.prefill_inputs(B, Hq, Hkv, Nq, Nk, D, "bf16", seed=Nq * 7 + Nk)
    g = torch.Generator("cpu").manual_seed(Nq + 3)
    do = torch.randn(B, Hq, Nq, D, generator=g).to(torch.bfloat16)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = binding.attn_fwd(qd, kd, vd, causal=causal, window=window)
    gq, gk, gv = (guarded(q.shape, torch.float32, dev), guarded(k.shape, torch.bfloat16, dev),
                  guarded(v.shape, torch.bfloat16, dev))
    gw = guarded((binding.lib().attn_bwd_workspace_size(B, Hq, Nq),), torch.uint8, dev)
    dq, dk, dv = binding.attn_bwd(qd, kd, vd, o, dod, lse, gq.t, gk.t, gv.t, gw.t, causal=causal, window=window)
    check_guards(gq, gk, gv, gw)
    dQ, dK, dV = oracle.attention_backward(q, k, v, do, 1 / math.sqrt(D), causal, window)
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
    def one(h):
        sl = slice(h, h + 1)
        return h, oracle.attention_backward(q[:, sl], k[:, sl], v[:, sl], do[:, sl], 1 / math.sqrt(D), False, 0)

    for h, (dQ, dK, dV) in parallel_map(one, (0, 17), threads=2):
        sl = slice(h, h + 1)
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
