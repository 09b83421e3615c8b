"""GPU test of attn_decode_noalloc, the decode entry point that allocates nothing.

It is meant for callers that cannot allocate device memory (for example a
plugin inside a host runtime that owns the device memory pool), so it keeps its
per-chunk partials in a scratch array inside the library instead of a
caller-provided workspace.  Two calls in a row, with different inputs and
sizes, must match the fp64 oracle's decode and the workspace-based entry points
(attn_decode_splitkv + attn_decode_combine) within the bf16 tolerances of the
other parity tests; a call without an LSE output must give the same O; a size
beyond the scratch capacity must be rejected on the host.

This file is named so that pytest collects it last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from softmax_attention_attn_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

BF16_O_TOL = 2e-2
BF16_LSE_REL = 1e-2
HQ, HKV, D, CHUNK = 32, 8, 128, 512


def make_case(seed, lens, nk_max, dev):
    B = len(lens)
    _, q = inputs.decode_seqlens_and_q(B, HQ, D, 1, 2, seed)
    kc = torch.full((B, nk_max, HKV, D), inputs.K_SENTINEL, dtype=torch.bfloat16)
    vc = torch.full((B, nk_max, HKV, D), inputs.V_SENTINEL, dtype=torch.bfloat16)
    for b, n in enumerate(lens):
        kb, vb = inputs.decode_kv_rows(seed, b, n, HKV, D)
        kc[b, :n], vc[b, :n] = kb, vb
    return q.to(dev), kc.to(dev), vc.to(dev), torch.tensor(lens, dtype=torch.int32, device=dev)


def call_noalloc(L, q, kc, vc, sl, o, lse, B, nk_max):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.attn_decode_noalloc(p(q), p(kc), p(vc), p(sl), p(o), p(lse), B, HQ, HKV, nk_max, D,
                                 1 / math.sqrt(D), CHUNK, stream)


def _close(o, lse, ref_o, ref_lse):
    """max-abs O error and relative LSE error (|dLSE| / max(1, |LSE|)) against a reference."""
    err_o = float(np.abs(o - ref_o).max())
    err_l = 0.0 if lse is None else float((np.abs(lse - ref_lse) / np.maximum(1.0, np.abs(ref_lse))).max())
    return err_o, err_l


def test_noalloc_matches_workspace_entry_points(cuda_lib):
    dev = torch.device("cuda:0")
    L = binding.lib()
    cases = [(31, [1, 700, 4096, 2049, 512, 3000], 4096),   # first call on the device
             (32, [8192, 5, 1537, 2500], 8192)]              # second call: new inputs and sizes
    for seed, lens, nk_max in cases:
        B = len(lens)
        assert binding.attn_decode_workspace_size(B, HQ, D, nk_max, CHUNK) <= 16 << 20
        q, kc, vc, sl = make_case(seed, lens, nk_max, dev)
        ref_o, ref_lse = binding.attn_decode(q, kc, vc, sl, chunk=CHUNK)
        o = torch.full((B, HQ, D), float("nan"), device=dev, dtype=torch.bfloat16)
        lse = torch.full((B, HQ), float("nan"), device=dev, dtype=torch.float32)
        assert call_noalloc(L, q, kc, vc, sl, o, lse, B, nk_max) == 0
        torch.cuda.synchronize()
        assert binding.get_device_error() == 0
        oo, ro = o.float().cpu().numpy(), ref_o.float().cpu().numpy()
        ll, rl = lse.cpu().numpy(), ref_lse.cpu().numpy()
        assert np.isfinite(oo).all() and np.isfinite(ll).all()
        # against the workspace-based entry points
        err_o, err_l = _close(oo, ll, ro, rl)
        assert err_o <= BF16_O_TOL and err_l <= BF16_LSE_REL, (err_o, err_l)
        # against the fp64 oracle on the same inputs
        O, Lse = oracle.decode_forward(q.cpu(), kc.cpu(), vc.cpu(), lens, 1 / math.sqrt(D))
        err_o, err_l = _close(oo, ll, O, Lse)
        assert err_o <= BF16_O_TOL and err_l <= BF16_LSE_REL, (err_o, err_l)
        # the LSE output is optional: without it, O is unchanged
        o2 = torch.full((B, HQ, D), float("nan"), device=dev, dtype=torch.bfloat16)
        assert call_noalloc(L, q, kc, vc, sl, o2, None, B, nk_max) == 0
        torch.cuda.synchronize()
        assert binding.get_device_error() == 0
        assert torch.equal(o2, o)


def test_noalloc_rejects_sizes_beyond_capacity(cuda_lib):
    dev = torch.device("cuda:0")
    L = binding.lib()
    q, kc, vc, sl = make_case(33, [64], 64, dev)
    o = torch.empty(1, HQ, D, device=dev, dtype=torch.bfloat16)
    lse = torch.empty(1, HQ, device=dev, dtype=torch.float32)
    # B=64, Nk_max=32768 needs 67.6 MB of partials: more than the 16 MiB scratch
    assert call_noalloc(L, q, kc, vc, sl, o, lse, 64, 32768) == -12   # ATTN_ERR_CAPACITY
    assert binding.get_device_error() == 0
