"""Host-side checks of the C ABI (CPU only, no kernel launches).

The library must load without a GPU, export every entry point that
``include/attn.h`` declares, and reject bad arguments on the host before it
makes any CUDA call.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def L():
    from softmax_attention_attn_gb300 import binding, build
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("attn_fwd", "attn_fwd_fp16", "attn_fwd_fp32", "attn_decode_splitkv", "attn_decode_combine",
                 "attn_decode_splitkv_fp8", "attn_decode_splitkv_paged_fp8", "attn_fwd_fp8",
                 "attn_decode_workspace_size", "attn_get_device_error", "attn_strerror"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    from softmax_attention_attn_gb300 import binding
    names = declared_functions()
    for n in names:
        assert hasattr(L, n), f"{n} not exported"
    assert set(names) <= set(binding.SIGNATURES), "binding lacks a signature"


def test_no_library_gemm_symbols():
    """The library links no cuBLAS / cuDNN / CUTLASS code."""
    from softmax_attention_attn_gb300 import build
    path = build.build()
    import subprocess
    out = subprocess.run(["nm", "-D", path], capture_output=True, text=True).stdout
    assert not re.search(r"cublas|cudnn|cutlass", out, re.I)


def test_strerror_and_status_codes(L):
    from softmax_attention_attn_gb300 import binding
    text = open(HEADER).read()
    codes = {name: int(val) for name, val in re.findall(r"(ATTN_(?:OK|ERR_[A-Z_0-9]+))\s*=\s*(-?\d+)", text)}
    assert codes == {v: k for k, v in binding.STATUS.items()}
    for code in codes.values():
        assert L.attn_strerror(code) and L.attn_strerror(code) != b"unknown status code"
    assert L.attn_strerror(12345) == b"unknown status code"


P = ctypes.c_void_p(256)     # a 16-byte aligned non-null dummy: never dereferenced
MIS = ctypes.c_void_p(258)   # misaligned dummy


def fwd(L, name="attn_fwd", q=P, k=P, v=P, o=P, lse=P, B=1, Hq=4, Hkv=2, Nq=8, Nk=8, D=128,
        scale=0.1, causal=0, window=0):
    return getattr(L, name)(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window, None)


@pytest.mark.parametrize("name", ["attn_fwd", "attn_fwd_fp16", "attn_fwd_fp32"])
def test_forward_argument_errors(L, name):
    assert fwd(L, name, q=None) == -1
    assert fwd(L, name, o=None) == -1
    assert fwd(L, name, B=0) == -2
    assert fwd(L, name, Nk=-3) == -2
    assert fwd(L, name, B=70000) == -2
    assert fwd(L, name, Hq=6, Hkv=4) == -3
    assert fwd(L, name, D=96) == -4
    assert fwd(L, name, k=MIS) == -5
    assert fwd(L, name, lse=MIS) == -5
    assert fwd(L, name, scale=0.0) == -6
    assert fwd(L, name, scale=float("nan")) == -6
    assert fwd(L, name, scale=float("inf")) == -6


def test_head_dim_per_entry_point(L):
    assert fwd(L, "attn_fwd", D=32) == -4
    assert fwd(L, "attn_fwd_fp16", D=256) == -4
    assert fwd(L, "attn_fwd_fp32", D=256) == -4


def test_decode_argument_errors(L):
    def split(q=P, kc=P, vc=P, sl=P, ws=P, B=4, Hq=32, Hkv=8, Nk_max=1024, D=128, scale=0.1, chunk=512):
        return L.attn_decode_splitkv(q, kc, vc, sl, ws, B, Hq, Hkv, Nk_max, D, scale, chunk, None)

    assert split(sl=None) == -1
    assert split(ws=None) == -1
    assert split(B=0) == -2
    assert split(Hq=12, Hkv=8) == -3
    assert split(Hq=64, Hkv=1) == -3          # group of 64 not supported
    assert split(Hq=24, Hkv=2) == -3          # group of 12 not supported
    assert split(D=96) == -4
    assert split(D=256) == -4
    assert split(chunk=500) == -11
    assert split(chunk=2048) == -11
    assert split(B=5000) == -12
    assert split(kc=MIS) == -5
    assert split(scale=-1.0) == -6

    def comb(ws=P, sl=P, o=P, lse=P, B=4, Hq=32, Nk_max=1024, D=128, chunk=512):
        return L.attn_decode_combine(ws, sl, o, lse, B, Hq, Nk_max, D, chunk, None)

    assert comb(o=None) == -1
    assert comb(chunk=100) == -11
    assert comb(D=256) == -4
    assert comb(lse=MIS) == -5


def test_paged_decode_argument_errors(L):
    def paged(q=P, kp=P, vp=P, bt=P, sl=P, ws=P, B=4, Hq=32, Hkv=8, num_pages=100, page_size=256,
              max_pages=8, D=128, scale=0.1, chunk=512):
        return L.attn_decode_splitkv_paged(q, kp, vp, bt, sl, ws, B, Hq, Hkv, num_pages, page_size,
                                           max_pages, D, scale, chunk, None)

    assert paged(bt=None) == -1
    assert paged(page_size=100) == -2          # not a multiple of 64
    assert paged(page_size=0) == -2
    assert paged(num_pages=0) == -2
    assert paged(max_pages=-1) == -2
    assert paged(Hq=32, Hkv=3) == -3
    assert paged(D=32) == -4
    assert paged(chunk=96) == -11
    assert paged(bt=MIS) == -5
    assert paged(scale=0.0) == -6


def test_fp8_decode_argument_errors(L):
    def fp8(q=P, kc=P, vc=P, ks=0.5, vs=2.0, sl=P, ws=P, B=4, Hq=32, Hkv=8, Nk=1024, D=128, scale=0.1,
            chunk=512):
        return L.attn_decode_splitkv_fp8(q, kc, vc, ks, vs, sl, ws, B, Hq, Hkv, Nk, D, scale, chunk, None)

    def paged8(q=P, kp=P, vp=P, ks=0.5, vs=2.0, bt=P, sl=P, ws=P, B=4, Hq=32, Hkv=8, num_pages=100,
               page_size=256, max_pages=8, D=128, scale=0.1, chunk=512):
        return L.attn_decode_splitkv_paged_fp8(q, kp, vp, ks, vs, bt, sl, ws, B, Hq, Hkv, num_pages,
                                               page_size, max_pages, D, scale, chunk, None)

    for f in (fp8, paged8):
        assert f(q=None) == -1
        assert f(Hq=32, Hkv=3) == -3
        assert f(D=256) == -4
        assert f(chunk=96) == -11
        assert f(sl=MIS) == -5
        assert f(scale=0.0) == -6
        assert f(ks=0.0) == -6
        assert f(vs=-1.0) == -6
        assert f(ks=float("nan")) == -6
        assert f(vs=float("inf")) == -6
    assert paged8(bt=None) == -1
    assert paged8(page_size=100) == -2


def test_softcap_sink_argument_errors(L):
    def f(q=P, k=P, v=P, o=P, lse=P, B=2, Hq=8, Hkv=2, Nq=128, Nk=128, D=128, scale=0.1, causal=0,
          window=0, cap=30.0, sinks=P):
        return L.attn_fwd_softcap_sink(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, D, scale, causal, window, cap,
                                       sinks, None)

    assert f(q=None) == -1
    assert f(D=96) == -4
    assert f(Hq=8, Hkv=3) == -3
    assert f(scale=0.0) == -6
    assert f(cap=float("nan")) == -6
    assert f(cap=float("inf")) == -6
    assert f(sinks=ctypes.c_void_p(258)) == -5   # not 4-byte aligned


def test_fp8_forward_argument_errors(L):
    def f(q=P, k=P, v=P, qs=1.0, ks=1.0, vs=1.0, o=P, lse=P, ws=P, B=1, Hq=4, Hkv=2, Nq=8, Nk=8, D=128,
          scale=0.1, causal=0, window=0):
        return L.attn_fwd_fp8(q, k, v, qs, ks, vs, o, lse, ws, B, Hq, Hkv, Nq, Nk, D, scale, causal, window,
                              None)

    assert f(v=None) == -1
    assert f(ws=None) == -1
    assert f(Nq=0) == -2
    assert f(Hq=6, Hkv=4) == -3
    assert f(D=64) == -4
    assert f(D=256) == -4
    assert f(ws=MIS) == -5
    assert f(q=MIS) == -5
    assert f(qs=0.0) == -6
    assert f(ks=float("nan")) == -6
    assert f(vs=-1.0) == -6
    assert f(vs=float("inf")) == -6
    assert f(scale=1e-30, qs=1e-10, ks=1e-10) == -6      # product underflows to 0
    assert f(scale=1e30, qs=1e10, ks=1e10) == -6         # product overflows
    assert L.attn_fwd_fp8_workspace_size(2, 8, 1000, 128) == 2 * 8 * 1000 * 128 * 2
    assert L.attn_fwd_fp8_workspace_size(0, 8, 1000, 128) == 0


def test_backward_argument_errors(L):
    def f(q=P, k=P, v=P, o=P, do=P, lse=P, dq=P, dk=P, dv=P, ws=P, B=2, Hq=8, Hkv=2, Nq=128, Nk=128, D=128,
          scale=0.1, causal=0):
        return L.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, B, Hq, Hkv, Nq, Nk, D, scale, causal, 0, None)

    assert f(do=None) == -1
    assert f(ws=None) == -1
    assert f(Nq=0) == -2
    assert f(Hq=8, Hkv=3) == -3
    assert f(D=96) == -4
    assert f(D=256) == -4
    assert f(dq=MIS) == -5
    assert f(scale=-1.0) == -6
    assert L.attn_bwd_workspace_size(2, 8, 100) == 2 * 2 * 8 * 128 * 4
    assert L.attn_bwd_workspace_size(1, 3, 130) == 2 * 1 * 3 * 256 * 4   # 128 rows per head


def test_workspace_size(L):
    # O_part [B,Hq,S_max,D] + LSE_part [B,Hq,S_max], fp32, rounded up to 256 bytes
    n = L.attn_decode_workspace_size(64, 32, 128, 32768, 512)
    assert n == 64 * 32 * 64 * 129 * 4
    assert L.attn_decode_workspace_size(1, 1, 128, 100, 64) == (2 * 129 * 4 + 255) // 256 * 256
    assert L.attn_decode_workspace_size(0, 1, 128, 100, 64) == 0
