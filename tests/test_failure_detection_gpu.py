"""Failure detection on the GPU without a GPU fault.

Every wait in the kernels is bounded: when a barrier phase never completes, the
waiting thread gives up after the limit, records ATTN_ERR_TIMEOUT in the device
error word and raises its CTA's abort flag so that the other roles stop waiting
too.  This test makes such a wait run out on purpose (a barrier that nothing
arrives on) and checks the status and that the CUDA context stays usable.
"""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "cuda", "wait_timeout_probe.cu")


@pytest.fixture(scope="module")
def probe(cuda_lib):
    from softmax_attention_attn_gb300 import build
    out_dir = os.path.join(ROOT, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libwait_timeout_probe.so")
    subprocess.run([build.nvcc_path(), *build.NVCC_FLAGS, "-shared", SRC, "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.wait_timeout_probe.argtypes = [ctypes.c_void_p] * 3
    lib.wait_timeout_probe.restype = ctypes.c_int
    return lib


def test_bounded_wait_times_out_and_reports(probe):
    dev = torch.device("cuda:0")
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    result = torch.full((2,), 7, dtype=torch.int32, device=dev)
    elapsed = torch.zeros(2, dtype=torch.int64, device=dev)
    assert probe.wait_timeout_probe(ctypes.c_void_p(err.data_ptr()), ctypes.c_void_p(result.data_ptr()),
                                    ctypes.c_void_p(elapsed.data_ptr())) == 0
    assert int(err.item()) == -8                      # ATTN_ERR_TIMEOUT
    assert result.tolist() == [0, 0]                  # both waiters gave up
    ns = elapsed.cpu().tolist()
    assert max(ns) >= 1.9e9 and max(ns) < 30e9       # the 2 s limit, not a hang
    # the context is still usable: a real forward call after the probe works
    from softmax_attention_attn_gb300 import binding, inputs
    q, k, v = (x.to(dev) for x in inputs.prefill_inputs(1, 2, 2, 256, 256, 128, "bf16", 3))
    o, lse = binding.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all().item()
    assert binding.get_device_error() == 0
