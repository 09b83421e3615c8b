"""GB300 (sm_103a) fused softmax-attention forward: bf16 tcgen05 prefill, fp32
SIMT prefill and split-KV decode, exposed through a C ABI (``include/attn.h``)
and the thin ctypes binding in :mod:`.binding`.

Submodules are imported lazily so that the seeded input generators
(:mod:`.inputs`) can be used without loading the CUDA library.
"""
import importlib

__all__ = ["binding", "inputs", "build", "attn_fwd", "attn_fwd_fp32", "attn_decode",
           "attn_decode_splitkv", "attn_decode_combine", "attn_decode_workspace_size",
           "get_device_error", "AttnError"]

_BINDING_NAMES = {"attn_fwd", "attn_fwd_fp32", "attn_decode", "attn_decode_splitkv",
                  "attn_decode_combine", "attn_decode_workspace_size", "get_device_error",
                  "AttnError"}


def __getattr__(name):
    if name in ("binding", "inputs", "build"):
        return importlib.import_module(f".{name}", __name__)
    if name in _BINDING_NAMES:
        return getattr(importlib.import_module(".binding", __name__), name)
    raise AttributeError(name)
