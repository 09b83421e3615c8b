"""CPU oracle for the attention forward and split-KV decode (fp64, numpy).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` and by nothing else.  It shares no code with
the CUDA library and never imports it.
"""
from .attention import *  # noqa: F401,F403
