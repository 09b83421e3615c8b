"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path (through the tests and the benchmark)
and the CPU oracle consume what it returns, so the two sides always see the
same values.

Recipe (every draw uses ``torch.Generator("cpu")``):

* prefill workloads: one generator seeded with ``seed`` draws fp32 N(0, 1)
  tensors in the order Q ``[B,Hq,Nq,D]``, K ``[B,Hkv,Nk,D]``, V ``[B,Hkv,Nk,D]``;
  bf16 / fp16 workloads cast those fp32 values with round-to-nearest-even.
* fp8 prefill workloads (``prefill_inputs_fp8``): the same fp32 draws rounded
  to the nearest OCP FP8 E4M3 value (torch's float8_e4m3fn conversion) and
  stored as uint8 codes; the per-tensor scales are the caller's.
* decode workloads: a generator seeded with ``seed`` draws the per-sequence
  key counts ``Nk_b ~ U{nk_lo..nk_hi}`` first and then Q ``[B,Hq,D]``.  Sequence
  ``b`` then draws its own K and V rows ``[Nk_b,Hkv,D]`` (K first) from a
  generator seeded with ``decode_row_seed(seed, b)``, so any single sequence can
  be regenerated without replaying the others.  Cache rows at or beyond
  ``Nk_b`` hold finite sentinels (K = 64, V = 1e4) so that a masking leak
  shows up as a large error instead of passing unnoticed.
* an fp8 KV cache (``kv_dtype="e4m3"``) holds the same fp32 draws rounded to
  the nearest OCP FP8 E4M3 value (torch's float8_e4m3fn conversion), stored as
  uint8 codes; the tail sentinels are K = 64 and V = 448 (the largest finite
  E4M3 value).  The value of a code is set by the caller's per-tensor scale.
* large decode workloads may draw each sequence's K/V rows on a CUDA device
  instead (``device=...``): same per-sequence seeds and distribution, but a
  CUDA generator, so the values differ from the CPU draw; a check against the
  oracle then copies the sampled sequences' rows back from that device.
"""
from __future__ import annotations

import torch

K_SENTINEL = 64.0
V_SENTINEL = 1.0e4
V_SENTINEL_FP8 = 448.0

_KV_CODES = {"e4m3": torch.float8_e4m3fn}

_DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16}


def _cast(t: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype not in _DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    return t if dtype == "fp32" else t.to(_DTYPES[dtype])


def prefill_inputs(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, D: int,
                   dtype: str = "bf16", seed: int = 0):
    """Q, K, V for one prefill workload, contiguous ``[B,H,N,D]`` CPU tensors."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, Hq, Nq, D, generator=g, dtype=torch.float32)
    k = torch.randn(B, Hkv, Nk, D, generator=g, dtype=torch.float32)
    v = torch.randn(B, Hkv, Nk, D, generator=g, dtype=torch.float32)
    return _cast(q, dtype), _cast(k, dtype), _cast(v, dtype)


def prefill_inputs_fp8(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, D: int, seed: int = 0,
                       fmt: str = "e4m3"):
    """The fp32 draws of :func:`prefill_inputs` rounded to the nearest value of the
    fp8 format ``fmt`` and returned as its uint8 codes (Q, K, V)."""
    q, k, v = prefill_inputs(B, Hq, Hkv, Nq, Nk, D, "fp32", seed)
    return _codes(q, fmt), _codes(k, fmt), _codes(v, fmt)


def varlen_inputs(lens_q, lens_k, Hq: int, Hkv: int, D: int, dtype: str = "bf16", seed: int = 0):
    """Ragged batch, packed token-major: ``(q [Tq,Hq,D], k [Tk,Hkv,D], v, cu_q, cu_k)``.

    One generator seeded with ``seed`` draws fp32 N(0, 1) Q, then K, then V for
    the whole packed batch; ``cu_q`` / ``cu_k`` are int32 prefix sums of the lengths.
    """
    g = torch.Generator("cpu").manual_seed(seed)
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    q = torch.randn(tq, Hq, D, generator=g, dtype=torch.float32)
    k = torch.randn(tk, Hkv, D, generator=g, dtype=torch.float32)
    v = torch.randn(tk, Hkv, D, generator=g, dtype=torch.float32)
    cu = lambda lens: torch.tensor([0] + list(torch.cumsum(torch.tensor(lens), 0).tolist()), dtype=torch.int32)  # noqa: E731
    return _cast(q, dtype), _cast(k, dtype), _cast(v, dtype), cu(lens_q), cu(lens_k)


def decode_row_seed(seed: int, b: int) -> int:
    """Seed of the generator that draws sequence ``b``'s K/V rows."""
    return seed * 1_000_003 + 1 + b


def decode_seqlens_and_q(B: int, Hq: int, D: int, nk_lo: int, nk_hi: int,
                         seed: int = 0, dtype: str = "bf16"):
    """Per-sequence key counts (int32 ``[B]``) and the query ``[B,Hq,D]``."""
    g = torch.Generator("cpu").manual_seed(seed)
    seqlens = torch.randint(nk_lo, nk_hi + 1, (B,), generator=g, dtype=torch.int64)
    q = torch.randn(B, Hq, D, generator=g, dtype=torch.float32)
    return seqlens.to(torch.int32), _cast(q, dtype)


def _codes(t: torch.Tensor, kv_dtype: str) -> torch.Tensor:
    """fp32 values -> uint8 codes of the fp8 format ``kv_dtype`` (nearest value)."""
    if kv_dtype not in _KV_CODES:
        raise ValueError(f"unknown fp8 cache type {kv_dtype!r}")
    return t.to(_KV_CODES[kv_dtype]).view(torch.uint8)


def decode_kv_rows(seed: int, b: int, nk: int, Hkv: int, D: int, dtype: str = "bf16",
                   device="cpu", kv_dtype: str | None = None):
    """The ``nk`` valid K and V rows ``[nk,Hkv,D]`` of sequence ``b`` (fp8 codes
    when ``kv_dtype`` names an fp8 format)."""
    g = torch.Generator(device).manual_seed(decode_row_seed(seed, b))
    k = torch.randn(nk, Hkv, D, generator=g, dtype=torch.float32, device=device)
    v = torch.randn(nk, Hkv, D, generator=g, dtype=torch.float32, device=device)
    if kv_dtype is not None:
        return _codes(k, kv_dtype), _codes(v, kv_dtype)
    return _cast(k, dtype), _cast(v, dtype)


def _sentinels(kv_dtype: str | None):
    """(K, V) tail fill: values, or fp8 codes of K = 64 and V = 448."""
    if kv_dtype is None:
        return K_SENTINEL, V_SENTINEL
    return (int(_codes(torch.tensor([K_SENTINEL]), kv_dtype)[0]),
            int(_codes(torch.tensor([V_SENTINEL_FP8]), kv_dtype)[0]))


def decode_inputs(B: int, Hq: int, Hkv: int, D: int, nk_lo: int, nk_hi: int,
                  seed: int = 0, nk_max: int | None = None, dtype: str = "bf16",
                  pin_memory: bool = False, device="cpu", kv_dtype: str | None = None):
    """Full decode workload: ``(q, k_cache, v_cache, seqlens)``.

    ``k_cache``/``v_cache`` are ``[B,Nk_max,Hkv,D]`` with ``Nk_max`` defaulting to
    ``nk_hi``; rows past each sequence's length hold the sentinels.  With a
    CUDA ``device`` the caches are drawn and returned on that device (``q`` and
    ``seqlens`` are always drawn on the CPU and returned there).
    """
    seqlens, q = decode_seqlens_and_q(B, Hq, D, nk_lo, nk_hi, seed, dtype)
    nk_max = nk_hi if nk_max is None else nk_max
    if int(seqlens.max()) > nk_max:
        raise ValueError("nk_max is below a drawn sequence length")
    tdt = _DTYPES[dtype] if kv_dtype is None else torch.uint8
    on_cpu = torch.device(device).type == "cpu"
    k_cache = torch.empty(B, nk_max, Hkv, D, dtype=tdt, device=device, pin_memory=pin_memory and on_cpu)
    v_cache = torch.empty(B, nk_max, Hkv, D, dtype=tdt, device=device, pin_memory=pin_memory and on_cpu)
    k_fill, v_fill = _sentinels(kv_dtype)
    for b in range(B):
        nk = int(seqlens[b])
        kb, vb = decode_kv_rows(seed, b, nk, Hkv, D, dtype, device, kv_dtype)
        k_cache[b, :nk] = kb
        v_cache[b, :nk] = vb
        k_cache[b, nk:] = k_fill
        v_cache[b, nk:] = v_fill
    return q, k_cache, v_cache, seqlens


def paged_decode_inputs(B: int, Hq: int, Hkv: int, D: int, nk_lo: int, nk_hi: int,
                        page_size: int, seed: int = 0, dtype: str = "bf16", device="cpu",
                        spare_pages: int = 0, kv_dtype: str | None = None):
    """Paged decode workload: ``(q, k_pages, v_pages, block_table, seqlens)``.

    Sequence lengths, Q and every sequence's K/V rows are the draws of
    :func:`decode_inputs` (same seed, same device rule).  The pages a sequence
    needs are placed at page ids given by a permutation drawn from a generator
    seeded ``seed + 7`` (so sequences are scattered over the pool); the tail of
    a last page holds the sentinels, ``spare_pages`` unused pages are added to
    the pool, and unused block-table entries are 0.
    """
    seqlens, q = decode_seqlens_and_q(B, Hq, D, nk_lo, nk_hi, seed, dtype)
    lens = [int(x) for x in seqlens]
    max_pages = -(-nk_hi // page_size)
    need = [-(-n // page_size) for n in lens]
    num_pages = sum(need) + spare_pages
    perm = torch.randperm(num_pages, generator=torch.Generator("cpu").manual_seed(seed + 7))
    block_table = torch.zeros(B, max_pages, dtype=torch.int32)
    tdt = _DTYPES[dtype] if kv_dtype is None else torch.uint8
    k_fill, v_fill = _sentinels(kv_dtype)
    k_pages = torch.full((num_pages, page_size, Hkv, D), k_fill, dtype=tdt, device=device)
    v_pages = torch.full((num_pages, page_size, Hkv, D), v_fill, dtype=tdt, device=device)
    nxt = 0
    for b in range(B):
        kb, vb = decode_kv_rows(seed, b, lens[b], Hkv, D, dtype, device, kv_dtype)
        for i in range(need[b]):
            page = int(perm[nxt])
            nxt += 1
            block_table[b, i] = page
            rows = min(page_size, lens[b] - i * page_size)
            k_pages[page, :rows] = kb[i * page_size: i * page_size + rows]
            v_pages[page, :rows] = vb[i * page_size: i * page_size + rows]
    return q, k_pages, v_pages, block_table, seqlens
