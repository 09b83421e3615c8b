"""fp64 CPU oracle for the fused attention forward and split-KV decode.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The library's product
path never calls it and shares no code with it.

What it computes is the plain definition, written out step by step so that it
can be checked by eye:

    S = scale * Q K^T  (masked entries = -inf)
    P = softmax(S) along the key axis     (two passes: row max, then exp / sum)
    O = P V,   LSE = ln sum_j exp(S_ij)

Sources (pages on softmax attention):

* "Agent 帮我写 CUDA：一个 Softmax Attention 算子的开发全记录" (a fp32 softmax-attention
  CUDA development log), section 二 "参考基线": the operator is
  softmax(Q K^T / sqrt(D)) V on ``[B,H,N,D]`` tensors, checked against
  ``scaled_dot_product_attention``.  Section 四 "Tiled Attention 的核心思想" gives
  the online-softmax recurrence; online softmax reaches exactly the two-pass
  result below (up to rounding order), so the oracle uses the two-pass form.
* "Ask, Don't Equip: Question-Driven Coding Agents for Deep Kernel Optimization",
  section "研究动机": the feature surface (GQA, causal and sliding-window masks,
  split-KV decode).  It gives no formulas; the readings used here are:
    - GQA: query head h reads KV head ``h // (Hq // Hkv)``;
    - causal is bottom-right aligned: key j is visible to query i iff
      ``j <= i + Nk - Nq``;
    - a window w > 0 keeps the last w keys up to and including the diagonal:
      ``j > i + Nk - Nq - w``;
    - a row with no visible key has O = 0 and LSE = -inf;
    - LSE is the natural log of the softmax denominator of the scaled scores;
    - split-KV decode cuts each sequence's keys into chunks of ``chunk`` keys
      starting at key 0 (the last chunk may be short); each chunk yields its own
      normalised output and LSE, and the combine step weights chunk c by
      ``exp(LSE_c - max_c LSE_c)``;
    - a paged KV cache (paged and contiguous caches are both on the list) holds
      pages of ``page_size`` token rows ``[num_pages, page_size, Hkv, D]``; a
      block table ``[B, max_pages]`` names, for sequence b, the page of its
      logical page i, so key j of sequence b is row ``j % page_size`` of page
      ``block_table[b, j // page_size]``.
    - the backward pass (named as missing work, "then the backward pass"): the
      gradients of O with respect to Q, K and V for an upstream gradient dO,
      by the chain rule through S = scale Q K^T (masked entries constant),
      P = softmax(S) and O = P V; a KV head's K and V gradients sum over the
      query heads that read it;
    - softcap and attention sinks (both on the list of masks, after vLLM's
      feature surface, which the same section names): with a cap c > 0 each
      scaled score becomes ``c * tanh(s / c)`` (masked scores stay -inf); a
      sink is one logit per query head, ``sink[h]``, that joins the softmax
      denominator of every row of head h but carries no value:
      ``P_ij = exp(s_ij) / (sum_j exp(s_ij) + exp(sink[h]))``,
      ``LSE_i = ln(sum_j exp(s_ij) + exp(sink[h]))``; a row with no visible key
      then has O = 0 and LSE = sink[h];
    - an fp8 KV cache (fp8 e4m3 is on the list of data types) stores each K and
      V element as one OCP FP8 E4M3 code; the value is the code's E4M3 value
      times a per-tensor scale (``k_scale`` for K, ``v_scale`` for V).  E4M3:
      bit 7 sign, bits 6-3 exponent (bias 7), bits 2-0 mantissa; exponent 0
      encodes the subnormals ``m/8 * 2^-6``; exponent 15 with mantissa 7 is NaN;
      there are no infinities.
    - fp8 e4m3 Q, K and V (the "fp8 dense prefill" scenario that the same page's
      section "局限与改进" lists among the weakest, and its section "未来方向" among
      the work still open): each tensor holds E4M3 codes with its own per-tensor
      scale (``q_scale``, ``k_scale``, ``v_scale``); the values are code times
      scale and everything else is the plain forward.

Every pin of this module lives in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "visible_mask", "kv_head", "attention_forward", "attention_rows",
    "attention_probabilities", "decode_forward", "decode_split_partials",
    "decode_combine", "paged_rows", "decode_forward_paged", "attention_varlen",
    "e4m3_to_float", "decode_forward_fp8", "decode_forward_paged_fp8",
    "softcap_scores", "attention_forward_ext", "attention_rows_ext",
    "attention_backward", "attention_forward_fp8", "attention_rows_fp8",
]


def _f64(x) -> np.ndarray:
    """Exact fp64 copy of a tensor or array (bf16 and fp32 values are exact in fp64)."""
    if hasattr(x, "detach"):                      # torch tensor, bf16 included
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def kv_head(h: int, Hq: int, Hkv: int) -> int:
    """KV head read by query head ``h`` (GQA groups of consecutive query heads)."""
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (Hq // Hkv)


def visible_mask(rows: np.ndarray, Nq: int, Nk: int, causal: bool, window: int) -> np.ndarray:
    """Boolean ``[len(rows), Nk]``: True where key j is visible to query row i."""
    i = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(Nk, dtype=np.int64)[None, :]
    diag = i + (Nk - Nq)                   # bottom-right aligned diagonal
    vis = np.ones((i.shape[0], Nk), dtype=bool)
    if causal:
        vis &= j <= diag
    if window > 0:
        vis &= j > diag - window
    return vis


def _softmax_rows(S: np.ndarray):
    """Two-pass row softmax of a masked score block.

    Returns ``(P, lse)``.  Fully masked rows give P = 0 and lse = -inf.
    """
    M = S.max(axis=1)                                  # pass 1: row max
    empty = ~np.isfinite(M)                            # every key masked
    M_safe = np.where(empty, 0.0, M)
    E = np.exp(S - M_safe[:, None])                    # pass 2: exp (masked -> 0)
    l = E.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, l)[:, None])
        lse = np.where(empty, -np.inf, M_safe + np.log(np.where(empty, 1.0, l)))
    return P, lse


def _scores(q_rows: np.ndarray, k_head: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q_rows K^T, shape ``[rows, Nk]``."""
    return scale * (q_rows @ k_head.T)


def attention_forward(q, k, v, scale: float, causal: bool = False, window: int = 0,
                      row_block: int = 512):
    """Full forward: ``O [B,Hq,Nq,D]`` and ``LSE [B,Hq,Nq]`` in fp64.

    ``q``: ``[B,Hq,Nq,D]``; ``k``, ``v``: ``[B,Hkv,Nk,D]``.  S is formed
    explicitly for ``row_block`` query rows at a time.
    """
    Q, K, V = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, D = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    O = np.zeros((B, Hq, Nq, V.shape[3]))
    LSE = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            kh = kv_head(h, Hq, Hkv)
            for i0 in range(0, Nq, row_block):
                rows = np.arange(i0, min(i0 + row_block, Nq))
                S = _scores(Q[b, h, rows], K[b, kh], scale)
                S[~visible_mask(rows, Nq, Nk, causal, window)] = -np.inf
                P, lse = _softmax_rows(S)
                O[b, h, rows] = P @ V[b, kh]
                LSE[b, h, rows] = lse
    return O, LSE


def attention_rows(q, k, v, scale: float, rows, causal: bool = False, window: int = 0):
    """O and LSE of selected query rows only.

    ``rows`` is a sequence of ``(b, h, i)``; returns ``O [len(rows), D]`` and
    ``LSE [len(rows)]``.  Same definition as :func:`attention_forward`, one row at
    a time, for checking large workloads on sampled outputs.
    """
    B, Hq, Nq, _ = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    O = np.zeros((len(rows), v.shape[3]))
    LSE = np.zeros(len(rows))
    for n, (b, h, i) in enumerate(rows):
        kh = kv_head(h, Hq, Hkv)
        qi = _f64(q[b, h, i])[None, :]
        Kh, Vh = _f64(k[b, kh]), _f64(v[b, kh])
        S = _scores(qi, Kh, scale)
        S[~visible_mask(np.array([i]), Nq, Nk, causal, window)] = -np.inf
        P, lse = _softmax_rows(S)
        O[n] = (P @ Vh)[0]
        LSE[n] = lse[0]
    return O, LSE


def attention_probabilities(q, k, scale: float, causal: bool = False, window: int = 0):
    """The full probability matrix ``P [B,Hq,Nq,Nk]`` (small shapes only)."""
    Q, K = _f64(q), _f64(k)
    B, Hq, Nq, _ = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    P = np.zeros((B, Hq, Nq, Nk))
    for b in range(B):
        for h in range(Hq):
            S = _scores(Q[b, h], K[b, kv_head(h, Hq, Hkv)], scale)
            S[~visible_mask(np.arange(Nq), Nq, Nk, causal, window)] = -np.inf
            P[b, h] = _softmax_rows(S)[0]
    return P


def attention_varlen(q, k, v, cu_q, cu_k, scale: float, causal: bool = False, window: int = 0):
    """Ragged batch in packed token-major layout.

    ``q``: ``[total_q, Hq, D]``, ``k``/``v``: ``[total_k, Hkv, D]``; sequence b owns
    query rows ``cu_q[b]:cu_q[b+1]`` and key rows ``cu_k[b]:cu_k[b+1]``.  Each
    sequence is an independent :func:`attention_forward` (masks per sequence).
    Returns ``O [total_q, Hq, D]`` and ``LSE [Hq, total_q]``.
    """
    Q, K, V = _f64(q), _f64(k), _f64(v)
    cq, ck = [int(x) for x in cu_q], [int(x) for x in cu_k]
    O = np.zeros((Q.shape[0], Q.shape[1], V.shape[2]))
    LSE = np.zeros((Q.shape[1], Q.shape[0]))
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        if q1 == q0:
            continue
        if k1 == k0:   # no keys: every row sees nothing
            LSE[:, q0:q1] = -np.inf
            continue
        Ob, Lb = attention_forward(Q[q0:q1].transpose(1, 0, 2)[None], K[k0:k1].transpose(1, 0, 2)[None],
                                   V[k0:k1].transpose(1, 0, 2)[None], scale, causal, window)
        O[q0:q1] = Ob[0].transpose(1, 0, 2)
        LSE[:, q0:q1] = Lb[0]
    return O, LSE


# ---------------------------------------------------------------------------
# Decode: one query token per sequence against a contiguous KV cache
# ``[B, Nk_max, Hkv, D]`` of which sequence b uses the first ``seqlens[b]`` rows.
# ---------------------------------------------------------------------------

def _decode_one(q_bh: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """O and LSE of one query vector against key rows ``K`` / value rows ``V``."""
    S = _scores(q_bh[None, :], K, scale)
    P, lse = _softmax_rows(S)
    return (P @ V)[0], lse[0]


def decode_forward(q, k_cache, v_cache, seqlens, scale: float, batches=None):
    """Unsplit decode: ``O [B,Hq,D]``, ``LSE [B,Hq]`` over keys ``j < seqlens[b]``.

    ``batches`` optionally restricts the work to some sequences (other rows are
    left at zero).
    """
    B, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    lens = [int(x) for x in seqlens]
    O = np.zeros((B, Hq, v_cache.shape[3]))
    LSE = np.zeros((B, Hq))
    for b in (range(B) if batches is None else batches):
        Kb = _f64(k_cache[b, :lens[b]])                 # [Nk_b, Hkv, D]
        Vb = _f64(v_cache[b, :lens[b]])
        qb = _f64(q[b])
        for h in range(Hq):
            kh = kv_head(h, Hq, Hkv)
            O[b, h], LSE[b, h] = _decode_one(qb[h], Kb[:, kh], Vb[:, kh], scale)
    return O, LSE


def decode_split_partials(q, k_cache, v_cache, seqlens, scale: float, chunk: int,
                          batches=None):
    """Split-KV step: per (b, h, chunk c) the chunk's normalised output and LSE.

    Returns ``O_part [B,Hq,S_max,D]``, ``LSE_part [B,Hq,S_max]`` and the number
    of chunks per sequence ``n_split [B]``; entries at ``c >= n_split[b]`` stay 0.
    """
    B, Hq, D = q.shape
    Hkv, Nk_max = k_cache.shape[2], k_cache.shape[1]
    S_max = -(-Nk_max // chunk)
    lens = [int(x) for x in seqlens]
    n_split = np.array([-(-n // chunk) for n in lens], dtype=np.int64)
    O_part = np.zeros((B, Hq, S_max, v_cache.shape[3]))
    LSE_part = np.zeros((B, Hq, S_max))
    for b in (range(B) if batches is None else batches):
        qb = _f64(q[b])
        for c in range(n_split[b]):
            j0, j1 = c * chunk, min((c + 1) * chunk, lens[b])
            Kc = _f64(k_cache[b, j0:j1])
            Vc = _f64(v_cache[b, j0:j1])
            for h in range(Hq):
                kh = kv_head(h, Hq, Hkv)
                O_part[b, h, c], LSE_part[b, h, c] = _decode_one(qb[h], Kc[:, kh], Vc[:, kh], scale)
    return O_part, LSE_part, n_split


def decode_combine(O_part, LSE_part, n_split):
    """Combine step: LSE-weighted merge of the chunk results.

    ``M = max_c LSE_c``, ``w_c = exp(LSE_c - M)``, ``O = sum_c w_c O_c / sum_c w_c``,
    ``LSE = M + ln sum_c w_c`` over the valid chunks ``c < n_split[b]``.
    """
    O_part, LSE_part = _f64(O_part), _f64(LSE_part)
    B, Hq, _, D = O_part.shape
    O = np.zeros((B, Hq, D))
    LSE = np.zeros((B, Hq))
    for b in range(B):
        n = int(n_split[b])
        L = LSE_part[b, :, :n]                          # [Hq, n]
        M = L.max(axis=1)
        w = np.exp(L - M[:, None])
        s = w.sum(axis=1)
        O[b] = np.einsum("hc,hcd->hd", w, O_part[b, :, :n]) / s[:, None]
        LSE[b] = M + np.log(s)
    return O, LSE


# ---------------------------------------------------------------------------
# Paged KV cache: key j of sequence b is row j % page_size of page
# block_table[b, j // page_size].
# ---------------------------------------------------------------------------

def paged_rows(pages, block_table_b, n: int):
    """The first ``n`` token rows of one sequence, gathered from its pages."""
    page_size = pages.shape[1]
    j = np.arange(n)
    page = np.asarray(block_table_b)[j // page_size]
    return _f64(pages[page, j % page_size]) if n else np.zeros((0,) + tuple(pages.shape[2:]))


def decode_forward_paged(q, k_pages, v_pages, block_table, seqlens, scale: float, batches=None):
    """Decode against a paged cache: ``O [B,Hq,D]``, ``LSE [B,Hq]``.

    Same definition as :func:`decode_forward`, with sequence b's keys gathered
    through its block-table row.
    """
    B, Hq, D = q.shape
    Hkv = k_pages.shape[2]
    bt = np.asarray(block_table)
    lens = [int(x) for x in seqlens]
    O = np.zeros((B, Hq, v_pages.shape[3]))
    LSE = np.zeros((B, Hq))
    for b in (range(B) if batches is None else batches):
        Kb = paged_rows(k_pages, bt[b], lens[b])          # [Nk_b, Hkv, D]
        Vb = paged_rows(v_pages, bt[b], lens[b])
        qb = _f64(q[b])
        for h in range(Hq):
            kh = kv_head(h, Hq, Hkv)
            O[b, h], LSE[b, h] = _decode_one(qb[h], Kb[:, kh], Vb[:, kh], scale)
    return O, LSE


def e4m3_to_float(codes) -> np.ndarray:
    """fp64 value of each OCP FP8 E4M3 code (uint8 array), from the format's
    definition: sign bit 7, exponent bits 6-3 with bias 7, mantissa bits 2-0;
    exponent 0 is subnormal (``m/8 * 2^-6``); code S.1111.111 is NaN."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)
    return sign * mag


def decode_forward_fp8(q, k_codes, v_codes, k_scale: float, v_scale: float, seqlens, scale: float,
                       batches=None):
    """Decode against an fp8 (E4M3) cache ``[B,Nk_max,Hkv,D]`` of codes: the
    plain decode of :func:`decode_forward` on the values ``code * k_scale`` /
    ``code * v_scale`` (only each sequence's first ``Nk_b`` rows are decoded)."""
    B, Hq, D = q.shape
    Hkv = k_codes.shape[2]
    lens = [int(x) for x in seqlens]
    kc, vc = np.asarray(k_codes), np.asarray(v_codes)
    O = np.zeros((B, Hq, vc.shape[3]))
    LSE = np.zeros((B, Hq))
    for b in (range(B) if batches is None else batches):
        Kb = e4m3_to_float(kc[b, :lens[b]]) * float(k_scale)
        Vb = e4m3_to_float(vc[b, :lens[b]]) * float(v_scale)
        qb = _f64(q[b])
        for h in range(Hq):
            kh = kv_head(h, Hq, Hkv)
            O[b, h], LSE[b, h] = _decode_one(qb[h], Kb[:, kh], Vb[:, kh], scale)
    return O, LSE


def decode_forward_paged_fp8(q, k_pages, v_pages, k_scale: float, v_scale: float, block_table,
                             seqlens, scale: float, batches=None):
    """:func:`decode_forward_paged` on a paged cache of E4M3 codes, values as in
    :func:`decode_forward_fp8`."""
    B, Hq, D = q.shape
    kp, vp = np.asarray(k_pages), np.asarray(v_pages)
    Hkv = kp.shape[2]
    page_size = kp.shape[1]
    bt = np.asarray(block_table)
    lens = [int(x) for x in seqlens]
    O = np.zeros((B, Hq, vp.shape[3]))
    LSE = np.zeros((B, Hq))
    for b in (range(B) if batches is None else batches):
        j = np.arange(lens[b])
        page = bt[b][j // page_size]
        Kb = e4m3_to_float(kp[page, j % page_size]) * float(k_scale)
        Vb = e4m3_to_float(vp[page, j % page_size]) * float(v_scale)
        qb = _f64(q[b])
        for h in range(Hq):
            kh = kv_head(h, Hq, Hkv)
            O[b, h], LSE[b, h] = _decode_one(qb[h], Kb[:, kh], Vb[:, kh], scale)
    return O, LSE


def attention_forward_fp8(q_codes, k_codes, v_codes, q_scale: float, k_scale: float,
                          v_scale: float, scale: float, causal: bool = False, window: int = 0):
    """Forward on fp8 (E4M3) Q, K and V ``[B,H,N,D]`` of codes: the plain forward of
    :func:`attention_forward` on the values ``code * q_scale``, ``code * k_scale``
    and ``code * v_scale``."""
    Q = e4m3_to_float(q_codes) * float(q_scale)
    K = e4m3_to_float(k_codes) * float(k_scale)
    V = e4m3_to_float(v_codes) * float(v_scale)
    return attention_forward(Q, K, V, scale, causal, window)


def attention_rows_fp8(q_codes, k_codes, v_codes, q_scale: float, k_scale: float, v_scale: float,
                       scale: float, rows, causal: bool = False, window: int = 0):
    """:func:`attention_rows` (selected ``(b, h, i)`` rows) on E4M3 codes, values as in
    :func:`attention_forward_fp8`; only the K/V heads the rows read are decoded."""
    rows = list(rows)
    Hq, Hkv = q_codes.shape[1], k_codes.shape[1]
    O = np.zeros((len(rows), v_codes.shape[3]))
    LSE = np.zeros(len(rows))
    for n, (b, h, i) in enumerate(rows):
        kh = kv_head(h, Hq, Hkv)
        q1 = e4m3_to_float(q_codes[b:b + 1, h:h + 1]) * float(q_scale)
        k1 = e4m3_to_float(k_codes[b:b + 1, kh:kh + 1]) * float(k_scale)
        v1 = e4m3_to_float(v_codes[b:b + 1, kh:kh + 1]) * float(v_scale)
        o, lse = attention_rows(q1, k1, v1, scale, [(0, 0, i)], causal, window)
        O[n], LSE[n] = o[0], lse[0]
    return O, LSE


def softcap_scores(S: np.ndarray, cap: float) -> np.ndarray:
    """``cap * tanh(S / cap)`` for ``cap > 0`` (masked -inf entries stay -inf);
    ``S`` unchanged for ``cap <= 0``."""
    if not cap > 0:
        return S
    with np.errstate(invalid="ignore"):
        return np.where(np.isneginf(S), -np.inf, cap * np.tanh(S / cap))


def _softmax_rows_sink(S: np.ndarray, sink: float):
    """Two-pass row softmax with one extra denominator term ``exp(sink)`` (no
    value attached).  ``sink = -inf`` is the plain softmax.  Returns ``(P, lse)``."""
    M = np.maximum(S.max(axis=1), sink)                # pass 1: max over keys and the sink
    empty = ~np.isfinite(M)                            # every key masked and no sink
    M_safe = np.where(empty, 0.0, M)
    E = np.exp(S - M_safe[:, None])                    # pass 2: exp (masked -> 0)
    l = E.sum(axis=1) + np.exp(sink - M_safe)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, l)[:, None])
        lse = np.where(empty, -np.inf, M_safe + np.log(np.where(empty, 1.0, l)))
    return P, lse


def _sink_of(sinks, h: int) -> float:
    return -np.inf if sinks is None else float(np.asarray(sinks, dtype=np.float64)[h])


def attention_forward_ext(q, k, v, scale: float, causal: bool = False, window: int = 0,
                          softcap: float = 0.0, sinks=None, row_block: int = 512):
    """:func:`attention_forward` with a softcap on the scaled scores and one sink
    logit per query head (``sinks`` ``[Hq]``, or None for none)."""
    Q, K, V = _f64(q), _f64(k), _f64(v)
    B, Hq, Nq, D = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    O = np.zeros((B, Hq, Nq, V.shape[3]))
    LSE = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            kh = kv_head(h, Hq, Hkv)
            for i0 in range(0, Nq, row_block):
                rows = np.arange(i0, min(i0 + row_block, Nq))
                S = _scores(Q[b, h, rows], K[b, kh], scale)
                S[~visible_mask(rows, Nq, Nk, causal, window)] = -np.inf
                P, lse = _softmax_rows_sink(softcap_scores(S, softcap), _sink_of(sinks, h))
                O[b, h, rows] = P @ V[b, kh]
                LSE[b, h, rows] = lse
    return O, LSE


def attention_rows_ext(q, k, v, scale: float, rows, causal: bool = False, window: int = 0,
                       softcap: float = 0.0, sinks=None):
    """:func:`attention_rows` with softcap and sinks, one ``(b, h, i)`` row at a time."""
    B, Hq, Nq, _ = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    O = np.zeros((len(rows), v.shape[3]))
    LSE = np.zeros(len(rows))
    for n, (b, h, i) in enumerate(rows):
        kh = kv_head(h, Hq, Hkv)
        S = _scores(_f64(q[b, h, i])[None, :], _f64(k[b, kh]), scale)
        S[~visible_mask(np.array([i]), Nq, Nk, causal, window)] = -np.inf
        P, lse = _softmax_rows_sink(softcap_scores(S, softcap), _sink_of(sinks, h))
        O[n] = (P @ _f64(v[b, kh]))[0]
        LSE[n] = lse[0]
    return O, LSE


def _backward_head(Qh, Kh, Vh, dOh, scale: float, vis):
    """One query head against its KV head: ``(dQ_h, dK_h, dV_h)``.

    dV = P^T dO;  dP = dO V^T;  dS = P * (dP - rowsum(P * dP));
    dQ = scale dS K;  dK = scale dS^T Q."""
    S = _scores(Qh, Kh, scale)
    S[~vis] = -np.inf
    P, _ = _softmax_rows(S)
    dV = P.T @ dOh
    dP = dOh @ Vh.T
    dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
    return scale * (dS @ Kh), scale * (dS.T @ Qh), dV


def attention_backward(q, k, v, do, scale: float, causal: bool = False, window: int = 0):
    """Gradients of :func:`attention_forward`'s O for the upstream gradient
    ``do`` ``[B,Hq,Nq,D]``: ``(dQ [B,Hq,Nq,D], dK [B,Hkv,Nk,D], dV [B,Hkv,Nk,D])``
    in fp64."""
    Q, K, V, dO = _f64(q), _f64(k), _f64(v), _f64(do)
    B, Hq, Nq, D = Q.shape
    Hkv, Nk = K.shape[1], K.shape[2]
    vis = visible_mask(np.arange(Nq), Nq, Nk, causal, window)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for b in range(B):
        for h in range(Hq):
            kh = kv_head(h, Hq, Hkv)
            gq, gk, gv = _backward_head(Q[b, h], K[b, kh], V[b, kh], dO[b, h], scale, vis)
            dQ[b, h] = gq
            dK[b, kh] += gk
            dV[b, kh] += gv
    return dQ, dK, dV
