"""Pins of the fp64 oracle against what the mathematics fixes (CPU only).

Each ``pin_*`` function checks the oracle module passed in against a closed
form, an invariant, a hand-derived example or an independent brute force.
``test_mutants_are_caught`` plants plausible mistakes in the oracle (on the CPU)
and checks that at least one pin fails for each, so the battery is known to
have teeth.
"""
import math
import os
import re

import numpy as np
import pytest
import torch

import oracle.attention as ORA

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def visible_list(i, Nq, Nk, causal, window):
    return [j for j in range(Nk)
            if (not causal or j <= i + Nk - Nq) and (window <= 0 or j > i + Nk - Nq - window)]


# ---------------------------------------------------------------- brute force
def brute_force(q, k, v, scale, causal, window):
    """Pure-Python loops with exactly rounded sums (math.fsum)."""
    B, Hq, Nq, D = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    g = Hq // Hkv
    O = np.zeros((B, Hq, Nq, v.shape[3]))
    L = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            kh = h // g
            for i in range(Nq):
                js = visible_list(i, Nq, Nk, causal, window)
                if not js:
                    L[b, h, i] = -math.inf
                    continue
                s = {j: scale * math.fsum(float(q[b, h, i, d]) * float(k[b, kh, j, d]) for d in range(D))
                     for j in js}
                m = max(s.values())
                e = {j: math.exp(s[j] - m) for j in js}
                l = math.fsum(e.values())
                for d in range(v.shape[3]):
                    O[b, h, i, d] = math.fsum(e[j] * float(v[b, kh, j, d]) for j in js) / l
                L[b, h, i] = m + math.log(l)
    return O, L


CASES = [  # (B, Hq, Hkv, Nq, Nk, D, causal, window)
    (1, 2, 1, 3, 5, 4, False, 0),
    (2, 4, 2, 5, 5, 3, True, 0),
    (1, 2, 2, 4, 7, 2, True, 0),      # Nq < Nk: bottom-right causal
    (1, 3, 1, 6, 6, 3, True, 2),      # causal + window
    (1, 2, 1, 5, 4, 2, False, 3),     # window without causal
    (1, 2, 1, 6, 3, 2, True, 0),      # Nq > Nk: some rows fully masked
]


def pin_brute_force(ora):
    for n, (B, Hq, Hkv, Nq, Nk, D, causal, window) in enumerate(CASES):
        q, k, v = rnd(10 + n, B, Hq, Nq, D), rnd(20 + n, B, Hkv, Nk, D), rnd(30 + n, B, Hkv, Nk, D)
        scale = 1.0 / math.sqrt(D)
        O, L = ora.attention_forward(q, k, v, scale, causal, window, row_block=2)
        Ob, Lb = brute_force(q, k, v, scale, causal, window)
        assert np.allclose(O, Ob, rtol=0, atol=1e-12), f"case {n}: O differs from brute force"
        fin = np.isfinite(Lb)
        assert np.array_equal(fin, np.isfinite(L)), f"case {n}: LSE finiteness differs"
        assert np.allclose(L[fin], Lb[fin], rtol=0, atol=1e-12), f"case {n}: LSE differs"
        assert np.all(L[~fin] == -np.inf) and np.all(O[~fin] == 0)


def pin_sdpa(ora):
    """Agreement with torch's scaled_dot_product_attention in float64 on CPU."""
    for n, (B, Hq, Hkv, Nq, Nk, D) in enumerate([(2, 4, 2, 9, 9, 8), (1, 8, 2, 17, 17, 16)]):
        q, k, v = rnd(40 + n, B, Hq, Nq, D), rnd(50 + n, B, Hkv, Nk, D), rnd(60 + n, B, Hkv, Nk, D)
        for causal in (False, True):
            O, _ = ora.attention_forward(q, k, v, 0.3, causal, 0)
            g = Hq // Hkv
            kt = torch.from_numpy(k).repeat_interleave(g, dim=1)
            vt = torch.from_numpy(v).repeat_interleave(g, dim=1)
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q), kt, vt, is_causal=causal, scale=0.3).numpy()
            assert np.allclose(O, ref, rtol=0, atol=1e-12), "O differs from SDPA"


# ---------------------------------------------------------------- closed forms
def pin_zero_query(ora):
    """Q = 0: O = mean of the visible V rows, LSE = ln(#visible)."""
    for (B, Hq, Hkv, Nq, Nk, D, causal, window) in CASES:
        q = np.zeros((B, Hq, Nq, D))
        k, v = rnd(1, B, Hkv, Nk, D), rnd(2, B, Hkv, Nk, D)
        O, L = ora.attention_forward(q, k, v, 0.7, causal, window)
        for b in range(B):
            for h in range(Hq):
                kh = h // (Hq // Hkv)
                for i in range(Nq):
                    js = visible_list(i, Nq, Nk, causal, window)
                    if not js:
                        assert L[b, h, i] == -np.inf and np.all(O[b, h, i] == 0)
                        continue
                    assert abs(L[b, h, i] - math.log(len(js))) < 1e-13
                    assert np.allclose(O[b, h, i], v[b, kh, js].mean(axis=0), rtol=0, atol=1e-13)


def pin_single_key(ora):
    """Nk = 1: O = V[0] of the query head's KV head, LSE = scale * q . k0."""
    B, Hq, Hkv, Nq, D = 2, 6, 3, 4, 5
    q, k, v = rnd(3, B, Hq, Nq, D), rnd(4, B, Hkv, 1, D), rnd(5, B, Hkv, 1, D)
    O, L = ora.attention_forward(q, k, v, 0.4, False, 0)
    for b in range(B):
        for h in range(Hq):
            kh = h // 2
            for i in range(Nq):
                assert np.allclose(O[b, h, i], v[b, kh, 0], rtol=0, atol=1e-14)
                assert abs(L[b, h, i] - 0.4 * float(np.dot(q[b, h, i], k[b, kh, 0]))) < 1e-13


def pin_probability_rows(ora):
    """Rows of P sum to 1 (0 for fully masked rows) and sum_j exp(s_ij - LSE_i) = 1."""
    for (B, Hq, Hkv, Nq, Nk, D, causal, window) in CASES:
        q, k, v = rnd(6, B, Hq, Nq, D), rnd(7, B, Hkv, Nk, D), rnd(8, B, Hkv, Nk, D)
        P = ora.attention_probabilities(q, k, 0.5, causal, window)
        _, L = ora.attention_forward(q, k, v, 0.5, causal, window)
        for b in range(B):
            for h in range(Hq):
                kh = h // (Hq // Hkv)
                for i in range(Nq):
                    js = visible_list(i, Nq, Nk, causal, window)
                    hidden = [j for j in range(Nk) if j not in js]
                    assert np.all(P[b, h, i, hidden] == 0)
                    if js:
                        assert abs(P[b, h, i].sum() - 1) < 1e-13
                        s = [0.5 * math.fsum(q[b, h, i] * k[b, kh, j]) for j in js]
                        assert abs(math.fsum(math.exp(x - L[b, h, i]) for x in s) - 1) < 1e-12


def pin_causal_first_row(ora):
    """Causal with Nq = Nk: row 0 returns V[0] and LSE_0 = scale * q0 . k0."""
    B, Hq, Hkv, N, D = 2, 4, 2, 7, 6
    q, k, v = rnd(9, B, Hq, N, D), rnd(10, B, Hkv, N, D), rnd(11, B, Hkv, N, D)
    O, L = ora.attention_forward(q, k, v, 0.25, True, 0)
    for b in range(B):
        for h in range(Hq):
            kh = h // 2
            assert np.allclose(O[b, h, 0], v[b, kh, 0], rtol=0, atol=1e-14)
            assert abs(L[b, h, 0] - 0.25 * float(np.dot(q[b, h, 0], k[b, kh, 0]))) < 1e-13


def pin_dominant_key(ora):
    """A key parallel to the query with a huge score selects its V row."""
    B, H, Nq, Nk, D = 1, 1, 3, 9, 8
    q, k, v = rnd(12, B, H, Nq, D), rnd(13, B, H, Nk, D), rnd(14, B, H, Nk, D)
    i, jstar, scale = 1, 6, 1 / math.sqrt(D)
    others = max(scale * float(np.dot(q[0, 0, i], k[0, 0, j])) for j in range(Nk) if j != jstar)
    c = (others + 60.0) / (scale * float(np.dot(q[0, 0, i], q[0, 0, i])))
    k[0, 0, jstar] = c * q[0, 0, i]
    O, L = ora.attention_forward(q, k, v, scale, False, 0)
    assert np.allclose(O[0, 0, i], v[0, 0, jstar], rtol=1e-18, atol=1e-20 * float(np.abs(v).max()) + 1e-24)
    assert abs(L[0, 0, i] - scale * float(np.dot(q[0, 0, i], k[0, 0, jstar]))) < 1e-12


# ---------------------------------------------------------------- invariants
def pin_invariants(ora):
    B, Hq, Hkv, Nq, Nk, D = 1, 4, 2, 6, 6, 5
    q, k, v = rnd(15, B, Hq, Nq, D), rnd(16, B, Hkv, Nk, D), rnd(17, B, Hkv, Nk, D)
    O, L = ora.attention_forward(q, k, v, 0.6, False, 0)
    # joint permutation of K and V rows (non-causal)
    perm = np.random.default_rng(18).permutation(Nk)
    Op, Lp = ora.attention_forward(q, k[:, :, perm], v[:, :, perm], 0.6, False, 0)
    assert np.allclose(Op, O, atol=1e-13) and np.allclose(Lp, L, atol=1e-13), "permutation"
    # V -> a V + c maps O -> a O + c
    Oa, _ = ora.attention_forward(q, k, 2.5 * v - 1.25, 0.6, False, 0)
    assert np.allclose(Oa, 2.5 * O - 1.25, atol=1e-12), "affine V"
    # adding w to every key shifts row i's scores by scale*q_i.w: O fixed, LSE shifted
    w = rnd(19, D)
    Ow, Lw = ora.attention_forward(q, k + w, v, 0.6, False, 0)
    assert np.allclose(Ow, O, atol=1e-12), "score shift changes O"
    assert np.allclose(Lw, L + 0.6 * np.einsum("bhid,d->bhi", q, w), atol=1e-12), "score shift LSE"
    # GQA equals MHA on repeated K/V
    g = Hq // Hkv
    Om, Lm = ora.attention_forward(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), 0.6, False, 0)
    assert np.allclose(Om, O, atol=1e-14) and np.allclose(Lm, L, atol=1e-14), "GQA vs MHA"
    # causal (Nq = Nk) row i equals dense attention over keys 0..i
    Oc, Lc = ora.attention_forward(q, k, v, 0.6, True, 0)
    for i in range(Nq):
        Od, Ld = ora.attention_forward(q[:, :, i:i + 1], k[:, :, :i + 1], v[:, :, :i + 1], 0.6, False, 0)
        assert np.allclose(Oc[:, :, i], Od[:, :, 0], atol=1e-13) and np.allclose(Lc[:, :, i], Ld[:, :, 0], atol=1e-13)
    # causal + window w, row i equals dense attention over keys i-w+1..i
    wdw = 2
    Ow2, Lw2 = ora.attention_forward(q, k, v, 0.6, True, wdw)
    for i in range(Nq):
        j0 = max(0, i - wdw + 1)
        Od, Ld = ora.attention_forward(q[:, :, i:i + 1], k[:, :, j0:i + 1], v[:, :, j0:i + 1], 0.6, False, 0)
        assert np.allclose(Ow2[:, :, i], Od[:, :, 0], atol=1e-13) and np.allclose(Lw2[:, :, i], Ld[:, :, 0], atol=1e-13)
    # selected rows agree with the full forward
    rows = [(0, 3, 2), (0, 0, 5), (0, 1, 0)]
    Or, Lr = ora.attention_rows(q, k, v, 0.6, rows, True, 0)
    for n, (b, h, i) in enumerate(rows):
        assert np.allclose(Or[n], Oc[b, h, i], atol=1e-14) and abs(Lr[n] - Lc[b, h, i]) < 1e-14


def _decode_case(seed=21, B=3, Hq=4, Hkv=2, D=6, Nk_max=11):
    r = np.random.default_rng(seed)
    seqlens = np.array([11, 1, 7][:B])
    q = r.standard_normal((B, Hq, D))
    kc = r.standard_normal((B, Nk_max, Hkv, D))
    vc = r.standard_normal((B, Nk_max, Hkv, D))
    for b in range(B):                          # sentinels in the unused tail
        kc[b, seqlens[b]:] = 64.0
        vc[b, seqlens[b]:] = 1e4
    return q, kc, vc, seqlens


def pin_decode(ora):
    """Decode = prefill of one query against the sequence's keys; split+combine = unsplit."""
    q, kc, vc, lens = _decode_case()
    B, Hq, D = q.shape
    O, L = ora.decode_forward(q, kc, vc, lens, 0.45)
    for b in range(B):
        n = lens[b]
        kb = kc[b, :n].transpose(1, 0, 2)[None]      # [1, Hkv, n, D]
        vb = vc[b, :n].transpose(1, 0, 2)[None]
        Op, Lp = brute_force(q[b][None, :, None, :], kb, vb, 0.45, False, 0)
        assert np.allclose(O[b], Op[0, :, 0], atol=1e-12) and np.allclose(L[b], Lp[0, :, 0], atol=1e-12)
    for chunk in (1, 2, 3, 4, 8, 16):
        Op, Lp, ns = ora.decode_split_partials(q, kc, vc, lens, 0.45, chunk)
        assert list(ns) == [-(-int(n) // chunk) for n in lens]
        Oc, Lc = ora.decode_combine(Op, Lp, ns)
        assert np.allclose(Oc, O, atol=1e-12) and np.allclose(Lc, L, atol=1e-12), f"chunk {chunk}"
    # each partial is the attention of its own chunk
    Op, Lp, ns = ora.decode_split_partials(q, kc, vc, lens, 0.45, 4)
    b, c = 0, 2                                    # keys 8..10 of sequence 0
    kb = kc[b, 8:11].transpose(1, 0, 2)[None]
    vb = vc[b, 8:11].transpose(1, 0, 2)[None]
    Oe, Le = brute_force(q[b][None, :, None, :], kb, vb, 0.45, False, 0)
    assert np.allclose(Op[b, :, c], Oe[0, :, 0], atol=1e-12) and np.allclose(Lp[b, :, c], Le[0, :, 0], atol=1e-12)


def pin_paged_decode(ora):
    """Paged decode equals contiguous decode of the same rows, for any page placement."""
    q, kc, vc, lens = _decode_case()
    B, Hq, D = q.shape
    Nk_max, Hkv = kc.shape[1], kc.shape[2]
    O, L = ora.decode_forward(q, kc, vc, lens, 0.45)
    for page_size in (1, 2, 4):
        max_pages = -(-Nk_max // page_size)
        perm = np.random.default_rng(page_size).permutation(B * max_pages)
        bt = perm.reshape(B, max_pages)
        kp = np.full((B * max_pages, page_size, Hkv, D), np.nan)
        vp = np.full((B * max_pages, page_size, Hkv, D), np.nan)
        for b in range(B):
            for j in range(Nk_max):
                kp[bt[b, j // page_size], j % page_size] = kc[b, j]
                vp[bt[b, j // page_size], j % page_size] = vc[b, j]
        Op, Lp = ora.decode_forward_paged(q, kp, vp, bt, lens, 0.45)
        assert np.allclose(Op, O, rtol=0, atol=1e-14) and np.allclose(Lp, L, rtol=0, atol=1e-14), page_size
    # a hand-built 2-page layout of the golden example's keys (pages in reverse order)
    G = _read_golden("closed_form_tiny.txt")
    Kg, Vg = G[("input", "K")], G[("input", "V")]            # [3, 2]
    kp = np.zeros((2, 2, 1, 2))
    vp = np.zeros((2, 2, 1, 2))
    kp[1, :, 0], kp[0, :1, 0] = Kg[:2], Kg[2:]
    vp[1, :, 0], vp[0, :1, 0] = Vg[:2], Vg[2:]
    Op, Lp = ora.decode_forward_paged(G[("input", "Q")][:1][None], kp, vp, [[1, 0]], [3], 1.0)
    assert np.allclose(Op[0, 0], G[("dense", "O")][0], atol=1e-14)
    assert abs(Lp[0, 0] - G[("dense", "LSE")][0][0]) < 1e-14


def pin_varlen(ora):
    """Ragged batch = each sequence on its own (brute force), empty sequences included."""
    lens_q, lens_k = [3, 0, 5, 2], [3, 4, 7, 0]
    Hq, Hkv, D = 4, 2, 3
    r = np.random.default_rng(31)
    q = r.standard_normal((sum(lens_q), Hq, D))
    k = r.standard_normal((sum(lens_k), Hkv, D))
    v = r.standard_normal((sum(lens_k), Hkv, D))
    cq, ck = np.concatenate([[0], np.cumsum(lens_q)]), np.concatenate([[0], np.cumsum(lens_k)])
    for causal, window in ((False, 0), (True, 0), (True, 2)):
        O, L = ora.attention_varlen(q, k, v, cq, ck, 0.5, causal, window)
        for b in range(4):
            q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
            if q1 == q0:
                continue
            if k1 == k0:
                assert np.all(O[q0:q1] == 0) and np.all(L[:, q0:q1] == -np.inf)
                continue
            Ob, Lb = brute_force(q[q0:q1].transpose(1, 0, 2)[None], k[k0:k1].transpose(1, 0, 2)[None],
                                 v[k0:k1].transpose(1, 0, 2)[None], 0.5, causal, window)
            assert np.allclose(O[q0:q1], Ob[0].transpose(1, 0, 2), atol=1e-12)
            fin = np.isfinite(Lb[0])
            assert np.array_equal(np.isfinite(L[:, q0:q1]), fin)
            assert np.allclose(L[:, q0:q1][fin], Lb[0][fin], atol=1e-12)


# ---------------------------------------------------------------- golden
def _read_golden(name):
    env = {"ln": math.log}
    table = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            head, vals = line.split(":")
            case, field, row = head.split()
            assert re.fullmatch(r"[0-9lnN()/.+\- ]*", vals), vals
            table.setdefault((case, field), {})[int(row)] = [eval(t, {"__builtins__": {}}, env) for t in vals.split()]
    return {key: np.array([rows[r] for r in sorted(rows)]) for key, rows in table.items()}


def pin_golden(ora):
    G = _read_golden("closed_form_tiny.txt")
    Q, K, V = (G[("input", f)][None, None] for f in "QKV")
    for case, causal, window in (("dense", False, 0), ("causal", True, 0), ("window1", True, 1)):
        O, L = ora.attention_forward(Q, K, V, 1.0, causal, window)
        assert np.allclose(O[0, 0], G[(case, "O")], rtol=0, atol=1e-14), case
        assert np.allclose(L[0, 0], G[(case, "LSE")][0], rtol=0, atol=1e-14), case
    # split-KV of query row 0 with chunk 2, against the hand-derived partials
    q = Q[0, :, 0][None]                          # [1, 1, D]
    kc = K[0].transpose(1, 0, 2)[None]            # [1, Nk, 1, D]
    vc = V[0].transpose(1, 0, 2)[None]
    Op, Lp, ns = ora.decode_split_partials(q, kc, vc, [3], 1.0, 2)
    assert np.allclose(Op[0, 0], G[("split2", "O")], atol=1e-14)
    assert np.allclose(Lp[0, 0], G[("split2", "LSE")][0], atol=1e-14)
    Oc, Lc = ora.decode_combine(Op, Lp, ns)
    assert np.allclose(Oc[0, 0], G[("split2", "combinedO")][0], atol=1e-14)
    assert abs(Lc[0, 0] - G[("split2", "combinedLSE")][0][0]) < 1e-14


def _golden_e4m3():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "e4m3_codes.txt")
    out = []
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        code, expr = line.split()
        out.append((int(code, 16), float("nan") if expr == "nan" else float(eval(expr, {"__builtins__": {}}))))
    return out


def pin_e4m3_codes(ora):
    """E4M3 decoding against the hand-derived codes of tests/golden/e4m3_codes.txt
    (format definition) and against torch's float8_e4m3fn conversion for all 256
    codes (an independent implementation of the same format)."""
    for code, want in _golden_e4m3():
        got = float(ora.e4m3_to_float(np.array([code], dtype=np.uint8))[0])
        if math.isnan(want):
            assert math.isnan(got), (hex(code), got)
        else:
            assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), (hex(code), got, want)
    codes = np.arange(256, dtype=np.uint8)
    mine = ora.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(mine[fin], ref[fin])


def pin_fp8_decode(ora):
    """fp8-cache decode: brute force (math.fsum) on the decoded values for a tiny
    case, the folding of k_scale into the score scale and of v_scale into O, and
    paged == contiguous on pages laid out in a random order."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, nmax = 2, 4, 2, 8, 11
    lens = [11, 5]
    q = rng.standard_normal((B, Hq, D))
    kc = rng.integers(0, 256, (B, nmax, Hkv, D), dtype=np.uint8)
    vc = rng.integers(0, 256, (B, nmax, Hkv, D), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0x3A          # no NaN codes in the valid rows
    vc[(vc & 0x7F) == 0x7F] = 0x41
    kc[1, 5:] = 0x7F                         # NaN codes past sequence 1: never read
    vc[1, 5:] = 0xFF
    ks, vs, sc = 0.0625, 0.25, 0.3
    O, L = ora.decode_forward_fp8(q, kc, vc, ks, vs, lens, sc)
    # brute force from the format definition, one element at a time
    def val(c):
        c = int(c)
        sgn = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 15, c & 7
        return sgn * ((m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    for b in range(B):
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            s = [sc * math.fsum(q[b, h, d] * val(kc[b, j, kh, d]) * ks for d in range(D)) for j in range(lens[b])]
            mx = max(s)
            w = [math.exp(x - mx) for x in s]
            den = math.fsum(w)
            for d in range(D):
                o = math.fsum(w[j] * val(vc[b, j, kh, d]) * vs for j in range(lens[b])) / den
                assert abs(O[b, h, d] - o) < 1e-12 * max(1.0, abs(o)), (b, h, d)
            assert abs(L[b, h] - (mx + math.log(den))) < 1e-12
    O2, L2 = ora.decode_forward_fp8(q, kc, vc, 1.0, vs, lens, sc * ks)
    assert np.allclose(O2, O, rtol=1e-13, atol=1e-13) and np.allclose(L2, L, rtol=1e-13, atol=1e-13)
    O3, L3 = ora.decode_forward_fp8(q, kc, vc, ks, 3 * vs, lens, sc)
    assert np.allclose(O3, 3 * O, rtol=1e-13, atol=1e-13) and np.allclose(L3, L, rtol=1e-13, atol=1e-13)
    page = 4
    need = [-(-n // page) for n in lens]
    perm = rng.permutation(sum(need) + 2)
    kp = np.full((len(perm), page, Hkv, D), 0x7F, dtype=np.uint8)
    vp = np.full((len(perm), page, Hkv, D), 0xFF, dtype=np.uint8)
    bt = np.zeros((B, max(need)), dtype=np.int32)
    nxt = 0
    for b in range(B):
        for i in range(need[b]):
            pg = int(perm[nxt]); nxt += 1
            bt[b, i] = pg
            rows = min(page, lens[b] - i * page)
            kp[pg, :rows] = kc[b, i * page: i * page + rows]
            vp[pg, :rows] = vc[b, i * page: i * page + rows]
    O4, L4 = ora.decode_forward_paged_fp8(q, kp, vp, ks, vs, bt, lens, sc)
    assert np.allclose(O4, O, rtol=1e-13, atol=1e-13) and np.allclose(L4, L, rtol=1e-13, atol=1e-13)


def pin_fp8_prefill(ora):
    """fp8 Q/K/V prefill: brute force (math.fsum) on the values decoded from the
    format definition for a tiny GQA case under causal and window masks, the
    folding of q_scale * k_scale into the score scale and of v_scale into O, and
    sampled rows == the full forward."""
    rng = np.random.default_rng(17)
    B, Hq, Hkv, Nq, Nk, D = 1, 4, 2, 5, 7, 6
    qc = rng.integers(0, 256, (B, Hq, Nq, D), dtype=np.uint8)
    kc = rng.integers(0, 256, (B, Hkv, Nk, D), dtype=np.uint8)
    vc = rng.integers(0, 256, (B, Hkv, Nk, D), dtype=np.uint8)
    for c in (qc, kc, vc):
        c[(c & 0x7F) == 0x7F] = 0x38         # no NaN codes
    qs, ks, vs, sc = 0.125, 0.03125, 0.5, 0.2

    def val(c):
        c = int(c)
        sgn = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 15, c & 7
        return sgn * ((m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    for causal, window in ((False, 0), (True, 0), (True, 3), (False, 2)):
        O, L = ora.attention_forward_fp8(qc, kc, vc, qs, ks, vs, sc, causal, window)
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            for i in range(Nq):
                vis = [j for j in range(Nk)
                       if (not causal or j <= i + Nk - Nq) and (window <= 0 or j > i + Nk - Nq - window)]
                s = {j: sc * math.fsum(val(qc[0, h, i, d]) * qs * val(kc[0, kh, j, d]) * ks for d in range(D))
                     for j in vis}
                mx = max(s.values())
                w = {j: math.exp(s[j] - mx) for j in vis}
                den = math.fsum(w.values())
                for d in range(D):
                    o = math.fsum(w[j] * val(vc[0, kh, j, d]) * vs for j in vis) / den
                    assert abs(O[0, h, i, d] - o) < 1e-12 * max(1.0, abs(o)), (causal, window, h, i, d)
                assert abs(L[0, h, i] - (mx + math.log(den))) < 1e-12
        O2, L2 = ora.attention_forward_fp8(qc, kc, vc, 1.0, 1.0, vs, sc * qs * ks, causal, window)
        assert np.allclose(O2, O, rtol=1e-13, atol=1e-13) and np.allclose(L2, L, rtol=1e-13, atol=1e-13)
        O3, L3 = ora.attention_forward_fp8(qc, kc, vc, qs, ks, 3 * vs, sc, causal, window)
        assert np.allclose(O3, 3 * O, rtol=1e-13, atol=1e-13) and np.allclose(L3, L, rtol=1e-13, atol=1e-13)
        rows = [(0, 3, 4), (0, 0, 0), (0, 1, 2)]
        Or, Lr = ora.attention_rows_fp8(qc, kc, vc, qs, ks, vs, sc, rows, causal, window)
        for n, (b, h, i) in enumerate(rows):
            assert np.allclose(Or[n], O[b, h, i], rtol=1e-13, atol=1e-13) and abs(Lr[n] - L[b, h, i]) < 1e-12


def pin_softcap_sink(ora):
    """Softcap and sinks: brute force (math.tanh, math.fsum) on tiny inputs with
    causal / window masks and sinks from dominant to -inf, the Q = 0 closed form,
    a row with no visible key, and the reductions to the plain forward."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, Nq, Nk, D = 1, 4, 2, 5, 7, 3
    q = rng.standard_normal((B, Hq, Nq, D)) * 2.0
    k = rng.standard_normal((B, Hkv, Nk, D)) * 2.0
    v = rng.standard_normal((B, Hkv, Nk, D))
    sinks = np.array([0.7, -2.0, 6.0, -np.inf])
    sc, cap = 0.8, 2.5
    for causal, window in ((False, 0), (True, 0), (True, 3), (False, 2)):
        O, L = ora.attention_forward_ext(q, k, v, sc, causal, window, cap, sinks)
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            for i in range(Nq):
                vis = [j for j in range(Nk) if (not causal or j <= i + Nk - Nq)
                       and (window <= 0 or j > i + Nk - Nq - window)]
                s = {j: cap * math.tanh(sc * math.fsum(q[0, h, i, d] * k[0, kh, j, d] for d in range(D)) / cap)
                     for j in vis}
                terms = [math.exp(x) for x in s.values()] + ([math.exp(sinks[h])] if np.isfinite(sinks[h]) else [])
                den = math.fsum(terms)
                for d in range(D):
                    o = math.fsum(math.exp(s[j]) * v[0, kh, j, d] for j in vis) / den if vis else 0.0
                    assert abs(O[0, h, i, d] - o) < 1e-12, (causal, window, h, i, d)
                want = math.log(den) if terms else -math.inf
                assert (L[0, h, i] == want) if not terms else abs(L[0, h, i] - want) < 1e-12
    # Q = 0: every visible softcapped score is 0
    z = np.zeros_like(q)
    O0, L0 = ora.attention_forward_ext(z, k, v, sc, False, 0, cap, sinks)
    for h in range(Hq):
        kh = h // (Hq // Hkv)
        extra = math.exp(sinks[h]) if np.isfinite(sinks[h]) else 0.0
        assert np.allclose(O0[0, h], v[0, kh].sum(axis=0) / (Nk + extra), atol=1e-13)
        assert np.allclose(L0[0, h], math.log(Nk + extra), atol=1e-13)
    # no visible key (causal with Nq > Nk): O = 0, LSE = sink
    q2 = rng.standard_normal((1, Hq, 6, D))
    k2, v2 = rng.standard_normal((1, Hkv, 2, D)), rng.standard_normal((1, Hkv, 2, D))
    O2, L2 = ora.attention_forward_ext(q2, k2, v2, sc, True, 0, cap, sinks)
    for h in range(Hq):
        assert np.all(O2[0, h, :4] == 0.0)
        assert np.all(L2[0, h, :4] == sinks[h])
    # reductions: no cap and no sinks is the plain forward; a huge cap is no cap
    Op, Lp = ora.attention_forward(q, k, v, sc, True, 0)
    Oe, Le = ora.attention_forward_ext(q, k, v, sc, True, 0, 0.0, None)
    assert np.allclose(Oe, Op, atol=1e-14) and np.allclose(Le, Lp, atol=1e-14)
    Oh, Lh = ora.attention_forward_ext(q, k, v, sc, True, 0, 1e9, np.full(Hq, -np.inf))
    assert np.allclose(Oh, Op, atol=1e-9) and np.allclose(Lh, Lp, atol=1e-9)
    # sampled rows agree with the full forward
    rows = [(0, h, i) for h in range(Hq) for i in (0, 2, 4)]
    Or, Lr = ora.attention_rows_ext(q, k, v, sc, rows, True, 3, cap, sinks)
    Of, Lf = ora.attention_forward_ext(q, k, v, sc, True, 3, cap, sinks)
    for n, (b, h, i) in enumerate(rows):
        assert np.allclose(Or[n], Of[b, h, i], atol=1e-14) and abs(Lr[n] - Lf[b, h, i]) < 1e-14


def pin_backward(ora):
    """Backward: central finite differences of the loss sum(dO * O) through the
    oracle's own forward, and float64 autograd through torch's SDPA (GQA by
    repeated K/V heads), causal, windowed and dense."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, Nq, Nk, D = 1, 4, 2, 5, 6, 3
    q, k, v = (rng.standard_normal(sh) for sh in ((B, Hq, Nq, D), (B, Hkv, Nk, D), (B, Hkv, Nk, D)))
    do = rng.standard_normal((B, Hq, Nq, D))
    sc, eps = 0.6, 1e-6
    for causal, window in ((False, 0), (True, 0), (True, 3)):
        dQ, dK, dV = ora.attention_backward(q, k, v, do, sc, causal, window)
        loss = lambda qq, kk, vv: float((ora.attention_forward(qq, kk, vv, sc, causal, window)[0] * do).sum())  # noqa: E731
        for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
            for idx in [(0, 0, 0, 0), (0, 1, 2, 1), (0, Hkv - 1, 4, 2), (0, 0, 3, 2)]:
                if idx[1] >= x.shape[1] or idx[2] >= x.shape[2]:
                    continue
                xp, xm = x.copy(), x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                assert abs(fd - g[idx]) < 1e-7 * max(1.0, abs(fd)), (causal, window, name, idx, fd, g[idx])
    for causal in (False, True):
        B, Hq, Hkv, N, D = 2, 4, 2, 9, 8
        q, k, v, do = (rng.standard_normal(sh) for sh in ((B, Hq, N, D), (B, Hkv, N, D), (B, Hkv, N, D), (B, Hq, N, D)))
        tq = torch.tensor(q, requires_grad=True)
        tk = torch.tensor(k, requires_grad=True)
        tv = torch.tensor(v, requires_grad=True)
        out = torch.nn.functional.scaled_dot_product_attention(
            tq, tk.repeat_interleave(2, dim=1), tv.repeat_interleave(2, dim=1), is_causal=causal, scale=0.4)
        out.backward(torch.tensor(do))
        dQ, dK, dV = ora.attention_backward(q, k, v, do, 0.4, causal, 0)
        for mine, ref in ((dQ, tq.grad), (dK, tk.grad), (dV, tv.grad)):
            assert np.allclose(mine, ref.numpy(), rtol=0, atol=1e-12)


PINS = [pin_brute_force, pin_sdpa, pin_zero_query, pin_single_key, pin_probability_rows,
        pin_causal_first_row, pin_dominant_key, pin_invariants, pin_decode, pin_paged_decode, pin_varlen,
        pin_golden, pin_e4m3_codes, pin_fp8_decode, pin_fp8_prefill, pin_softcap_sink, pin_backward]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(ORA)


# ---------------------------------------------------------------- mutation
def _mut_no_scale(q_rows, k_head, scale):
    return q_rows @ k_head.T


def _mut_sqrt_scale(q_rows, k_head, scale):
    return math.sqrt(scale) * (q_rows @ k_head.T)


def _mut_kv_head_modulo(h, Hq, Hkv):
    return h % Hkv


def _mut_causal_top_left(rows, Nq, Nk, causal, window):
    i = np.asarray(rows)[:, None]
    j = np.arange(Nk)[None, :]
    vis = np.ones((i.shape[0], Nk), bool)
    if causal:
        vis &= j <= i
    if window > 0:
        vis &= j > i + Nk - Nq - window
    return vis


def _mut_causal_strict(rows, Nq, Nk, causal, window):
    i = np.asarray(rows)[:, None]
    j = np.arange(Nk)[None, :]
    vis = np.ones((i.shape[0], Nk), bool)
    if causal:
        vis &= j < i + Nk - Nq
    if window > 0:
        vis &= j > i + Nk - Nq - window
    return vis


def _mut_window_wide(rows, Nq, Nk, causal, window):
    i = np.asarray(rows)[:, None]
    j = np.arange(Nk)[None, :]
    vis = np.ones((i.shape[0], Nk), bool)
    if causal:
        vis &= j <= i + Nk - Nq
    if window > 0:
        vis &= j >= i + Nk - Nq - window
    return vis


def _wrap_softmax(kind):
    good = ORA._softmax_rows

    def bad(S):
        P, lse = good(S)
        if kind == "log2":
            return P, lse / math.log(2)
        if kind == "no_max":
            M = np.where(np.isfinite(S.max(axis=1)), S.max(axis=1), 0.0)
            return P, lse - M
        if kind == "key_axis_swapped":
            E = np.exp(S - np.where(np.isfinite(S), S, -np.inf).max(axis=0, keepdims=True))
            E = np.nan_to_num(E)
            with np.errstate(invalid="ignore", divide="ignore"):
                P2 = np.nan_to_num(E / E.sum(axis=0, keepdims=True))
            return P2, lse
        raise AssertionError(kind)
    return bad


def _mut_combine_unweighted(O_part, LSE_part, n_split):
    O_part, LSE_part = np.asarray(O_part), np.asarray(LSE_part)
    B, Hq, _, D = O_part.shape
    O = np.zeros((B, Hq, D))
    L = np.zeros((B, Hq))
    for b in range(B):
        n = int(n_split[b])
        O[b] = O_part[b, :, :n].mean(axis=1)
        L[b] = np.log(np.exp(LSE_part[b, :, :n]).sum(axis=1))
    return O, L


def _mut_paged_rows_swapped(pages, block_table_b, n):
    page_size = pages.shape[1]
    j = np.arange(n)
    page = np.asarray(block_table_b)[j % page_size] if n else np.zeros(0, dtype=int)
    return np.asarray(pages[page, j // page_size], dtype=np.float64) if n else np.zeros((0,) + tuple(pages.shape[2:]))


def _mut_e4m3_bias8(codes):
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -7, (1.0 + m / 8.0) * np.exp2((e - 8).astype(np.float64)))
    return sign * np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)


def _mut_e4m3_no_subnormals(codes):
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, (c & 0x7).astype(np.float64)
    mag = (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64))
    return sign * np.where((e == 15) & (c & 0x7 == 7), np.nan, mag)


def _mut_fp8_paged_swapped(q, k_pages, v_pages, k_scale, v_scale, block_table, seqlens, scale, batches=None):
    kp, vp = np.asarray(k_pages), np.asarray(v_pages)
    page = kp.shape[1]
    perm = [np.asarray(block_table)[b] for b in range(len(seqlens))]
    B, Hq, D = q.shape
    kc = np.zeros((B, int(max(seqlens)), kp.shape[2], kp.shape[3]), dtype=np.uint8)
    vc = np.zeros_like(kc)
    for b, n in enumerate(int(x) for x in seqlens):
        j = np.arange(n)
        kc[b, :n] = kp[perm[b][j % page] % kp.shape[0], j // page]
        vc[b, :n] = vp[perm[b][j % page] % vp.shape[0], j // page]
    return ORA.decode_forward_fp8(q, kc, vc, k_scale, v_scale, seqlens, scale, batches)


def _mut_fp8_prefill_scales_swapped(q_codes, k_codes, v_codes, q_scale, k_scale, v_scale, scale,
                                    causal=False, window=0):
    return _GOOD_FP8_PREFILL(q_codes, k_codes, v_codes, q_scale, v_scale, k_scale, scale, causal, window)


def _mut_softcap_no_divide(S, cap):
    if not cap > 0:
        return S
    with np.errstate(invalid="ignore"):
        return np.where(np.isneginf(S), -np.inf, cap * np.tanh(S))


def _mut_sink_unshifted(S, sink):
    M = S.max(axis=1)
    empty = ~np.isfinite(M)
    M_safe = np.where(empty, 0.0, M)
    E = np.exp(S - M_safe[:, None])
    l = E.sum(axis=1) + np.exp(sink)
    with np.errstate(divide="ignore", invalid="ignore"):
        P = np.where(empty[:, None], 0.0, E / np.where(empty, 1.0, l)[:, None])
        lse = np.where(empty, -np.inf, M_safe + np.log(np.where(empty, 1.0, l)))
    return P, lse


def _mut_sink_dropped(S, sink):
    return ORA._softmax_rows(S)


def _mut_bwd_no_dsum(Qh, Kh, Vh, dOh, scale, vis):
    S = ORA._scores(Qh, Kh, scale)
    S[~vis] = -np.inf
    P, _ = ORA._softmax_rows(S)
    dS = P * (dOh @ Vh.T)
    return scale * (dS @ Kh), scale * (dS.T @ Qh), P.T @ dOh


def _mut_bwd_dk_unscaled(Qh, Kh, Vh, dOh, scale, vis):
    S = ORA._scores(Qh, Kh, scale)
    S[~vis] = -np.inf
    P, _ = ORA._softmax_rows(S)
    dP = dOh @ Vh.T
    dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
    return scale * (dS @ Kh), dS.T @ Qh, P.T @ dOh


def _mut_bwd_dv_untransposed(Qh, Kh, Vh, dOh, scale, vis):
    gq, gk, gv = _GOOD_BWD(Qh, Kh, Vh, dOh, scale, vis)
    S = ORA._scores(Qh, Kh, scale)
    S[~vis] = -np.inf
    P, _ = ORA._softmax_rows(S)
    if P.shape[0] == P.shape[1]:
        return gq, gk, P @ dOh
    return gq, gk, (P.T @ dOh)[::-1]


_GOOD_BWD = ORA._backward_head
_GOOD_FP8_PREFILL = ORA.attention_forward_fp8


MUTANTS = {
    "no_scale": ("_scores", _mut_no_scale),
    "sqrt_scale": ("_scores", _mut_sqrt_scale),
    "kv_head_modulo": ("kv_head", _mut_kv_head_modulo),
    "causal_top_left": ("visible_mask", _mut_causal_top_left),
    "causal_strict": ("visible_mask", _mut_causal_strict),
    "window_off_by_one": ("visible_mask", _mut_window_wide),
    "lse_log2": ("_softmax_rows", _wrap_softmax("log2")),
    "lse_missing_max": ("_softmax_rows", _wrap_softmax("no_max")),
    "softmax_over_queries": ("_softmax_rows", _wrap_softmax("key_axis_swapped")),
    "combine_unweighted": ("decode_combine", _mut_combine_unweighted),
    "paged_index_swapped": ("paged_rows", _mut_paged_rows_swapped),
    "e4m3_bias_8": ("e4m3_to_float", _mut_e4m3_bias8),
    "e4m3_no_subnormals": ("e4m3_to_float", _mut_e4m3_no_subnormals),
    "fp8_paged_index_swapped": ("decode_forward_paged_fp8", _mut_fp8_paged_swapped),
    "fp8_prefill_k_v_scales_swapped": ("attention_forward_fp8", _mut_fp8_prefill_scales_swapped),
    "softcap_without_divide": ("softcap_scores", _mut_softcap_no_divide),
    "sink_unshifted": ("_softmax_rows_sink", _mut_sink_unshifted),
    "sink_dropped": ("_softmax_rows_sink", _mut_sink_dropped),
    "bwd_missing_rowsum_term": ("_backward_head", _mut_bwd_no_dsum),
    "bwd_dk_unscaled": ("_backward_head", _mut_bwd_dk_unscaled),
    "bwd_dv_untransposed": ("_backward_head", _mut_bwd_dv_untransposed),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(ORA, attr, fn)
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(ORA)
        except (AssertionError, ValueError, IndexError, ZeroDivisionError):
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
