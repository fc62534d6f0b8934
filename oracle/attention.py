"""Masked softmax attention with grouped-query heads, in float64 (test infrastructure only).

For a query row ``i`` and query head ``h`` the key/value head is
``h // G`` with ``G = Hq / Hkv``: each key/value head serves G consecutive
query heads, which is what repeating K/V with ``repeat_interleave`` across the
query heads computes ([FASTLLM] Summary: its SDPA paths copy every K/V head
once per query head of its group).

    allowed keys  A_i = { k : mask[i, k] }            (in increasing k order)
    s_k  = scale * <q_ih, k_k>                         k in A_i
    o_ih = sum_k softmax(s)_k * v_k
    lse_ih = log sum_k exp(s_k)

Softmax is evaluated with the maximum subtracted (exact in real arithmetic).
A row with no allowed key has output 0 and lse = -inf (a reading: the pages
give pad queries no output).  Keys are gathered in increasing index order
before any arithmetic, so two calls that see the same allowed keys in the
same order give bit-identical results, however many masked keys surround them.
"""

from __future__ import annotations

import math

import numpy as np


def attend_row(qv: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float):
    """One query vector against an explicit key/value list: returns (o, lse)."""
    s = scale * (keys @ qv)
    m = s.max()
    e = np.exp(s - m)
    l = e.sum()
    o = (e @ values) / l
    return o, m + math.log(l)


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray, scale: float):
    """q [Sq, Hq, D], k/v [Sk, Hkv, D] (float64), mask [Sq, Sk] bool.

    Returns o [Sq, Hq, D] float64 and lse [Sq, Hq] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    sq, hq, d = q.shape
    hkv = k.shape[1]
    if hq % hkv:
        raise ValueError("query heads must be a multiple of key/value heads")
    g = hq // hkv
    o = np.zeros((sq, hq, d), dtype=np.float64)
    lse = np.full((sq, hq), -np.inf, dtype=np.float64)
    for i in range(sq):
        idx = np.flatnonzero(mask[i])
        if idx.size == 0:
            continue
        for h in range(hq):
            kh = np.ascontiguousarray(k[idx, h // g, :])
            vh = np.ascontiguousarray(v[idx, h // g, :])
            o[i, h], lse[i, h] = attend_row(q[i, h], kh, vh, scale)
    return o, lse


def masked_attention_loops(q, k, v, mask, scale):
    """Pure-Python brute force of :func:`masked_attention` (tiny inputs only).

    Every sum is an explicit loop and every exponential is ``math.exp``; no
    max subtraction, so it also checks that the stabilised form is exact.
    """
    sq, hq, d = len(q), len(q[0]), len(q[0][0])
    hkv = len(k[0])
    g = hq // hkv
    o = [[[0.0] * d for _ in range(hq)] for _ in range(sq)]
    lse = [[-math.inf] * hq for _ in range(sq)]
    for i in range(sq):
        for h in range(hq):
            weights = []
            for j in range(len(k)):
                if mask[i][j]:
                    dot = 0.0
                    for c in range(d):
                        dot += float(q[i][h][c]) * float(k[j][h // g][c])
                    weights.append((j, math.exp(scale * dot)))
            if not weights:
                continue
            total = sum(w for _, w in weights)
            for c in range(d):
                acc = 0.0
                for j, w in weights:
                    acc += w * float(v[j][h // g][c])
                o[i][h][c] = acc / total
            lse[i][h] = math.log(total)
    return np.array(o), np.array(lse)
