"""Whole-workload oracle drivers (test infrastructure only).

They compose the predicate (``masks``), fp64 attention (``attention``) and the
compact-cache index model (``compact``):

* :func:`prefill`          -- every query of a left-padded batch against the
                              full prompt (chunking does not change the result:
                              keys of later chunks are never allowed, except
                              future same-image keys, and image blocks never
                              straddle a chunk).
* :func:`prefill_rows`     -- the same for selected query rows only.
* :func:`varlen_rows`      -- packed documents given by cu_seqlens.
* :func:`prefill_backward` -- gradients of a left-padded batch's attention
                              (q, k, v) for an upstream gradient of the output.
* :func:`varlen_backward`  -- the same for packed documents.
* :func:`varlen_backward_rows` -- packed documents, selected query rows: their
                              dq and their contributions to dk, dv.
* :func:`decode_full`      -- the decode loop over a full-length cache that is
                              never compacted (positions 0 .. S+T-1).
* :func:`decode_compact`   -- the same decode loop through the compact W+64
                              cache, its runtime mask and rolls.

All inputs are converted to float64 (bf16 values widen exactly).
"""

from __future__ import annotations

import numpy as np

from . import attention, backward, masks
from .compact import CompactModel, RingModel


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor (any dtype): widen exactly
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def prefill(q, k, v, window: int, scale: float, valid_start=None, img=None):
    """q [B, S, Hq, D], k/v [B, S, Hkv, D] -> o [B, S, Hq, D], lse [B, S, Hq]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    b_count, s = q.shape[0], q.shape[1]
    vs = np.zeros(b_count, dtype=np.int64) if valid_start is None else np.asarray(valid_start)
    o = np.zeros(q.shape, dtype=np.float64)
    lse = np.zeros(q.shape[:3], dtype=np.float64)
    for b in range(b_count):
        img_b = None if img is None else np.asarray(img[b])
        m = masks.prefill_mask(s, window, int(vs[b]), img_b)
        o[b], lse[b] = attention.masked_attention(q[b], k[b], v[b], m, scale)
    return o, lse


def prefill_rows(q, k, v, window: int, scale: float, b: int, rows, valid_start=None, img=None):
    """Selected query rows of sequence ``b``: o [len(rows), Hq, D], lse [len(rows), Hq]."""
    s = k.shape[1]
    vs = 0 if valid_start is None else int(np.asarray(valid_start)[b])
    img_b = None if img is None else np.asarray(img[b])
    m = masks.prefill_mask(s, window, vs, img_b, None, rows=list(rows))
    return attention.masked_attention(_f64(q[b][list(rows)]), _f64(k[b]), _f64(v[b]), m, scale)


def varlen_rows(q, k, v, cu_seqlens, window: int, scale: float, rows):
    """Packed documents: q [T, Hq, D], k/v [T, Hkv, D]; selected rows."""
    total = k.shape[0]
    doc = masks.doc_ids_from_cu_seqlens(cu_seqlens, total)
    m = masks.prefill_mask(total, window, 0, None, doc, rows=list(rows))
    return attention.masked_attention(_f64(q[list(rows)]), _f64(k), _f64(v), m, scale)


def prefill_backward(q, k, v, dout, window: int, scale: float, valid_start=None, img=None):
    """q, dout [B, S, Hq, D], k/v [B, S, Hkv, D] -> dq [B, S, Hq, D], dk, dv [B, S, Hkv, D]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    b_count, s = q.shape[0], q.shape[1]
    vs = np.zeros(b_count, dtype=np.int64) if valid_start is None else np.asarray(valid_start)
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    for b in range(b_count):
        img_b = None if img is None else np.asarray(img[b])
        m = masks.prefill_mask(s, window, int(vs[b]), img_b)
        dq[b], dk[b], dv[b] = backward.masked_attention_backward(q[b], k[b], v[b], m, scale, dout[b])
    return dq, dk, dv


def varlen_backward(q, k, v, dout, cu_seqlens, window: int, scale: float):
    """Packed documents: q, dout [T, Hq, D], k/v [T, Hkv, D] -> dq, dk, dv."""
    total = k.shape[0]
    doc = masks.doc_ids_from_cu_seqlens(cu_seqlens, total)
    m = masks.prefill_mask(total, window, 0, None, doc)
    return backward.masked_attention_backward(_f64(q), _f64(k), _f64(v), m, scale, _f64(dout))


def varlen_backward_rows(q, k, v, dout, cu_seqlens, window: int, scale: float, rows):
    """Packed documents, selected query rows (matrix form per head): dq of
    those rows [len(rows), Hq, D], and dk, dv [T, Hkv, D] summed over those
    rows only -- exact for keys that no other query admits."""
    total = k.shape[0]
    rows = list(rows)
    doc = masks.doc_ids_from_cu_seqlens(cu_seqlens, total)
    m = masks.prefill_mask(total, window, 0, None, doc, rows=rows)
    return backward.masked_attention_backward_heads(_f64(q[rows]), _f64(k), _f64(v), m, scale, _f64(dout[rows]))


def decode_full(prompt_k, prompt_v, dec_q, dec_k, dec_v, prompt_len: int, window: int,
                scale: float, valid_start=None, steps=None):
    """Decode loop over a full-length cache.

    prompt_k/v [B, P, Hkv, D] hold positions [S - P, S) of the prompt
    (P = S for a whole prompt).  dec_q [T, B, Hq, D], dec_k/v [T, B, Hkv, D]
    are the decode tokens at positions S, S+1, ...  Returns
    o [T, B, Hq, D] and lse [T, B, Hq] for the requested steps (default all).
    """
    pk, pv = _f64(prompt_k), _f64(prompt_v)
    dq, dk, dv = _f64(dec_q), _f64(dec_k), _f64(dec_v)
    t_count, b_count = dq.shape[0], dq.shape[1]
    p_rows = pk.shape[1]
    start = prompt_len - p_rows
    vs = np.zeros(b_count, dtype=np.int64) if valid_start is None else np.asarray(valid_start)
    steps = range(t_count) if steps is None else steps
    o = np.zeros(dq.shape, dtype=np.float64)
    lse = np.full(dq.shape[:3], -np.inf, dtype=np.float64)
    for t in steps:
        p = prompt_len + t
        for b in range(b_count):
            keys = np.concatenate([pk[b], dk[:t + 1, b]], axis=0)
            vals = np.concatenate([pv[b], dv[:t + 1, b]], axis=0)
            # key i of this list is at position start + i
            positions = start + np.arange(keys.shape[0])
            allow = masks.decode_mask_full(p, window, int(vs[b]), positions)
            ob, lb = attention.masked_attention(dq[t, b][None], keys, vals, allow[None, :], scale)
            o[t, b], lse[t, b] = ob[0], lb[0]
    return o, lse


def decode_compact(prompt_k, prompt_v, dec_q, dec_k, dec_v, prompt_len: int, window: int,
                   scale: float, valid_start=None, on_step=None, ring: bool = False):
    """The same decode loop through the compact cache model (or, with
    ``ring``, through the modular ring model).

    The compact cache of each sequence is materialised from the model's
    row -> position map; the runtime mask comes from the model.  ``on_step``
    (optional) is called as ``on_step(t, model, mask)`` after each mask build.
    """
    pk, pv = _f64(prompt_k), _f64(prompt_v)
    dq, dk, dv = _f64(dec_q), _f64(dec_k), _f64(dec_v)
    t_count, b_count = dq.shape[0], dq.shape[1]
    p_rows = pk.shape[1]
    start = prompt_len - p_rows
    vs = np.zeros(b_count, dtype=np.int64) if valid_start is None else np.asarray(valid_start)
    model = RingModel(prompt_len, window) if ring else CompactModel(prompt_len, window)
    o = np.zeros(dq.shape, dtype=np.float64)
    lse = np.full(dq.shape[:3], -np.inf, dtype=np.float64)
    for t in range(t_count):
        if model.needs_roll():
            model.roll()
        mask = model.begin_step(vs)
        if on_step is not None:
            on_step(t, model, mask)
        for b in range(b_count):
            # keys by position, from the first stored prompt position on
            lo = max(start, 0)
            full_k = np.concatenate([pk[b][lo - start:], dk[:t + 1, b]], axis=0)
            full_v = np.concatenate([pv[b][lo - start:], dv[:t + 1, b]], axis=0)
            ck = model.expected_cache(full_k, lo)
            cv = model.expected_cache(full_v, lo)
            ob, lb = attention.masked_attention(dq[t, b][None], ck, cv, mask[b][None, :], scale)
            o[t, b], lse[t, b] = ob[0], lb[0]
    return o, lse
