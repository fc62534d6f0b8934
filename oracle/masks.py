"""Sliding-layer masks, written out literally (test infrastructure only).

The predicate for a query at padded position ``q`` and a key at padded
position ``k`` of the same sequence:

    allowed(q, k) =  k >= valid_start and q >= valid_start      (left padding)
                 and doc(q) == doc(k)                          (packed documents)
                 and q - k < W                                  (sliding window)
                 and (k <= q or (img(q) >= 0 and img(q) == img(k)))
                                                                (causal OR same image)

Sources:
  * sliding layers admit a key inside the window that is causal or in the
    query's image block, global layers stay causal: [SPYRE] Summary, the bullet on matching the Transformers VLM
    mask composition.
  * future same-image pairs are allowed, old same-image pairs outside the
    window are rejected: [SPYRE] Correctness, the mask-order regression bullet.
  * left padding is preserved: [SPYRE] Summary.
  * causal + document mask for packed documents given by cu_seqlens:
    [FASTLLM] Summary (the dense attn_mask path and preprocessing).
  * vision vs text token types: [BONSAI] discussion of the Gemma3 mask.

Readings where the pages are silent (listed again in the design notes):
  * the window holds W keys including the query itself (0 <= q - k < W);
  * the window is one-sided, so future same-image keys always pass it;
  * an image is a contiguous run of one non-negative id; ``img == -1`` is text;
  * pad queries attend to nothing (their output is defined as zero).
"""

from __future__ import annotations

import numpy as np


def allowed(q: int, k: int, window: int, valid_start: int = 0,
            img_q: int = -1, img_k: int = -1, doc_q: int = 0, doc_k: int = 0) -> bool:
    """The sliding-layer predicate for one (query, key) pair, term by term."""
    if q < valid_start or k < valid_start:
        return False
    if doc_q != doc_k:
        return False
    if q - k >= window:
        return False
    if k <= q:
        return True
    return img_q >= 0 and img_q == img_k


def doc_ids_from_cu_seqlens(cu_seqlens, total: int) -> np.ndarray:
    """Document index of every packed token: doc[t] = d for cu[d] <= t < cu[d+1].

    [FASTLLM] Summary: documents of a packed batch are given by cu_seqlens and
    the mask path needs a per-token document index.
    """
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    doc = np.full(total, -1, dtype=np.int64)
    for d in range(len(cu) - 1):
        doc[cu[d]:cu[d + 1]] = d
    if (doc < 0).any():
        raise ValueError("cu_seqlens does not cover every token")
    return doc


def prefill_mask(n: int, window: int, valid_start: int = 0, img=None, doc=None,
                 rows=None) -> np.ndarray:
    """Dense boolean mask of one sequence: [n, n], or [len(rows), n] for selected queries.

    The same predicate as :func:`allowed`, evaluated for every pair at once.
    ``img`` and ``doc`` are per-token arrays (or None for all-text / one
    document); ``rows`` selects query positions (default: all n).
    """
    qi = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    q = qi[:, None]
    k = np.arange(n)[None, :]
    img = np.full(n, -1, dtype=np.int64) if img is None else np.asarray(img, dtype=np.int64)
    doc = np.zeros(n, dtype=np.int64) if doc is None else np.asarray(doc, dtype=np.int64)
    valid = (q >= valid_start) & (k >= valid_start)
    same_doc = doc[qi][:, None] == doc[None, :]
    in_window = (q - k) < window
    causal = k <= q
    same_img = (img[qi][:, None] >= 0) & (img[qi][:, None] == img[None, :])
    return valid & same_doc & in_window & (causal | same_img)


def prefill_mask_loops(n: int, window: int, valid_start: int = 0, img=None, doc=None) -> np.ndarray:
    """Brute-force version of :func:`prefill_mask`: calls :func:`allowed` per pair."""
    img = [-1] * n if img is None else [int(x) for x in img]
    doc = [0] * n if doc is None else [int(x) for x in doc]
    out = np.zeros((n, n), dtype=bool)
    for q in range(n):
        for k in range(n):
            out[q, k] = allowed(q, k, window, valid_start, img[q], img[k], doc[q], doc[k])
    return out


def decode_mask_full(p: int, window: int, valid_start: int, positions) -> np.ndarray:
    """Which of the keys at ``positions`` a decode query at position ``p`` sees.

    Decode queries are text tokens and the current token attends to itself
    (it is appended before attention), so the predicate reduces to
    ``valid_start <= k <= p``, ``k >= 0`` and ``p - k < W``.
    """
    k = np.asarray(positions, dtype=np.int64)
    return (k >= valid_start) & (k >= 0) & (k <= p) & ((p - k) < window) & (p >= valid_start)
