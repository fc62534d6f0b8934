"""Gradients of masked grouped-query attention, in float64 (test infrastructure only).

The pages measure the training step of packed-document attention forward and
backward ([FASTLLM] Summary and its timing tables, "fwd+bwd" at head size 512)
but print no formula for the backward pass.  The gradient is fixed by the
forward definition alone, so this module writes out its derivative.  For one
query row ``i`` and query head ``h`` with allowed keys ``A_i`` (increasing
order), key/value head ``g = h // G``, and the upstream gradient ``do = dL/do_ih``:

    s_k   = scale * <q_ih, k_kg>             k in A_i
    p     = softmax(s)                       (max subtracted, exact)
    o_ih  = sum_k p_k v_kg
    dp_k  = <do, v_kg>                       dL/dp_k
    delta = <do, o_ih> = sum_k p_k dp_k
    ds_k  = p_k (dp_k - delta)               dL/ds_k  (softmax Jacobian)
    dq_ih      = scale * sum_k ds_k k_kg
    dk_kg     += scale * ds_k q_ih           (summed over the G heads of group g)
    dv_kg     += p_k do                      (summed over the G heads of group g)

Only ``o`` is differentiated (``lse`` is an auxiliary output).  A row with no
allowed key has the constant output 0, so it contributes nothing.  Query heads
that share a key/value head add their contributions: that is the derivative of
repeating K/V across the group ([FASTLLM] Summary: K/V repeated per query head
with repeat_interleave).
"""

from __future__ import annotations

import numpy as np


def masked_attention_backward(q, k, v, mask, scale: float, do):
    """q, do [Sq, Hq, D]; k, v [Sk, Hkv, D]; mask [Sq, Sk] bool (all float64).

    Returns dq [Sq, Hq, D], dk [Sk, Hkv, D], dv [Sk, Hkv, D] in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    sq, hq, d = q.shape
    hkv = k.shape[1]
    if hq % hkv:
        raise ValueError("query heads must be a multiple of key/value heads")
    g = hq // hkv
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    for i in range(sq):
        idx = np.flatnonzero(mask[i])
        if idx.size == 0:
            continue
        for h in range(hq):
            kh = k[idx, h // g, :]
            vh = v[idx, h // g, :]
            s = scale * (kh @ q[i, h])
            e = np.exp(s - s.max())
            p = e / e.sum()
            o = p @ vh
            dp = vh @ do[i, h]
            ds = p * (dp - do[i, h] @ o)
            dq[i, h] = scale * (ds @ kh)
            dk[idx, h // g, :] += scale * np.outer(ds, q[i, h])
            dv[idx, h // g, :] += np.outer(p, do[i, h])
    return dq, dk, dv


def masked_attention_backward_heads(q, k, v, mask, scale: float, do):
    """The same gradients in matrix form, one query head at a time, for a
    subset of query rows.

    q, do [Sq, Hq, D] are the selected query rows, mask [Sq, Sk] their rows of
    the mask, k, v [Sk, Hkv, D] every key.  Per head, with masked entries of P
    zero: S = scale Q K^T, P = softmax over each row's allowed keys,
    dP = dO V^T, delta = rowsum(P * dP), dS = P * (dP - delta),
    dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.  Returns dq [Sq, Hq, D]
    and the selected rows' contributions to dk, dv [Sk, Hkv, D]: exact for
    every key that only the selected rows admit.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    hq = q.shape[1]
    hkv = k.shape[1]
    g = hq // hkv
    mask = np.asarray(mask, dtype=bool)
    live = mask.any(axis=1)
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(v.shape, dtype=np.float64)
    for h in range(hq):
        kh, vh = k[:, h // g, :], v[:, h // g, :]
        s = np.where(mask, scale * (q[:, h, :] @ kh.T), -np.inf)
        m = np.where(live, s.max(axis=1), 0.0)
        e = np.where(mask, np.exp(s - m[:, None]), 0.0)
        tot = e.sum(axis=1)
        p = e / np.where(live, tot, 1.0)[:, None]
        dp = do[:, h, :] @ vh.T
        delta = (p * dp).sum(axis=1)
        ds = p * (dp - delta[:, None])
        dq[:, h, :] = scale * (ds @ kh)
        dk[:, h // g, :] += scale * (ds.T @ q[:, h, :])
        dv[:, h // g, :] += p.T @ do[:, h, :]
    return dq, dk, dv
