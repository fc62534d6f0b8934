"""Pins of the oracle's fp64 attention gradients (CPU only).

The backward oracle is the chain rule written out, so each pin checks it
against something that does not use those formulas:

* central finite differences of the forward oracle's loss sum(dout * o)
  (the forward is pinned on its own), on tiny inputs;
* a library routine: torch autograd through scaled_dot_product_attention in
  float64 on the CPU with the boolean mask (rows with at least one key);
* invariants that hold for any mask: the key gradients of one key/value head
  sum to zero (softmax is unchanged when every score of a row moves by the
  same amount), and the value gradients sum to the upstream gradients of the
  non-empty rows;
* closed forms: W = 1 (each row sees only itself) gives dq = dk = 0 and
  dv = the sum of the group's upstream gradients; pad rows and pad keys get
  zero gradients and pad rows' upstream gradients change nothing;
* GQA: the Hkv-head gradients equal the repeated-K/V gradients summed over
  each group; packed documents equal each document on its own, bit for bit;
* the matrix form (one head at a time, optionally a subset of query rows)
  equals the row-by-row form.
"""

import numpy as np
import torch

from oracle import attention, backward, masks, reference


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _loss(q, k, v, m, scale, do):
    o, _ = attention.masked_attention(q, k, v, m, scale)
    return float((o * do).sum())


def test_against_finite_differences():
    rng = np.random.default_rng(10)
    n, hq, hkv, d, w = 7, 4, 2, 3, 4
    q, k, v, do = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d), _rand(rng, n, hq, d)
    img = np.full(n, -1)
    img[3:6] = 0  # one image block: future same-image keys are allowed
    m = masks.prefill_mask(n, w, 1, img)
    scale = 0.71
    dq, dk, dv = backward.masked_attention_backward(q, k, v, m, scale, do)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            keep = x[idx]
            x[idx] = keep + eps
            lp = _loss(q, k, v, m, scale, do)
            x[idx] = keep - eps
            lm = _loss(q, k, v, m, scale, do)
            x[idx] = keep
            num[idx] = (lp - lm) / (2 * eps)
        assert np.allclose(g, num, rtol=0, atol=1e-7), np.abs(g - num).max()


def test_against_torch_autograd_float64():
    rng = np.random.default_rng(11)
    n, hq, hkv, d, w = 41, 4, 2, 16, 13
    q, k, v, do = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d), _rand(rng, n, hq, d)
    doc = masks.doc_ids_from_cu_seqlens([0, 17, 30, 41], n)
    m = masks.prefill_mask(n, w, 0, None, doc)
    assert m.any(axis=1).all()  # no empty row: SDPA would give NaN there
    scale = d ** -0.5
    dq, dk, dv = backward.masked_attention_backward(q, k, v, m, scale, do)
    tq = torch.from_numpy(q).requires_grad_()
    tk = torch.from_numpy(k).requires_grad_()
    tv = torch.from_numpy(v).requires_grad_()
    g = hq // hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.repeat_interleave(g, dim=1).permute(1, 0, 2)[None],
        tv.repeat_interleave(g, dim=1).permute(1, 0, 2)[None], attn_mask=torch.from_numpy(m), scale=scale)
    o[0].permute(1, 0, 2).backward(torch.from_numpy(do))
    assert np.allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


def test_gradient_sums_for_any_mask():
    rng = np.random.default_rng(12)
    n, hq, hkv, d, w = 60, 6, 2, 8, 9
    q, k, v, do = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d), _rand(rng, n, hq, d)
    img = np.full(n, -1)
    img[20:31] = 0  # longer than W: old same-image pairs are rejected
    img[31:35] = 1
    m = masks.prefill_mask(n, w, 5, img)
    dq, dk, dv = backward.masked_attention_backward(q, k, v, m, 0.4, do)
    assert np.abs(dk.sum(axis=0)).max() < 1e-11
    rows = m.any(axis=1)
    g = hq // hkv
    want = do[rows].reshape(rows.sum(), hkv, g, d).sum(axis=(0, 2))
    assert np.allclose(dv.sum(axis=0), want, rtol=0, atol=1e-11)


def test_window_one_closed_form_and_padding():
    rng = np.random.default_rng(13)
    n, hq, hkv, d, vs = 12, 4, 2, 5, 3
    q, k, v, do = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d), _rand(rng, n, hq, d)
    m = masks.prefill_mask(n, 1, vs)
    dq, dk, dv = backward.masked_attention_backward(q, k, v, m, 0.5, do)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    want = do.reshape(n, hkv, hq // hkv, d).sum(axis=2)
    want[:vs] = 0.0
    assert np.allclose(dv, want, rtol=0, atol=1e-15)
    # a sliding window with padding: pad rows and pad keys get zero gradients, and
    # the pad rows' upstream gradients change nothing
    m = masks.prefill_mask(n, 4, vs)
    g1 = backward.masked_attention_backward(q, k, v, m, 0.5, do)
    do2 = do.copy()
    do2[:vs] = 1e6
    g2 = backward.masked_attention_backward(q, k, v, m, 0.5, do2)
    for a, b in zip(g1, g2):
        assert np.array_equal(a, b)
    assert np.all(g1[0][:vs] == 0.0) and np.all(g1[1][:vs] == 0.0) and np.all(g1[2][:vs] == 0.0)


def test_gqa_equals_repeated_heads_summed():
    rng = np.random.default_rng(14)
    n, hq, hkv, d, w = 25, 6, 3, 7, 8
    q, k, v, do = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d), _rand(rng, n, hq, d)
    m = masks.prefill_mask(n, w, 2)
    dq, dk, dv = backward.masked_attention_backward(q, k, v, m, 0.3, do)
    g = hq // hkv
    rq, rk, rv = backward.masked_attention_backward(q, np.repeat(k, g, axis=1), np.repeat(v, g, axis=1), m, 0.3, do)
    assert np.array_equal(dq, rq)
    assert np.allclose(dk, rk.reshape(n, hkv, g, d).sum(axis=2), rtol=0, atol=1e-12)
    assert np.allclose(dv, rv.reshape(n, hkv, g, d).sum(axis=2), rtol=0, atol=1e-12)


def test_packed_documents_equal_each_document_alone():
    rng = np.random.default_rng(15)
    cu = [0, 9, 30, 34, 50]
    n, hq, hkv, d, w = cu[-1], 4, 2, 6, 10
    q, k, v, do = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d), _rand(rng, n, hq, d)
    dq, dk, dv = reference.varlen_backward(q, k, v, do, cu, w, 0.45)
    for a, b in zip(cu[:-1], cu[1:]):
        m = masks.prefill_mask(b - a, w)
        eq, ek, ev = backward.masked_attention_backward(q[a:b], k[a:b], v[a:b], m, 0.45, do[a:b])
        assert np.array_equal(dq[a:b], eq) and np.array_equal(dk[a:b], ek) and np.array_equal(dv[a:b], ev)


def test_matrix_form_equals_row_form():
    rng = np.random.default_rng(16)
    n, hq, hkv, d, w = 70, 4, 2, 9, 12
    q, k, v, do = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d), _rand(rng, n, hq, d)
    img = np.full(n, -1)
    img[40:55] = 0
    m = masks.prefill_mask(n, w, 6, img)
    want = backward.masked_attention_backward(q, k, v, m, 0.35, do)
    got = backward.masked_attention_backward_heads(q, k, v, m, 0.35, do)
    for a, b in zip(want, got):
        assert np.allclose(a, b, rtol=0, atol=1e-12)
    # a subset of rows: exact dq for them, and exact dk / dv for the keys only
    # they admit (the last 5 keys are admitted only by the last 5 queries here)
    rows = list(range(n - 5, n))
    gq, gk, gv = backward.masked_attention_backward_heads(q[rows], k, v, m[rows], 0.35, do[rows])
    assert np.allclose(gq, want[0][rows], rtol=0, atol=1e-12)
    assert not m[:n - 5, n - 5:].any()
    assert np.allclose(gk[n - 5:], want[1][n - 5:], rtol=0, atol=1e-12)
    assert np.allclose(gv[n - 5:], want[2][n - 5:], rtol=0, atol=1e-12)
