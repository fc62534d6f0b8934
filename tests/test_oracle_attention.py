"""Pins of the oracle's fp64 masked attention (CPU only).

* brute force with pure-Python loops and math.exp on tiny inputs (1e-12);
* a library routine: torch's scaled_dot_product_attention in float64 on the
  CPU with the boolean mask, on rows that have at least one key (1e-12);
* closed forms: W = 1 gives the query's own value row; q = 0 gives the mean of
  the allowed value rows; a single allowed key gives that value row;
* GQA: Hkv heads give bit-identical results to K/V repeated per query head
  (repeat_interleave);
* zero weight: large finite values in masked rows leave outputs bit-identical.
"""

import numpy as np
import pytest
import torch

from oracle import attention, masks


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def test_against_python_loops():
    rng = np.random.default_rng(0)
    for n, hq, hkv, d, w in [(7, 2, 1, 4, 3), (12, 4, 2, 8, 5), (9, 3, 3, 6, 9)]:
        q, k, v = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d)
        img = np.full(n, -1)
        img[2:5] = 0
        m = masks.prefill_mask(n, w, 1, img)
        o, lse = attention.masked_attention(q, k, v, m, 0.37)
        o2, lse2 = attention.masked_attention_loops(q.tolist(), k.tolist(), v.tolist(), m.tolist(), 0.37)
        assert np.allclose(o, o2, rtol=0, atol=1e-12)
        finite = np.isfinite(lse2)
        assert np.array_equal(np.isfinite(lse), finite)
        assert np.allclose(lse[finite], lse2[finite], rtol=0, atol=1e-12)


def test_against_torch_sdpa_float64():
    rng = np.random.default_rng(1)
    n, hq, hkv, d, w = 37, 4, 2, 16, 11
    q, k, v = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d)
    img = np.full(n, -1)
    img[10:16] = 0
    img[16:20] = 1
    m = masks.prefill_mask(n, w, 3, img)
    scale = d ** -0.5
    o, lse = attention.masked_attention(q, k, v, m, scale)
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)[None]
    tv = torch.from_numpy(v).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=torch.from_numpy(m), scale=scale)[0].permute(1, 0, 2).numpy()
    rows = m.any(axis=1)
    assert rows.sum() < n  # the padded rows are empty
    assert np.allclose(o[rows], ref[rows], rtol=0, atol=1e-12)
    assert np.all(o[~rows] == 0.0) and np.all(np.isneginf(lse[~rows]))
    # lse against logsumexp of the masked scores
    s = np.einsum("qhd,khd->hqk", q, np.repeat(k, hq // hkv, axis=1)) * scale
    s = np.where(m[None], s, -np.inf)
    ref_lse = torch.logsumexp(torch.from_numpy(s), dim=-1).numpy().T
    assert np.allclose(lse[rows], ref_lse[rows], rtol=0, atol=1e-12)


def test_window_one_returns_own_value():
    rng = np.random.default_rng(2)
    n, hq, hkv, d = 10, 4, 2, 8
    q, k, v = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d)
    o, _ = attention.masked_attention(q, k, v, masks.prefill_mask(n, 1), 0.5)
    assert np.allclose(o, np.repeat(v, 2, axis=1), rtol=0, atol=1e-15)


def test_zero_query_gives_mean_of_allowed_values():
    rng = np.random.default_rng(3)
    n, d, w = 15, 6, 4
    k, v = _rand(rng, n, 1, d), _rand(rng, n, 1, d)
    m = masks.prefill_mask(n, w)
    o, lse = attention.masked_attention(np.zeros((n, 1, d)), k, v, m, 1.0)
    for i in range(n):
        idx = np.flatnonzero(m[i])
        assert np.allclose(o[i, 0], v[idx, 0].mean(axis=0), rtol=0, atol=1e-14)
        assert abs(lse[i, 0] - np.log(len(idx))) < 1e-14


def test_single_allowed_key():
    rng = np.random.default_rng(4)
    q, k, v = _rand(rng, 3, 2, 5), _rand(rng, 6, 1, 5), _rand(rng, 6, 1, 5)
    m = np.zeros((3, 6), dtype=bool)
    m[0, 4] = m[1, 0] = m[2, 5] = True
    o, lse = attention.masked_attention(q, k, v, m, 2.0)
    for i, j in enumerate([4, 0, 5]):
        assert np.array_equal(o[i, 0], v[j, 0]) and np.array_equal(o[i, 1], v[j, 0])
        assert abs(lse[i, 0] - 2.0 * q[i, 0] @ k[j, 0]) < 1e-13


def test_gqa_equals_repeat_interleave_bitwise():
    rng = np.random.default_rng(5)
    n, hq, hkv, d = 21, 8, 2, 16
    q, k, v = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d)
    m = masks.prefill_mask(n, 6, 2)
    o1, l1 = attention.masked_attention(q, k, v, m, 0.25)
    o2, l2 = attention.masked_attention(q, np.repeat(k, hq // hkv, axis=1), np.repeat(v, hq // hkv, axis=1), m, 0.25)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # a transposed grouping (h % Hkv instead of h // G) would differ
    o3, _ = attention.masked_attention(q, np.tile(k, (1, hq // hkv, 1)), np.tile(v, (1, hq // hkv, 1)), m, 0.25)
    assert not np.allclose(o1, o3)


def test_masked_rows_get_zero_weight_bitwise():
    rng = np.random.default_rng(6)
    n, hq, hkv, d, w, vs = 30, 4, 2, 8, 7, 5
    q, k, v = _rand(rng, n, hq, d), _rand(rng, n, hkv, d), _rand(rng, n, hkv, d)
    m = masks.prefill_mask(n, w, vs)
    o1, l1 = attention.masked_attention(q, k, v, m, 0.3)
    k2, v2 = k.copy(), v.copy()
    k2[:vs] = 1e30 * np.sign(_rand(rng, vs, hkv, d))
    v2[:vs] = -3e29
    o2, l2 = attention.masked_attention(q, k2, v2, m, 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
