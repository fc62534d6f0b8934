"""Derivation of the gradient tolerance used by the backward parity tests.

The pages time the training step of packed-document attention ("Add SDPA
attention implementation", Summary and its forward + backward tables) but fix
no tolerance for the gradients, and the flat output bound (1e-2) does not scale
with them.  The bound in tests/_gpu.py (``assert_grad_close``) is therefore
derived here, on the CPU, from the arithmetic the backward kernels do, and not
from the kernels' measured error:

* the forward output is stored in bf16 and ``delta = rowsum(dout * out)`` is
  taken from that stored output;
* the probabilities ``P = exp(scale * s - lse)`` are rounded to bf16 before
  the tensor-core products that use them (dV = P^T dout);
* ``dS = scale * P * (dP - delta)`` is formed from the unrounded P and rounded
  to bf16 before dQ = dS K and dK = dS^T Q;
* every gradient is accumulated in fp32 (here: fp64) and stored in bf16.

This emulation, on exactly the shapes of tests/test_gpu_backward.py, must stay
well inside the bound (at most 0.6 of it, per row and for the mean), so the
bound holds the kernels to those rounding points with room only for fp32
accumulation order, and a kernel that drops a term or mis-rounds still fails.
"""

import numpy as np
import pytest
import torch

from oracle import masks, reference
from sliding_window_gqa_swa_gb300 import synth
from tests._gpu import GRAD_FLOOR, GRAD_MEAN_REL, GRAD_ROW_REL, GRAD_TENSOR_REL
from tests.test_gpu_backward import BATCHED, PACKED

MARGIN = 0.6


def bf16(x: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest even) and widen back to float64."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


def kernel_rounding_backward(q, k, v, mask, scale, dout):
    """Gradients with the backward kernels' rounding points (module docstring);
    q, dout [S, Hq, D], k, v [S, Hkv, D] float64, mask [S, S] bool."""
    S, Hq, D = q.shape
    G = Hq // k.shape[1]
    dq, dk, dv = np.zeros(q.shape), np.zeros(k.shape), np.zeros(v.shape)
    for h in range(Hq):
        kh, vh = k[:, h // G], v[:, h // G]
        s = scale * (q[:, h] @ kh.T)
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1, initial=-np.inf)
        m_safe = np.where(np.isfinite(m), m, 0.0)
        e = np.where(mask, np.exp(s - m_safe[:, None]), 0.0)
        l = e.sum(axis=1)
        lse = np.where(l > 0, m_safe + np.log(np.where(l > 0, l, 1.0)), -np.inf)
        p = np.where(mask, np.exp(s - np.where(np.isfinite(lse), lse, 0.0)[:, None]), 0.0)
        out = bf16(p @ vh)
        delta = (dout[:, h] * out).sum(axis=1)
        dp = dout[:, h] @ vh.T
        ds = bf16(np.where(mask, scale * p * (dp - delta[:, None]), 0.0))
        dq[:, h] = ds @ kh
        dk[:, h // G] += ds.T @ q[:, h]
        dv[:, h // G] += bf16(p).T @ dout[:, h]
    return bf16(dq), bf16(dk), bf16(dv)


def ratios(ref, emu):
    """(worst row error / row bound, mean error / mean bound) of one gradient."""
    err = np.abs(emu - ref)
    top = np.abs(ref).max(initial=0.0)
    row_bound = GRAD_ROW_REL * np.abs(ref).max(axis=-1) + GRAD_TENSOR_REL * top + GRAD_FLOOR
    row = float((err.max(axis=-1) / row_bound).max())
    mean = float(err.mean() / (GRAD_MEAN_REL * np.abs(ref).mean() + GRAD_FLOOR / 10))
    return row, mean


def f64(t):
    return t.double().numpy()


@pytest.mark.parametrize("name", list(PACKED))
def test_packed_shapes_within_bound(name):
    seed, docs, Hq, Hkv, D, W = PACKED[name]
    c = synth.varlen_case(seed, doc_lens=docs, q_heads=Hq, kv_heads=Hkv, head_dim=D, window=W)
    dout = synth.upstream_grad(seed, c.q.shape)
    T = int(c.cu_seqlens[-1])
    mask = masks.prefill_mask(T, W, 0, None, masks.doc_ids_from_cu_seqlens(c.cu_seqlens.numpy(), T))
    ref = reference.varlen_backward(c.q, c.k, c.v, dout, c.cu_seqlens.numpy(), W, D ** -0.5)
    emu = kernel_rounding_backward(f64(c.q), f64(c.k), f64(c.v), mask, D ** -0.5, f64(dout))
    for what, r, e in zip(("dq", "dk", "dv"), ref, emu):
        row, mean = ratios(r, e)
        assert row <= MARGIN, f"{name} {what}: row error {row:.2f} of the bound"
        assert mean <= MARGIN, f"{name} {what}: mean error {mean:.2f} of the bound"


@pytest.mark.parametrize("name", list(BATCHED))
def test_batched_shapes_within_bound(name):
    seed, B, Hq, Hkv, D, W, S, max_pad, images = BATCHED[name]
    c = synth.prefill_case(seed, batch=B, q_heads=Hq, kv_heads=Hkv, head_dim=D, window=W, seq_len=S, chunk=S,
                           max_pad=max_pad, images=images)
    for b in range(B):  # the same finite garbage in the pad keys as the GPU test
        c.k[b, :int(c.valid_start[b])] = 300.0
        c.v[b, :int(c.valid_start[b])] = -300.0
    dout = synth.upstream_grad(seed, c.q.shape)
    img = None if c.img_id is None else c.img_id.numpy()
    ref = reference.prefill_backward(c.q, c.k, c.v, dout, W, D ** -0.5, c.valid_start.numpy(), img)
    emu = [np.zeros(r.shape) for r in ref]
    for b in range(B):
        mask = masks.prefill_mask(S, W, int(c.valid_start[b]), None if img is None else img[b])
        got = kernel_rounding_backward(f64(c.q[b]), f64(c.k[b]), f64(c.v[b]), mask, D ** -0.5, f64(dout[b]))
        for e, g in zip(emu, got):
            e[b] = g
    for what, r, e in zip(("dq", "dk", "dv"), ref, emu):
        row, mean = ratios(r, e)
        assert row <= MARGIN, f"{name} {what}: row error {row:.2f} of the bound"
        assert mean <= MARGIN, f"{name} {what}: mean error {mean:.2f} of the bound"


def test_bound_rejects_a_dropped_rounding_error_budget():
    """The bound is not loose enough to hide a plain mistake: leaving delta out
    of dS (a dropped term) on a small packed case exceeds it."""
    seed, docs, Hq, Hkv, D, W = PACKED["d256_ragged"]
    c = synth.varlen_case(seed, doc_lens=docs, q_heads=Hq, kv_heads=Hkv, head_dim=D, window=W)
    dout = synth.upstream_grad(seed, c.q.shape)
    T = int(c.cu_seqlens[-1])
    mask = masks.prefill_mask(T, W, 0, None, masks.doc_ids_from_cu_seqlens(c.cu_seqlens.numpy(), T))
    ref = reference.varlen_backward(c.q, c.k, c.v, dout, c.cu_seqlens.numpy(), W, D ** -0.5)
    q, k, v, g = f64(c.q), f64(c.k), f64(c.v), f64(dout)
    G = Hq // Hkv
    dq_bad = np.zeros(q.shape)
    for h in range(Hq):
        kh, vh = k[:, h // G], v[:, h // G]
        s = np.where(mask, D ** -0.5 * (q[:, h] @ kh.T), -np.inf)
        m = s.max(axis=1, initial=-np.inf)
        e = np.where(mask, np.exp(s - np.where(np.isfinite(m), m, 0.0)[:, None]), 0.0)
        p = e / np.maximum(e.sum(axis=1, keepdims=True), 1e-300)
        ds = np.where(mask, D ** -0.5 * p * (g[:, h] @ vh.T), 0.0)  # delta left out
        dq_bad[:, h] = ds @ kh
    row, _ = ratios(ref[0], bf16(dq_bad))
    assert row > 1.0
