"""Backward pass on the GPU against the fp64 oracle.

* packed documents (head size 512 and 256; a window that binds inside the
  documents and one that never does; an odd GQA group; a window of one key),
  with document lengths that leave ragged query and key tiles;
* left-padded batches through the same plan, with finite garbage in the pad
  keys (zero gradients there, and for pad rows), and image blocks (future
  same-image keys, a block longer than the window);
* the full packed training shape (4 x 4096 tokens, Hq=16, Hkv=8, D=512,
  W=4096) in the launch configuration the benchmark times: a whole 128-row
  query tile (its dq, and dk / dv of the keys only it admits) against the
  oracle, and the gradient sums every mask satisfies.

The forward pass that produces out and lse is the library's own prefill.
Gradients are compared row by row, relative to the reference's scale
(tests/_gpu.py: assert_grad_close).
"""

import numpy as np
import pytest
import torch

from oracle import reference
from sliding_window_gqa_swa_gb300 import synth
from tests._gpu import assert_grad_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swa():
    from tests._lib import ensure_built
    ensure_built()
    from sliding_window_gqa_swa_gb300 import swa as mod
    return mod


def run_packed(swa, c, dout):
    """Forward + backward of packed documents; returns (out, lse, dq, dk, dv)."""
    dev = torch.device("cuda")
    T, Hq, Hkv, D, W = int(c.cu_seqlens[-1]), c.q_heads, c.kv_heads, c.head_dim, c.window
    scale = D ** -0.5
    meta = swa.Meta(1, T, 0, T, W, cu_seqlens=c.cu_seqlens.to(dev))
    plan = swa.build_prefill_plan(meta)
    q, k, v, g = c.q.to(dev), c.k.to(dev), c.v.to(dev), dout.to(dev)
    out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, Hq, dtype=torch.float32, device=dev)
    swa.prefill(None, 0, swa.MODE_GENERIC, q, k, v, meta, scale, out, lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = swa.backward_workspace(Hq, meta)
    swa.prefill_backward(q, k, v, out, g, lse, meta, scale, dq, dk, dv, ws)
    torch.cuda.synchronize()
    swa.plan_check(plan)
    return out, lse, dq, dk, dv


PACKED = {
    # name: (seed, doc_lens, Hq, Hkv, D, W)
    "d512_window_binds": (4301, [300, 400, 300], 4, 2, 512, 256),
    "d512_window_wide": (4302, [700, 300, 1], 4, 2, 512, 4096),
    "d256_ragged": (4303, [129, 255, 64, 3], 4, 2, 256, 100),
    "d512_gqa3": (4304, [333], 3, 1, 512, 128),
    "d256_window_one": (4305, [200, 57], 2, 1, 256, 1),
    "d512_mha": (4306, [260], 2, 2, 512, 300),
}


@pytest.mark.parametrize("name", list(PACKED))
def test_packed_backward(swa, name):
    seed, docs, Hq, Hkv, D, W = PACKED[name]
    c = synth.varlen_case(seed, doc_lens=docs, q_heads=Hq, kv_heads=Hkv, head_dim=D, window=W)
    dout = synth.upstream_grad(seed, c.q.shape)
    _, _, dq, dk, dv = run_packed(swa, c, dout)
    rq, rk, rv = reference.varlen_backward(c.q, c.k, c.v, dout, c.cu_seqlens.numpy(), W, D ** -0.5)
    assert_grad_close(dq, rq, name + " dq")
    assert_grad_close(dk, rk, name + " dk")
    assert_grad_close(dv, rv, name + " dv")


BATCHED = {
    # name: (seed, B, Hq, Hkv, D, W, S, max_pad, images)
    "padded_d256": (4311, 2, 4, 2, 256, 100, 300, 40, None),
    "padded_d512": (4312, 2, 4, 2, 512, 64, 200, 30, None),
    "images_d256": (4313, 1, 4, 2, 256, 64, 260, 5, {0: [(100, 180), (180, 200)]}),
}


@pytest.mark.parametrize("name", list(BATCHED))
def test_batched_backward(swa, name):
    seed, B, Hq, Hkv, D, W, S, max_pad, images = BATCHED[name]
    dev = torch.device("cuda")
    c = synth.prefill_case(seed, batch=B, q_heads=Hq, kv_heads=Hkv, head_dim=D, window=W, seq_len=S, chunk=S,
                           max_pad=max_pad, images=images)
    for b in range(B):  # pad keys carry finite garbage
        c.k[b, :int(c.valid_start[b])] = 300.0
        c.v[b, :int(c.valid_start[b])] = -300.0
    dout = synth.upstream_grad(seed, c.q.shape)
    scale = D ** -0.5
    vs = c.valid_start.to(dev)
    img = None if c.img_id is None else c.img_id.to(dev).contiguous()
    # forward through a prefill cache (the library's batched prefill), the same plan for both passes
    cache = swa.Cache(swa.CACHE_PREFILL, 1, B, Hkv, D, W, S, vs)
    meta = swa.Meta(B, S, 0, S, W, valid_start=vs, img_id=img)
    plan = swa.build_prefill_plan(meta, cache)
    q, k, v, g = c.q.to(dev), c.k.to(dev), c.v.to(dev), dout.to(dev)
    out = torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, S, Hq, dtype=torch.float32, device=dev)
    swa.prefill(cache, 0, swa.MODE_GENERIC, q, k, v, meta, scale, out, lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = swa.backward_workspace(Hq, meta)
    ws.fill_(0xFF)  # the backward needs no initialised workspace (0xFFFF is a bf16 NaN)
    swa.prefill_backward(q, k, v, out, g, lse, meta, scale, dq, dk, dv, ws)
    torch.cuda.synchronize()
    swa.plan_check(plan)
    rq, rk, rv = reference.prefill_backward(c.q, c.k, c.v, dout, W, scale, c.valid_start.numpy(),
                                            None if c.img_id is None else c.img_id.numpy())
    assert_grad_close(dq, rq, name + " dq")
    assert_grad_close(dk, rk, name + " dk")
    assert_grad_close(dv, rv, name + " dv")
    for b in range(B):
        pad = int(c.valid_start[b])
        assert torch.all(dq[b, :pad] == 0) and torch.all(dk[b, :pad] == 0) and torch.all(dv[b, :pad] == 0)


def test_packed_training_shape_full(swa):
    c = synth.workload5()
    T, Hq, Hkv, D, W = int(c.cu_seqlens[-1]), c.q_heads, c.kv_heads, c.head_dim, c.window
    dout = synth.upstream_grad(synth.SEED_BASE + 5, c.q.shape)
    _, _, dq, dk, dv = run_packed(swa, c, dout)
    cu = c.cu_seqlens.numpy()
    # the last query tile of document 1: rows [2 x 4096 - 128, 2 x 4096); only they
    # admit the keys of that tile
    rows = list(range(int(cu[2]) - 128, int(cu[2])))
    rq, rk, rv = reference.varlen_backward_rows(c.q, c.k, c.v, dout, cu, W, D ** -0.5, rows)
    assert_grad_close(dq[rows], rq, "dq (query tile)")
    assert_grad_close(dk[rows], rk[rows], "dk (key tile)")
    assert_grad_close(dv[rows], rv[rows], "dv (key tile)")
    # every mask: sum_j dv_j = sum_i dout_i over each KV head's query heads, and
    # sum_j dk_j = 0 (softmax is shift-invariant); bounds cover bf16 rounding of
    # each stored element and of the probabilities
    gv = dv.double().sum(dim=0).cpu().numpy()
    want = dout.double().reshape(T, Hkv, Hq // Hkv, D).sum(dim=(0, 2)).numpy()
    assert np.abs(gv - want).max() <= 2.0 ** -8 * dv.double().abs().sum(dim=0).max().item() + 0.05
    gk = dk.double().sum(dim=0).cpu().numpy()
    assert np.abs(gk).max() <= 2.0 ** -8 * dk.double().abs().sum(dim=0).max().item() + 0.05
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
