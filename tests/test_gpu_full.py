"""The four large workloads at full size on the GPU, in the launch
configuration the benchmark times, against the fp64 oracle (and bit for bit
on the decode masks at every step and on the device state).  Outputs are
compared element by element where the kernels change regime:

  * single-stream decode: every layer at the first and last step and at the
    steps on both sides of each of the 7 rolls;
  * batched decode: one step in every 16 and the steps around the rolls;
  * chunked VLM prefill: whole 128-row query tiles on both sides of every
    chunk boundary, at each sequence's first unpadded row and (sequence 1)
    at every image-block boundary;
  * packed documents: whole 128-row query tiles on both sides of every
    document boundary and at both ends of the packed batch;
  * the single-stream prompt: whole query tiles of the first and last layer.

  single-stream decode: prompt 8192, 26 layers, 512 steps, 7 rolls
  batched decode: 64 left-padded sequences (lengths U{16..8192}), 256 steps
  chunked prefill (4 x 2048) with image blocks (generic plan)
  packed documents 4 x 4096, D = 512, window 4096
"""

import numpy as np
import pytest
import torch

from oracle import reference
from oracle.compact import CompactModel
from sliding_window_gqa_swa_gb300 import synth
from tests._gpu import assert_close, assert_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swa():
    from tests._lib import ensure_built
    ensure_built()
    from sliding_window_gqa_swa_gb300 import swa as mod
    return mod


def _tile_rows(n, starts):
    """All rows of the 128-row query tiles that contain any of ``starts``."""
    rows = set()
    for x in starts:
        if 0 <= x < n:
            t0 = (x // 128) * 128
            rows.update(range(t0, min(n, t0 + 128)))
    return sorted(rows)


def test_batched_decode_full(swa):
    dev = torch.device("cuda")
    c = synth.workload3()
    S, W, D, B, Hq, Hkv = c.prompt_len, c.window, c.head_dim, c.batch, c.q_heads, c.kv_heads
    scale = D ** -0.5
    cache = swa.Cache(swa.CACHE_COMPACT, 1, B, Hkv, D, W, S, c.valid_start.to(dev))
    # state after compaction: rows [0, W) hold positions [S - W, S)
    cache.k[0, :, :, :W] = c.prompt_k[0].transpose(1, 2).to(dev)
    cache.v[0, :, :, :W] = c.prompt_v[0].transpose(1, 2).to(dev)
    model = CompactModel(S, W)
    mask = torch.empty(B, cache.rows, dtype=torch.uint8, device=dev)
    ws = swa.decode_workspace(cache, Hq)
    check = set(range(0, c.steps, 16)) | {1, 63, 64, 65, 127, 128, 129, 191, 192, 193, c.steps - 1}
    outs, lses = {}, {}
    dq, dk, dv = c.dec_q[:, 0].to(dev), c.dec_k[:, 0].to(dev), c.dec_v[:, 0].to(dev)
    for t in range(c.steps):
        if model.needs_roll():
            swa.roll(cache)
            model.roll()
        swa.build_decode_mask(cache, mask)
        mexp = model.begin_step(c.valid_start.numpy())
        o = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
        l = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        swa.decode(cache, 0, dq[t], dk[t], dv[t], mask, scale, o, ws, l)
        assert np.array_equal(mask.cpu().numpy().astype(bool), mexp), f"mask differs at step {t}"
        if t in check:
            outs[t], lses[t] = o, l
    cache.check()
    st = cache.state()
    assert (st["origin"], st["next_row"], st["step"]) == (model.origin, model.next_row, model.step)
    ro, rl = reference.decode_full(c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0], c.dec_v[:, 0],
                                   S, W, scale, c.valid_start.numpy(), steps=sorted(check))
    for t in sorted(check):
        assert_close(outs[t], ro[t], f"step {t}")
        assert_lse(lses[t], rl[t], f"step {t} lse")


def test_single_stream_full(swa):
    dev = torch.device("cuda")
    c = synth.workload2()
    L, S, W, D, B, Hq, Hkv = c.layers, c.prompt_len, c.window, c.head_dim, c.batch, c.q_heads, c.kv_heads
    scale = D ** -0.5
    pre = swa.Cache(swa.CACHE_PREFILL, L, B, Hkv, D, W, S)
    meta = swa.Meta(B, S, 0, S, W)
    rows = _tile_rows(S, [0, W - 1, W, S // 2, S - 1])  # whole query tiles of the prompt
    for layer in range(L):
        out = torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev)
        swa.prefill(pre, layer, swa.MODE_CAUSAL, c.prompt_q[layer].to(dev), c.prompt_k[layer].to(dev),
                    c.prompt_v[layer].to(dev), meta, scale, out)
        if layer in (0, L - 1):
            ro, _ = reference.prefill_rows(c.prompt_q[layer], c.prompt_k[layer], c.prompt_v[layer], W, scale,
                                           0, rows)
            assert_close(out[0, rows], ro, f"prefill layer {layer}")
    cache = swa.Cache(swa.CACHE_COMPACT, L, B, Hkv, D, W, S)
    swa.compact(pre, cache)
    model = CompactModel(S, W)
    mask = torch.empty(B, cache.rows, dtype=torch.uint8, device=dev)
    ws = swa.decode_workspace(cache, Hq)
    dq, dk, dv = c.dec_q.to(dev), c.dec_k.to(dev), c.dec_v.to(dev)
    # every layer at the steps around each roll, and at the first and last step
    steps = {0, c.steps - 1}
    for r in range(64, c.steps, 64):
        steps.update((r - 1, r, r + 1))
    steps = sorted(s_ for s_ in steps if s_ < c.steps)
    check = {(t, layer) for t in steps for layer in range(L)}
    outs = {}
    for t in range(c.steps):
        if model.needs_roll():
            swa.roll(cache)
            model.roll()
        swa.build_decode_mask(cache, mask)
        mexp = model.begin_step([0])
        for layer in range(L):
            o = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
            swa.decode(cache, layer, dq[t, layer], dk[t, layer], dv[t, layer], mask, scale, o, ws)
            if (t, layer) in check:
                outs[(t, layer)] = o
        assert np.array_equal(mask.cpu().numpy().astype(bool), mexp), f"mask differs at step {t}"
    cache.check()
    for layer in range(L):
        ro, _ = reference.decode_full(c.prompt_k[layer][:, -W:], c.prompt_v[layer][:, -W:], c.dec_q[:, layer],
                                      c.dec_k[:, layer], c.dec_v[:, layer], S, W, scale, None, steps=steps)
        for t in steps:
            assert_close(outs[(t, layer)], ro[t], f"decode step {t} layer {layer}")


def test_chunked_vlm_prefill_full(swa):
    dev = torch.device("cuda")
    c = synth.workload4()
    B, S, Hq, Hkv, D, W, C = c.batch, c.seq_len, c.q_heads, c.kv_heads, c.head_dim, c.window, c.chunk
    scale = D ** -0.5
    vs = c.valid_start.to(dev)
    img = c.img_id.to(dev)
    cache = swa.Cache(swa.CACHE_PREFILL, 1, B, Hkv, D, W, S, vs)
    out = torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, S, Hq, dtype=torch.float32, device=dev)
    for c0 in range(0, S, C):
        meta = swa.Meta(B, S, c0, C, W, valid_start=vs, img_id=img)
        plan = swa.build_prefill_plan(meta, cache)
        o = torch.empty(B, C, Hq, D, dtype=torch.bfloat16, device=dev)
        l = torch.empty(B, C, Hq, dtype=torch.float32, device=dev)
        swa.prefill(cache, 0, swa.MODE_GENERIC, c.q[:, c0:c0 + C].to(dev).contiguous(),
                    c.k[:, c0:c0 + C].to(dev).contiguous(), c.v[:, c0:c0 + C].to(dev).contiguous(),
                    meta, scale, o, l)
        swa.plan_check(plan)
        out[:, c0:c0 + C] = o
        lse[:, c0:c0 + C] = l
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    for b in range(B):
        pad = int(c.valid_start[b])
        starts = [pad, S - 1] + [x for c0 in range(C, S, C) for x in (c0 - 1, c0)]
        if b == 1:  # image blocks [1536, 1792), [2560, 2816), [5120, 5376), [5376, 5632)
            starts += [1535, 1536, 1791, 1792, 2559, 2560, 2815, 2816, 5119, 5120, 5375, 5376, 5631, 5632]
        rows = _tile_rows(S, starts)
        ro, rl = reference.prefill_rows(c.q, c.k, c.v, W, scale, b, rows, c.valid_start.numpy(),
                                        c.img_id.numpy())
        assert_close(out[b, rows], ro, f"sequence {b}")
        assert_lse(lse[b, rows], rl, f"sequence {b} lse")


def test_packed_documents_full(swa):
    dev = torch.device("cuda")
    c = synth.workload5()
    T = int(c.cu_seqlens[-1])
    Hq, D, W = c.q_heads, c.head_dim, c.window
    scale = D ** -0.5
    meta = swa.Meta(1, T, 0, T, W, cu_seqlens=c.cu_seqlens.to(dev))
    swa.build_prefill_plan(meta)
    out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, Hq, dtype=torch.float32, device=dev)
    swa.prefill(None, 0, swa.MODE_GENERIC, c.q.to(dev), c.k.to(dev), c.v.to(dev), meta, scale, out, lse)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    cu = [int(x) for x in c.cu_seqlens]
    rows = _tile_rows(T, [0, T - 1] + [x for d0 in cu[1:-1] for x in (d0 - 1, d0)])
    ro, rl = reference.varlen_rows(c.q, c.k, c.v, c.cu_seqlens.numpy(), W, scale, rows)
    assert_close(out[rows], ro, "packed")
    assert_lse(lse[rows], rl, "packed lse")
