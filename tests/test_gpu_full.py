"""The four large workloads at full size on the GPU, in the launch
configuration the benchmark times, against the fp64 oracle on sampled
outputs (and bit for bit on the decode masks and the device state).

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


def _sample_rows(n, extra=(), k=24, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(int(x) for x in rng.choice(n, size=min(k, n), replace=False))
    rows.update(int(x) for x in extra if 0 <= x < n)
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
    check = {0, 1, 63, 64, 65, 130, 192, 255}
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
    rows = _sample_rows(S, extra=(0, 1, W - 1, W, W + 1, S - 1), k=16, seed=2)
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
    check = {(0, 0), (63, 5), (64, 25), (100, 13), (511, 0), (511, 25), (448, 7)}
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
        if t % 64 in (0, 1, 63):
            assert np.array_equal(mask.cpu().numpy().astype(bool), mexp), f"mask differs at step {t}"
    cache.check()
    for (t, layer), o in sorted(outs.items()):
        ro, _ = reference.decode_full(c.prompt_k[layer][:, -W:], c.prompt_v[layer][:, -W:], c.dec_q[:, layer],
                                      c.dec_k[:, layer], c.dec_v[:, layer], S, W, scale, None, steps=[t])
        assert_close(o, ro[t], f"decode step {t} layer {layer}")


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
        extra = [pad - 1, pad, pad + 1, 2047, 2048, 4095, 4096, S - 1]
        if b == 1:
            extra += [1536, 1600, 1791, 1792, 2560, 2815, 5119, 5120, 5375, 5376, 5631]
        rows = _sample_rows(S, extra=extra, k=12, seed=b)
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
    rows = _sample_rows(T, extra=(0, 1, 127, 128, 4095, 4096, 4097, 8191, 12288, T - 1), k=14, seed=5)
    ro, rl = reference.varlen_rows(c.q, c.k, c.v, c.cu_seqlens.numpy(), W, scale, rows)
    assert_close(out[rows], ro, "packed")
    assert_lse(lse[rows], rl, "packed lse")
