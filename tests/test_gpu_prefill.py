"""Prefill on the GPU against the fp64 oracle (small and ragged cases).

* the dense mask the kernel applies (expanded from the plan, or from the
  causal arithmetic) equals the oracle's mask bit for bit;
* outputs and lse of causal, generic (VLM image blocks, adjacent blocks, a
  block longer than the window) and packed-document prefill, whole and in
  chunks (chunked = unchunked), within the tolerances;
* pad rows give zero output and lse = -inf; pad keys with garbage get zero
  weight;
* an image block that crosses a chunk end is reported (SWA_EDEVICE).
"""

import numpy as np
import pytest
import torch

from oracle import masks, reference
from sliding_window_gqa_swa_gb300 import synth
from tests._gpu import assert_close, assert_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swa():
    from tests._lib import ensure_built
    ensure_built()
    from sliding_window_gqa_swa_gb300 import swa as mod
    return mod


def _oracle_masks(c):
    return [masks.prefill_mask(c.seq_len, c.window, int(c.valid_start[b]),
                               None if c.img_id is None else c.img_id[b].numpy())
            for b in range(c.batch)]


def run_cache_prefill(swa, c, mode, chunk):
    dev = torch.device("cuda")
    B, S, Hq, Hkv, D, W = c.batch, c.seq_len, c.q_heads, c.kv_heads, c.head_dim, c.window
    scale = D ** -0.5
    vs = c.valid_start.to(dev)
    img = None if c.img_id is None else c.img_id.to(dev).contiguous()
    cache = swa.Cache(swa.CACHE_PREFILL, 1, B, Hkv, D, W, S, vs)
    out = torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, S, Hq, dtype=torch.float32, device=dev)
    dense = torch.zeros(B, S, S, dtype=torch.uint8)
    for c0 in range(0, S, chunk):
        cl = min(chunk, S - c0)
        meta = swa.Meta(B, S, c0, cl, W, valid_start=vs, img_id=img)
        if mode == swa.MODE_GENERIC:
            plan = swa.build_prefill_plan(meta, cache)
            swa.plan_check(plan)
        dense[:, c0:c0 + cl] = swa.dense_debug_mask(meta).cpu()
        q = c.q[:, c0:c0 + cl].to(dev).contiguous()
        k = c.k[:, c0:c0 + cl].to(dev).contiguous()
        v = c.v[:, c0:c0 + cl].to(dev).contiguous()
        o = torch.empty(B, cl, Hq, D, dtype=torch.bfloat16, device=dev)
        l = torch.empty(B, cl, Hq, dtype=torch.float32, device=dev)
        swa.prefill(cache, 0, mode, q, k, v, meta, scale, o, l)
        out[:, c0:c0 + cl] = o
        lse[:, c0:c0 + cl] = l
    torch.cuda.synchronize()
    return out, lse, dense


CASES = {
    # name: (seed, batch, Hq, Hkv, D, W, S, chunk, max_pad, images)
    "causal_ragged": (4101, 2, 4, 2, 256, 64, 300, 300, 40, None),
    "causal_chunked": (4102, 2, 4, 2, 256, 100, 300, 128, 40, None),
    "causal_d512": (4103, 1, 4, 2, 512, 64, 200, 200, 7, None),
    "vlm_whole": (4104, 2, 8, 4, 256, 64, 384, 384, 20, {1: [(30, 60), (60, 100), (140, 230), (300, 330)]}),
    "vlm_chunked": (4105, 2, 8, 4, 256, 64, 384, 128, 20, {1: [(30, 60), (60, 100), (140, 230), (300, 330)],
                                                          0: [(260, 261)]}),
    "vlm_d512": (4106, 1, 4, 2, 512, 32, 256, 128, 0, {0: [(10, 100), (150, 200)]}),
    "causal_wide_window": (4108, 1, 2, 1, 256, 2000, 333, 333, 3, None),
    "causal_window_below_tile": (4109, 2, 2, 2, 256, 20, 200, 72, 11, None),
    # head size 256 runs query heads 2g and 2g + 1 as one CTA pair when the group
    # size is even, and one CTA per head otherwise
    "gqa3_single_cta": (4111, 1, 6, 2, 256, 96, 260, 260, 5, None),
    "gqa4_pairs": (4112, 1, 8, 2, 256, 96, 260, 130, 5, None),
    # head size 512: an even group runs as four-CTA clusters (a score pair and an
    # output pair per pair of heads); an odd group as column pairs that exchange
    # partial scores
    "d512_gqa3_column_pairs": (4113, 1, 3, 1, 512, 64, 200, 200, 7, None),
    "d512_gqa4_pairs": (4114, 1, 8, 2, 512, 96, 260, 130, 5, None),
}

# query scale that spreads scores over a wide range, so the running maximum of
# a row keeps growing across key tiles (exercises the rescaling of the output)
Q_SCALE = {"causal_big_scores": 4.0, "causal_big_scores_d512": 3.0}
CASES["causal_big_scores"] = (4110, 2, 4, 2, 256, 300, 400, 400, 9, None)
CASES["causal_big_scores_d512"] = (4115, 1, 4, 2, 512, 300, 400, 400, 9, None)


@pytest.mark.parametrize("name", list(CASES))
def test_cache_prefill(swa, name):
    seed, B, Hq, Hkv, D, W, S, chunk, max_pad, images = CASES[name]
    c = synth.prefill_case(seed, batch=B, q_heads=Hq, kv_heads=Hkv, head_dim=D, window=W, seq_len=S,
                           chunk=chunk, max_pad=max_pad, images=images)
    if name in Q_SCALE:
        c.q = (c.q.float() * Q_SCALE[name]).to(torch.bfloat16)
    for b in range(B):  # pad keys carry finite garbage
        c.k[b, :int(c.valid_start[b])] = 300.0
        c.v[b, :int(c.valid_start[b])] = -300.0
    mode = swa.MODE_GENERIC if images else swa.MODE_CAUSAL
    out, lse, dense = run_cache_prefill(swa, c, mode, chunk)
    om = _oracle_masks(c)
    for b in range(B):
        assert np.array_equal(dense[b].numpy().astype(bool), om[b]), f"mask differs for sequence {b}"
    ro, rl = reference.prefill(c.q, c.k, c.v, W, D ** -0.5, c.valid_start.numpy(),
                               None if c.img_id is None else c.img_id.numpy())
    assert_close(out, ro, name)
    assert_lse(lse, rl, name + " lse")
    for b in range(B):
        pad = int(c.valid_start[b])
        assert torch.all(out[b, :pad] == 0)


def test_generic_plan_equals_causal_without_images(swa):
    c = synth.prefill_case(4107, batch=2, q_heads=4, kv_heads=2, head_dim=256, window=50, seq_len=260,
                           chunk=260, max_pad=30)
    o1, l1, d1 = run_cache_prefill(swa, c, swa.MODE_CAUSAL, 260)
    o2, l2, d2 = run_cache_prefill(swa, c, swa.MODE_GENERIC, 130)
    assert torch.equal(d1, d2)
    ro, _ = reference.prefill(c.q, c.k, c.v, 50, 256 ** -0.5, c.valid_start.numpy())
    assert_close(o1, ro)
    assert_close(o2, ro)


@pytest.mark.parametrize("doc_lens,d,w", [([100, 37, 200, 1], 512, 50), ([129, 255, 64], 256, 1000),
                                          ([300], 512, 7)])
def test_packed_documents(swa, doc_lens, d, w):
    dev = torch.device("cuda")
    c = synth.varlen_case(4200 + len(doc_lens), doc_lens=doc_lens, q_heads=4, kv_heads=2, head_dim=d, window=w)
    T = int(c.cu_seqlens[-1])
    meta = swa.Meta(1, T, 0, T, w, cu_seqlens=c.cu_seqlens.to(dev))
    plan = swa.build_prefill_plan(meta)
    swa.plan_check(plan)
    dense = swa.dense_debug_mask(meta)[0].cpu().numpy().astype(bool)
    doc = masks.doc_ids_from_cu_seqlens(c.cu_seqlens.numpy(), T)
    assert np.array_equal(dense, masks.prefill_mask(T, w, 0, None, doc))
    out = torch.empty(T, 4, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, 4, dtype=torch.float32, device=dev)
    swa.prefill(None, 0, swa.MODE_GENERIC, c.q.to(dev), c.k.to(dev), c.v.to(dev), meta, d ** -0.5, out, lse)
    torch.cuda.synchronize()
    ro, rl = reference.varlen_rows(c.q, c.k, c.v, c.cu_seqlens.numpy(), w, d ** -0.5, range(T))
    assert_close(out, ro, "packed")
    assert_lse(lse, rl, "packed lse")


def test_image_crossing_chunk_is_reported(swa):
    dev = torch.device("cuda")
    img = torch.full((1, 256), -1, dtype=torch.int32)
    img[0, 100:140] = 0
    meta = swa.Meta(1, 256, 0, 128, 64, img_id=img.to(dev))
    plan = swa.build_prefill_plan(meta)
    with pytest.raises(swa.SwaError) as e:
        swa.plan_check(plan)
    assert e.value.status == swa.EDEVICE
    meta2 = swa.Meta(1, 256, 128, 128, 64, img_id=img.to(dev))
    swa.plan_check(swa.build_prefill_plan(meta2))
