"""Guard canaries: every buffer a kernel writes sits between two 4 KB guard
zones filled with a byte pattern, which must be intact after the calls
(out-of-bounds writes of prefill, compaction, decode, roll, the mask
builders and the backward pass would show there).  It checks the writes the
way a memory-checking tool would, without one.
"""

import numpy as np
import pytest
import torch

from sliding_window_gqa_swa_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side; keeps 256-byte alignment
PATTERN = 0xA5


@pytest.fixture(scope="module")
def swa():
    from tests._lib import ensure_built
    ensure_built()
    from sliding_window_gqa_swa_gb300 import swa as mod
    return mod


class Guarded:
    """A device buffer of `nbytes` between two guard zones."""

    def __init__(self, nbytes):
        self.n = int(nbytes)
        self.buf = torch.full((self.n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.mem = self.buf[GUARD:GUARD + self.n]

    def view(self, dtype, shape):
        return self.mem.view(dtype).view(shape)

    def intact(self):
        return bool((self.buf[:GUARD] == PATTERN).all()) and bool((self.buf[GUARD + self.n:] == PATTERN).all())


def _nbytes(shape, dtype):
    return int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()


@pytest.mark.parametrize("hq,hkv,d,s,chunk", [(4, 2, 256, 300, 300), (3, 3, 256, 200, 72), (4, 2, 512, 260, 130)])
def test_prefill_writes_stay_inside(swa, hq, hkv, d, s, chunk):
    c = synth.prefill_case(4300 + d + hq, batch=2, q_heads=hq, kv_heads=hkv, head_dim=d, window=96, seq_len=s,
                           chunk=chunk, max_pad=9)
    dev = torch.device("cuda")
    vs = c.valid_start.to(dev)
    gcache = Guarded(swa.cache_bytes(swa.CACHE_PREFILL, 1, 2, hkv, d, 96, s))
    cache = swa.Cache(swa.CACHE_PREFILL, 1, 2, hkv, d, 96, s, vs, mem=gcache.mem)
    guards = [gcache]
    for c0 in range(0, s, chunk):
        cl = min(chunk, s - c0)
        meta = swa.Meta(2, s, c0, cl, 96, valid_start=vs)
        go = Guarded(_nbytes((2, cl, hq, d), torch.bfloat16))
        gl = Guarded(_nbytes((2, cl, hq), torch.float32))
        guards += [go, gl]
        q = c.q[:, c0:c0 + cl].to(dev).contiguous()
        k = c.k[:, c0:c0 + cl].to(dev).contiguous()
        v = c.v[:, c0:c0 + cl].to(dev).contiguous()
        swa.prefill(cache, 0, swa.MODE_CAUSAL, q, k, v, meta, d ** -0.5, go.view(torch.bfloat16, (2, cl, hq, d)),
                    gl.view(torch.float32, (2, cl, hq)))
        gp = Guarded(meta.plan_bytes())
        guards.append(gp)
        swa.build_prefill_plan(meta, cache, out=gp.mem)
    torch.cuda.synchronize()
    cache.check()
    assert all(g.intact() for g in guards)


def test_decode_compact_roll_writes_stay_inside(swa):
    dev = torch.device("cuda")
    B, Hq, Hkv, D, W, S, T = 3, 8, 2, 256, 64, 130, 140
    c = synth.decode_case(4400, batch=B, q_heads=Hq, kv_heads=Hkv, head_dim=D, window=W, prompt_len=S,
                          steps=T, layers=2, with_prompt_q=False)
    vs = torch.tensor([0, 7, 3], dtype=torch.int32, device=dev)
    gpre = Guarded(swa.cache_bytes(swa.CACHE_PREFILL, 2, B, Hkv, D, W, S))
    pre = swa.Cache(swa.CACHE_PREFILL, 2, B, Hkv, D, W, S, vs, mem=gpre.mem)
    for layer in range(2):
        swa.prefill(pre, layer, swa.MODE_CAUSAL, torch.zeros(B, S, Hq, D, dtype=torch.bfloat16, device=dev),
                    c.prompt_k[layer].to(dev), c.prompt_v[layer].to(dev), swa.Meta(B, S, 0, S, W, valid_start=vs),
                    D ** -0.5, torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev))
    guards = [gpre]
    for kind in (swa.CACHE_COMPACT, swa.CACHE_RING):
        gc = Guarded(swa.cache_bytes(kind, 2, B, Hkv, D, W, S))
        cmp_ = swa.Cache(kind, 2, B, Hkv, D, W, S, vs, mem=gc.mem)
        swa.compact(pre, cmp_)
        gm = Guarded(B * cmp_.rows)
        gw = Guarded(swa.decode_workspace_bytes(cmp_, Hq))
        gw.mem.zero_()
        mask = gm.view(torch.uint8, (B, cmp_.rows))
        guards += [gc, gm, gw]
        for t in range(T):
            if cmp_.needs_roll():
                swa.roll(cmp_)
            swa.build_decode_mask(cmp_, mask)
            for layer in range(2):
                go = Guarded(_nbytes((B, Hq, D), torch.bfloat16))
                gl = Guarded(_nbytes((B, Hq), torch.float32))
                guards += [go, gl]
                swa.decode(cmp_, layer, c.dec_q[t, layer].to(dev), c.dec_k[t, layer].to(dev),
                           c.dec_v[t, layer].to(dev), mask, D ** -0.5, go.view(torch.bfloat16, (B, Hq, D)), gw.mem,
                           gl.view(torch.float32, (B, Hq)))
        torch.cuda.synchronize()
        cmp_.check()
    assert all(g.intact() for g in guards)


@pytest.mark.parametrize("docs,hq,hkv,d,w", [([300, 70], 4, 2, 512, 200), ([129, 1, 130], 3, 1, 256, 64)])
def test_backward_writes_stay_inside(swa, docs, hq, hkv, d, w):
    dev = torch.device("cuda")
    c = synth.varlen_case(4500 + d, doc_lens=docs, q_heads=hq, kv_heads=hkv, head_dim=d, window=w)
    T = int(c.cu_seqlens[-1])
    meta = swa.Meta(1, T, 0, T, w, cu_seqlens=c.cu_seqlens.to(dev))
    gp = Guarded(meta.plan_bytes())
    swa.build_prefill_plan(meta, out=gp.mem)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    g = synth.upstream_grad(4500 + d, c.q.shape).to(dev)
    out = torch.empty(T, hq, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, hq, dtype=torch.float32, device=dev)
    swa.prefill(None, 0, swa.MODE_GENERIC, q, k, v, meta, d ** -0.5, out, lse)
    gq = Guarded(_nbytes((T, hq, d), torch.bfloat16))
    gk = Guarded(_nbytes((T, hkv, d), torch.bfloat16))
    gv = Guarded(_nbytes((T, hkv, d), torch.bfloat16))
    gw = Guarded(swa.backward_workspace_bytes(hq, meta))
    swa.prefill_backward(q, k, v, out, g, lse, meta, d ** -0.5, gq.view(torch.bfloat16, (T, hq, d)),
                         gk.view(torch.bfloat16, (T, hkv, d)), gv.view(torch.bfloat16, (T, hkv, d)), gw.mem)
    torch.cuda.synchronize()
    swa.plan_check(gp.mem)
    assert all(x.intact() for x in (gp, gq, gk, gv, gw))
