"""The allocation-free decode entry point (swa_decode_noalloc).

Some callers cannot allocate device memory -- a plugin inside an inference
runtime that plans every buffer ahead and passes the plugin only its inputs
and outputs, for instance -- so they cannot provide swa_decode's workspace.
swa_decode_noalloc keeps that scratch in a static device array instead.  This
test calls it through the C ABI and checks its outputs against swa_decode's
on the same inputs, for two calls in a row and across two decode steps, with
the tolerance the other GPU tests use.  It is collected last (file name) so a
run that stops at the first failure has run everything else first; it works
alone in a fresh process as well as after the other tests.
"""

import ctypes

import pytest
import torch

from sliding_window_gqa_swa_gb300 import synth
from tests._gpu import assert_close, assert_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swa():
    from tests._lib import ensure_built
    ensure_built()
    from sliding_window_gqa_swa_gb300 import swa as mod
    return mod


def _noalloc(swa, cache, layer, q, k, v, mask, scale, out, lse):
    st = swa.lib().swa_decode_noalloc(cache.handle, layer, q.shape[-2], swa.ptr(q), swa.ptr(k), swa.ptr(v),
                                      swa.ptr(mask), float(scale), swa.ptr(out), swa.ptr(lse),
                                      swa.stream_handle(None))
    swa.check(st, "swa_decode_noalloc")


@pytest.mark.parametrize("batch,hq,hkv,d", [(2, 4, 2, 256), (3, 16, 8, 128)])
def test_noalloc_matches_workspace_decode(swa, batch, hq, hkv, d):
    dev = torch.device("cuda")
    W, S = 64, 300
    c = synth.decode_case(5100 + d, batch=batch, q_heads=hq, kv_heads=hkv, head_dim=d, window=W, prompt_len=S,
                          steps=2, layers=1, prompt_rows=W)
    cache = swa.Cache(swa.CACHE_COMPACT, 1, batch, hkv, d, W, S)
    cache.k[0, :, :, :W] = c.prompt_k[0].transpose(1, 2).to(dev)  # rows [0, W) hold positions [S - W, S)
    cache.v[0, :, :, :W] = c.prompt_v[0].transpose(1, 2).to(dev)
    mask = torch.empty(batch, cache.rows, dtype=torch.uint8, device=dev)
    ws = swa.decode_workspace(cache, hq)
    scale = d ** -0.5
    for t in range(2):
        swa.build_decode_mask(cache, mask)
        q, k, v = c.dec_q[t, 0].to(dev), c.dec_k[t, 0].to(dev), c.dec_v[t, 0].to(dev)
        ref = torch.empty(batch, hq, d, dtype=torch.bfloat16, device=dev)
        ref_lse = torch.empty(batch, hq, dtype=torch.float32, device=dev)
        swa.decode(cache, 0, q, k, v, mask, scale, ref, ws, ref_lse)
        for call in range(2):  # two calls in a row share the static scratch
            out = torch.full((batch, hq, d), 7.0, dtype=torch.bfloat16, device=dev)
            lse = torch.full((batch, hq), 7.0, dtype=torch.float32, device=dev)
            _noalloc(swa, cache, 0, q, k, v, mask, scale, out, lse)
            torch.cuda.synchronize()
            assert_close(out, ref.float().cpu().numpy(), f"step {t} call {call}")
            assert_lse(lse, ref_lse.cpu().numpy(), f"step {t} call {call} lse")
    cache.check()


def test_noalloc_rejects_oversized_shapes(swa):
    # a batch whose split-K scratch exceeds the static array is refused on the host
    cache = swa.Cache(swa.CACHE_COMPACT, 1, 512, 8, 512, 1024, 2048)
    need = swa.decode_workspace_bytes(cache, 64)
    assert need > 8 << 20
    mask = torch.zeros(512, cache.rows, dtype=torch.uint8, device="cuda")
    swa.build_decode_mask(cache, mask)
    q = torch.zeros(512, 64, 512, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(512, 8, 512, dtype=torch.bfloat16, device="cuda")
    st = swa.lib().swa_decode_noalloc(cache.handle, 0, 64, swa.ptr(q), swa.ptr(kv), swa.ptr(kv), swa.ptr(mask),
                                      ctypes.c_float(1.0), swa.ptr(q), None, swa.stream_handle(None))
    assert st == swa.EUNSUPPORTED
    assert "static array" in swa.last_error()
