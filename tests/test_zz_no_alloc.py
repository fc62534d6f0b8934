"""The allocation-free decode entry point (swa_decode_noalloc).

Some callers cannot allocate device memory -- a plugin inside an inference
runtime that plans every buffer ahead and passes the plugin only its inputs
and outputs, for instance -- so they cannot provide swa_decode's workspace.
swa_decode_noalloc keeps that scratch in a static device array instead.

The tests call it through the C ABI, two calls in a row per decode step, and
check its outputs against swa_decode's on the same inputs (the same kernels
and split, so bit for bit) and against the fp64 oracle with the tolerance the
other GPU tests use.  The shapes cover the paths that use the static array:
splits merged through the workspace (a large batch; a window longer than 16
clusters' worth of rows), shown on the host to write the workspace; and one
shape whose splits merge inside a thread-block cluster (no scratch at all).
This file is collected last (file name) so a run that stops at the first
failure has run everything else first; it works alone in a fresh process as
well as after the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

from oracle import reference
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
                                      swa.ptr(mask), ctypes.c_float(scale), swa.ptr(out), swa.ptr(lse),
                                      swa.stream_handle(None))
    swa.check(st, "swa_decode_noalloc")


SHAPES = {
    # name: (batch, Hq, Hkv, D, W, S, workspace merge)
    "throughput_batch": (32, 16, 8, 256, 64, 300, True),       # 256 slabs: two splits per slab
    "long_window": (1, 2, 1, 256, 4096, 4200, True),           # 64 splits of one slab
    "batched_1088_rows": (64, 16, 8, 256, 1024, 1100, True),   # the batched-decode shape: three splits
    "cluster_merge": (2, 4, 2, 256, 64, 300, False),           # splits merge inside one cluster
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_noalloc_matches_workspace_decode_and_oracle(swa, name):
    batch, hq, hkv, d, W, S, ws_merge = SHAPES[name]
    dev = torch.device("cuda")
    steps = 2
    c = synth.decode_case(5100 + d + batch, batch=batch, q_heads=hq, kv_heads=hkv, head_dim=d, window=W,
                          prompt_len=S, steps=steps, layers=1, prompt_rows=W)
    cache = swa.Cache(swa.CACHE_COMPACT, 1, batch, hkv, d, W, S)
    cache.k[0, :, :, :W] = c.prompt_k[0].transpose(1, 2).to(dev)  # rows [0, W) hold positions [S - W, S)
    cache.v[0, :, :, :W] = c.prompt_v[0].transpose(1, 2).to(dev)
    mask = torch.empty(batch, cache.rows, dtype=torch.uint8, device=dev)
    scale = d ** -0.5
    ref_o, ref_l = reference.decode_full(c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0], c.dec_v[:, 0],
                                         S, W, scale)
    for t in range(steps):
        swa.build_decode_mask(cache, mask)
        q, k, v = c.dec_q[t, 0].to(dev), c.dec_k[t, 0].to(dev), c.dec_v[t, 0].to(dev)
        # swa_decode with a workspace whose partial area holds a sentinel: the
        # shapes that merge through the workspace overwrite it
        ws = swa.decode_workspace(cache, hq)
        tickets = (batch * hkv * 4 + 255) // 256 * 256
        ws[tickets:] = 0x7F
        ref = torch.empty(batch, hq, d, dtype=torch.bfloat16, device=dev)
        ref_lse = torch.empty(batch, hq, dtype=torch.float32, device=dev)
        swa.decode(cache, 0, q, k, v, mask, scale, ref, ws, ref_lse)
        torch.cuda.synchronize()
        wrote = bool((ws[tickets:] != 0x7F).any())
        assert wrote == ws_merge, f"{name}: workspace merge expected {ws_merge}, partials written {wrote}"
        assert torch.all(ws[:tickets] == 0), "swa_decode leaves its tickets at zero"
        for call in range(2):  # two calls in a row share the static scratch
            out = torch.full((batch, hq, d), 7.0, dtype=torch.bfloat16, device=dev)
            lse = torch.full((batch, hq), 7.0, dtype=torch.float32, device=dev)
            _noalloc(swa, cache, 0, q, k, v, mask, scale, out, lse)
            torch.cuda.synchronize()
            assert torch.equal(out, ref), f"step {t} call {call}: differs from swa_decode"
            assert torch.equal(lse, ref_lse), f"step {t} call {call}: lse differs from swa_decode"
            assert_close(out, ref_o[t], f"{name} step {t} call {call}")
            assert_lse(lse, ref_l[t], f"{name} step {t} call {call} lse")
    cache.check()


def test_noalloc_rejects_oversized_shapes(swa):
    # 600 slabs of a 128-row cache take two splits each, merged through the
    # scratch: 9.8 MB of partials, more than the static array holds -- refused
    # on the host before any kernel runs
    B, Hq, Hkv, D, W = 300, 16, 2, 256, 64
    cache = swa.Cache(swa.CACHE_COMPACT, 1, B, Hkv, D, W, 200)
    need = swa.decode_workspace_bytes(cache, Hq)
    assert need > 8 << 20
    mask = torch.zeros(B, cache.rows, dtype=torch.uint8, device="cuda")
    swa.build_decode_mask(cache, mask)
    q = torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(B, Hkv, D, dtype=torch.bfloat16, device="cuda")
    st = swa.lib().swa_decode_noalloc(cache.handle, 0, Hq, swa.ptr(q), swa.ptr(kv), swa.ptr(kv), swa.ptr(mask),
                                      ctypes.c_float(1.0), swa.ptr(q), None, swa.stream_handle(None))
    assert st == swa.EUNSUPPORTED
    assert "static array" in swa.last_error()
