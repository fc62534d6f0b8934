"""End to end on the GPU: prefill -> compaction -> decode across a roll.

The tiny workload (prompt 200, window 64, 70 decode steps crossing one roll)
through the C ABI, against the fp64 oracle:
  * prefill outputs and lse within the tolerances;
  * the prefill cache, the compact cache after compaction, and the compact
    cache after every decode step and the roll, bit for bit against the
    oracle's index model (CompactModel);
  * the runtime decode mask bit for bit at every step;
  * the device state (origin, next_row, cur_row, step) at every step;
  * every decode output and lse against the full-length oracle decode;
  * one captured CUDA graph (mask + decode) replayed across positions gives
    the eager results (the pages' graph-reuse observation).
The same checks run through the modular ring cache (W rows, position p in
row p % W, no roll) against the oracle's RingModel.
"""

import numpy as np
import pytest
import torch

from oracle import reference
from oracle.compact import CompactModel, RingModel
from sliding_window_gqa_swa_gb300 import synth
from tests._gpu import assert_close, assert_lse, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swa():
    from tests._lib import ensure_built
    ensure_built()
    from sliding_window_gqa_swa_gb300 import swa as mod
    return mod


def _full_kv(c, b, t_count):
    """Full-length K/V (positions 0 .. S+t_count-1) of layer 0, sequence b."""
    k = torch.cat([c.prompt_k[0, b], c.dec_k[:t_count, 0, b]]).double().numpy()
    v = torch.cat([c.prompt_v[0, b], c.dec_v[:t_count, 0, b]]).double().numpy()
    return k, v


def run_decode_case(swa, c, check_every_step=True, ring=False):
    dev = torch.device("cuda")
    S, W, D = c.prompt_len, c.window, c.head_dim
    B, Hq, Hkv = c.batch, c.q_heads, c.kv_heads
    scale = D ** -0.5
    steps = c.steps
    vs = c.valid_start.to(dev)

    out = lse = None
    cmp_ = swa.Cache(swa.CACHE_RING if ring else swa.CACHE_COMPACT, 1, B, Hkv, D, W, S, vs)
    if D in (256, 512):
        # the whole path: prefill into the prompt-sized cache, then compaction
        pre = swa.Cache(swa.CACHE_PREFILL, 1, B, Hkv, D, W, S, vs)
        q = (c.prompt_q[0] if c.prompt_q is not None else torch.zeros(B, S, Hq, D, dtype=torch.bfloat16)).to(dev)
        k = c.prompt_k[0].to(dev).contiguous()
        v = c.prompt_v[0].to(dev).contiguous()
        meta = swa.Meta(B, S, 0, S, W, valid_start=vs)
        out = torch.empty_like(q)
        lse = torch.empty(B, S, Hq, dtype=torch.float32, device=dev)
        swa.prefill(pre, 0, swa.MODE_CAUSAL, q, k, v, meta, scale, out, lse)
        torch.cuda.synchronize()
        assert np.array_equal(bits(pre.k[0, :, :, :S].transpose(1, 2)), bits(c.prompt_k[0]))
        assert np.array_equal(bits(pre.v[0, :, :, :S].transpose(1, 2)), bits(c.prompt_v[0]))
        swa.compact(pre, cmp_)
    else:
        # prefill supports D = 256 / 512 only: place the prompt's last W positions
        # as compaction would (decode-only head sizes): anchored rows
        # [max(0, W - S), W), or ring rows pos % W
        n = min(S, W)
        if ring:
            for pos in range(S - n, S):
                cmp_.k[0, :, :, pos % W] = c.prompt_k[0, :, pos].to(dev)
                cmp_.v[0, :, :, pos % W] = c.prompt_v[0, :, pos].to(dev)
        else:
            cmp_.k[0, :, :, W - n:W] = c.prompt_k[0, :, S - n:].transpose(1, 2).to(dev)
            cmp_.v[0, :, :, W - n:W] = c.prompt_v[0, :, S - n:].transpose(1, 2).to(dev)
    model = RingModel(S, W) if ring else CompactModel(S, W)
    torch.cuda.synchronize()
    for b in range(B):
        fk, _ = _full_kv(c, b, 0)
        exp_k = torch.from_numpy(model.expected_cache(fk)).to(torch.bfloat16)
        assert np.array_equal(bits(cmp_.k[0, b].transpose(0, 1)), bits(exp_k))

    ref_o, ref_l = reference.decode_full(c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0],
                                         c.dec_v[:, 0], S, W, scale, c.valid_start.numpy())
    mask = torch.empty(B, cmp_.rows, dtype=torch.uint8, device=dev)
    ws = swa.decode_workspace(cmp_, Hq)
    dq, dk, dv = c.dec_q[:, 0].to(dev), c.dec_k[:, 0].to(dev), c.dec_v[:, 0].to(dev)
    outs, lses = [], []
    for t in range(steps):
        if model.needs_roll():
            assert cmp_.needs_roll()
            swa.roll(cmp_)
            model.roll()
        swa.build_decode_mask(cmp_, mask)
        mexp = model.begin_step(c.valid_start.numpy())
        o = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
        l = torch.empty(B, Hq, dtype=torch.float32, device=dev)
        swa.decode(cmp_, 0, dq[t], dk[t], dv[t], mask, scale, o, ws, l)
        outs.append(o)
        lses.append(l)
        if check_every_step or t in (0, steps - 1) or model.step % 64 in (0, 1):
            torch.cuda.synchronize()
            assert np.array_equal(mask.cpu().numpy().astype(bool), mexp), f"mask differs at step {t}"
            st = cmp_.state()
            if ring:
                exp_st = (0, (S + model.step) % W, model.cur_row, model.step, 0)
            else:
                exp_st = (model.origin, model.next_row, model.cur_row, model.step, 0)
            assert (st["origin"], st["next_row"], st["cur_row"], st["step"], st["error"]) == exp_st, (t, st)
            for b in range(B):
                fk, fv = _full_kv(c, b, t + 1)
                ek = torch.from_numpy(model.expected_cache(fk)).to(torch.bfloat16)
                ev = torch.from_numpy(model.expected_cache(fv)).to(torch.bfloat16)
                assert np.array_equal(bits(cmp_.k[0, b].transpose(0, 1)), bits(ek)), f"K differs at step {t}"
                assert np.array_equal(bits(cmp_.v[0, b].transpose(0, 1)), bits(ev)), f"V differs at step {t}"
    torch.cuda.synchronize()
    cmp_.check()
    return out, lse, torch.stack(outs), torch.stack(lses), ref_o, ref_l


def test_workload1_prefill_compact_decode(swa):
    c = synth.workload1()
    out, lse, dec_o, dec_l, ref_o, ref_l = run_decode_case(swa, c)
    po, pl = reference.prefill(c.prompt_q[0], c.prompt_k[0], c.prompt_v[0], c.window, c.head_dim ** -0.5,
                               c.valid_start.numpy())
    assert_close(out, po, "prefill")
    assert_lse(lse, pl, "prefill lse")
    assert_close(dec_o, ref_o, "decode")
    assert_lse(dec_l, ref_l, "decode lse")


# covers the three ways a decode merges its splits: one split per slab, one
# cluster per slab, and the workspace merge (many splits of a long window)
@pytest.mark.parametrize("batch,hq,hkv,d,w,s", [(3, 4, 2, 256, 64, 40), (2, 8, 2, 128, 64, 300),
                                                (2, 8, 1, 64, 128, 129), (1, 8, 8, 512, 64, 100),
                                                (1, 2, 1, 256, 4096, 4200), (1, 4, 2, 256, 1024, 1500)])
def test_decode_shapes_with_padding(swa, batch, hq, hkv, d, w, s):
    c = synth.decode_case(3100 + d + hq, batch=batch, q_heads=hq, kv_heads=hkv, head_dim=d, window=w,
                          prompt_len=s, steps=140, layers=1, with_prompt_q=False)
    vs = torch.tensor([0, min(s - 1, 13), 5][:batch], dtype=torch.int32)
    c.valid_start = vs
    # pad positions carry finite garbage that must get zero weight
    for b in range(batch):
        c.prompt_k[0, b, :int(vs[b])] = 50.0
        c.prompt_v[0, b, :int(vs[b])] = -70.0
    _, _, dec_o, dec_l, ref_o, ref_l = run_decode_case(swa, c, check_every_step=False)
    assert_close(dec_o, ref_o, "decode")
    assert_lse(dec_l, ref_l, "decode lse")


# The throughput regime (at least as many (sequence, KV head) slabs as SMs):
# eight compute warps per CTA, a few row-range splits per slab merged through
# the workspace.  Sequences of every length from one prompt token up (left
# padding filled with large finite garbage), so some splits admit no row and
# some a single one, across a roll; head sizes 64 to 512, groups of 1 to 8.
@pytest.mark.parametrize("batch,hq,hkv,d,w,s", [(40, 8, 4, 256, 64, 150), (20, 16, 8, 128, 256, 300),
                                                (160, 2, 1, 512, 128, 200), (40, 32, 4, 64, 128, 140),
                                                (80, 2, 2, 256, 256, 400)])
def test_throughput_regime_length_mix(swa, batch, hq, hkv, d, w, s):
    c = synth.decode_case(3600 + d + hq, batch=batch, q_heads=hq, kv_heads=hkv, head_dim=d, window=w,
                          prompt_len=s, steps=70, layers=1, with_prompt_q=False, lengths=(1, s), garbage=50.0)
    _, _, dec_o, dec_l, ref_o, ref_l = run_decode_case(swa, c, check_every_step=False)
    assert_close(dec_o, ref_o, "decode")
    assert_lse(dec_l, ref_l, "decode lse")


def test_workload1_ring(swa):
    c = synth.workload1()
    _, _, dec_o, dec_l, ref_o, ref_l = run_decode_case(swa, c, ring=True)
    assert_close(dec_o, ref_o, "ring decode")
    assert_lse(dec_l, ref_l, "ring decode lse")


@pytest.mark.parametrize("batch,hq,hkv,d,w,s", [(3, 4, 2, 256, 64, 40), (2, 8, 2, 128, 64, 300),
                                                (1, 4, 2, 256, 1024, 1500)])
def test_ring_decode_shapes_with_padding(swa, batch, hq, hkv, d, w, s):
    c = synth.decode_case(3300 + d + hq, batch=batch, q_heads=hq, kv_heads=hkv, head_dim=d, window=w,
                          prompt_len=s, steps=140, layers=1, with_prompt_q=False)
    vs = torch.tensor([0, min(s - 1, 13), 5][:batch], dtype=torch.int32)
    c.valid_start = vs
    for b in range(batch):
        c.prompt_k[0, b, :int(vs[b])] = 50.0
        c.prompt_v[0, b, :int(vs[b])] = -70.0
    _, _, dec_o, dec_l, ref_o, ref_l = run_decode_case(swa, c, check_every_step=False, ring=True)
    assert_close(dec_o, ref_o, "ring decode")
    assert_lse(dec_l, ref_l, "ring decode lse")


def test_ring_never_rolls(swa):
    dev = torch.device("cuda")
    cache = swa.Cache(swa.CACHE_RING, 1, 1, 2, 256, 64, 100)
    assert cache.rows == 64 and not cache.needs_roll()
    mask = torch.empty(1, 64, dtype=torch.uint8, device=dev)
    for _ in range(130):
        swa.build_decode_mask(cache, mask)
    assert not cache.needs_roll()
    with pytest.raises(swa.SwaError):
        swa.roll(cache)
    torch.cuda.synchronize()
    st = cache.state()
    assert (st["next_row"], st["cur_row"], st["step"], st["error"]) == ((100 + 130) % 64, (100 + 129) % 64, 130, 0)


@pytest.mark.parametrize("ring", [False, True])
def test_graph_replay_matches_eager(swa, ring):
    """One captured graph (mask + decode) serves every position between rolls."""
    dev = torch.device("cuda")
    c = synth.decode_case(3200, batch=2, q_heads=4, kv_heads=2, head_dim=256, window=64, prompt_len=150,
                          steps=130, layers=1)
    S, W, D, B, Hq, Hkv = c.prompt_len, c.window, c.head_dim, c.batch, c.q_heads, c.kv_heads
    scale = D ** -0.5
    results = {}
    for use_graph in (False, True):
        pre = swa.Cache(swa.CACHE_PREFILL, 1, B, Hkv, D, W, S)
        swa.prefill(pre, 0, swa.MODE_CAUSAL, torch.zeros(B, S, Hq, D, dtype=torch.bfloat16, device=dev),
                    c.prompt_k[0].to(dev), c.prompt_v[0].to(dev), swa.Meta(B, S, 0, S, W), scale,
                    torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev))
        cache = swa.Cache(swa.CACHE_RING if ring else swa.CACHE_COMPACT, 1, B, Hkv, D, W, S)
        swa.compact(pre, cache)
        mask = torch.empty(B, cache.rows, dtype=torch.uint8, device=dev)
        ws = swa.decode_workspace(cache, Hq)
        qb = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
        kb = torch.empty(B, Hkv, D, dtype=torch.bfloat16, device=dev)
        vb = torch.empty_like(kb)
        ob = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
        outs = []
        graph = None
        for t in range(c.steps):
            if cache.needs_roll():
                swa.roll(cache)
            qb.copy_(c.dec_q[t, 0])
            kb.copy_(c.dec_k[t, 0])
            vb.copy_(c.dec_v[t, 0])
            if not use_graph or t == 0:
                swa.build_decode_mask(cache, mask)
                swa.decode(cache, 0, qb, kb, vb, mask, scale, ob, ws)
            elif graph is None:
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=s):
                    swa.build_decode_mask(cache, mask, stream=s)
                    swa.decode(cache, 0, qb, kb, vb, mask, scale, ob, ws, stream=s)
                torch.cuda.current_stream().wait_stream(s)
                # the capture advanced the host mirror once without running a
                # kernel; this first replay advances the device to match
                graph.replay()
            else:
                graph.replay()
                cache.advance(1)
            outs.append(ob.clone())
        torch.cuda.synchronize()
        cache.check()
        results[use_graph] = torch.stack(outs)
    assert np.array_equal(bits(results[False]), bits(results[True]))


def test_inputs_ready_chain_under_graph(swa):
    """SWA_DECODE_INPUTS_READY: with every layer's inputs of a step staged before
    the step's mask, layers 1.. read them before waiting for the previous
    layer's decode.  One captured graph per step (mask + three layers) replayed
    across two rolls gives the same bits as plain decodes, and the oracle's
    results."""
    dev = torch.device("cuda")
    L = 3
    c = synth.decode_case(3300, batch=1, q_heads=4, kv_heads=2, head_dim=256, window=64, prompt_len=150,
                          steps=130, layers=L)
    S, W, D, B, Hq, Hkv = c.prompt_len, c.window, c.head_dim, c.batch, c.q_heads, c.kv_heads
    scale = D ** -0.5
    results = {}
    for ready in (False, True):
        pre = swa.Cache(swa.CACHE_PREFILL, L, B, Hkv, D, W, S)
        for layer in range(L):
            swa.prefill(pre, layer, swa.MODE_CAUSAL, torch.zeros(B, S, Hq, D, dtype=torch.bfloat16, device=dev),
                        c.prompt_k[layer].to(dev), c.prompt_v[layer].to(dev), swa.Meta(B, S, 0, S, W), scale,
                        torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev))
        cache = swa.Cache(swa.CACHE_COMPACT, L, B, Hkv, D, W, S)
        swa.compact(pre, cache)
        mask = torch.empty(B, cache.rows, dtype=torch.uint8, device=dev)
        ws = swa.decode_workspace(cache, Hq)
        qb = torch.empty(L, B, Hq, D, dtype=torch.bfloat16, device=dev)
        kb = torch.empty(L, B, Hkv, D, dtype=torch.bfloat16, device=dev)
        vb = torch.empty_like(kb)
        ob = torch.empty(L, B, Hq, D, dtype=torch.bfloat16, device=dev)

        def step(stream=None):
            swa.build_decode_mask(cache, mask, stream=stream)
            for layer in range(L):
                swa.decode(cache, layer, qb[layer], kb[layer], vb[layer], mask, scale, ob[layer], ws,
                           stream=stream, inputs_ready=ready and layer > 0)

        outs = []
        graph = None
        for t in range(c.steps):
            if cache.needs_roll():
                swa.roll(cache)
            qb.copy_(c.dec_q[t])
            kb.copy_(c.dec_k[t])
            vb.copy_(c.dec_v[t])
            if t == 0:
                step()
            elif graph is None:
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=s):
                    step(stream=s)
                torch.cuda.current_stream().wait_stream(s)
                graph.replay()  # the capture advanced only the host mirror
            else:
                graph.replay()
                cache.advance(1)
            outs.append(ob.clone())
        torch.cuda.synchronize()
        cache.check()
        results[ready] = torch.stack(outs)
    assert np.array_equal(bits(results[False]), bits(results[True]))
    check = [0, 1, 63, 64, 65, 127, 128, 129]
    for layer in range(L):
        ro, _ = reference.decode_full(c.prompt_k[layer], c.prompt_v[layer], c.dec_q[:, layer], c.dec_k[:, layer],
                                      c.dec_v[:, layer], S, W, scale, steps=check)
        for t in check:
            assert_close(results[True][t, layer], ro[t], f"inputs-ready chain step {t} layer {layer}")


def test_kv_sharing_layer(swa):
    """A KV-sharing layer (k_new = v_new = NULL) attends over the owning
    layer's rows, which already hold the step's token, and appends nothing."""
    dev = torch.device("cuda")
    c = synth.decode_case(3400, batch=2, q_heads=4, kv_heads=2, head_dim=256, window=64, prompt_len=150,
                          steps=90, layers=1)
    S, W, D, B, Hq, Hkv = c.prompt_len, c.window, c.head_dim, c.batch, c.q_heads, c.kv_heads
    scale = D ** -0.5
    gen = torch.Generator().manual_seed(3401)
    q_share = torch.randn(c.steps, B, Hq, D, generator=gen).to(torch.bfloat16)
    pre = swa.Cache(swa.CACHE_PREFILL, 1, B, Hkv, D, W, S)
    swa.prefill(pre, 0, swa.MODE_CAUSAL, torch.zeros(B, S, Hq, D, dtype=torch.bfloat16, device=dev),
                c.prompt_k[0].to(dev), c.prompt_v[0].to(dev), swa.Meta(B, S, 0, S, W), scale,
                torch.empty(B, S, Hq, D, dtype=torch.bfloat16, device=dev))
    cache = swa.Cache(swa.CACHE_COMPACT, 1, B, Hkv, D, W, S)
    swa.compact(pre, cache)
    mask = torch.empty(B, cache.rows, dtype=torch.uint8, device=dev)
    ws = swa.decode_workspace(cache, Hq)
    model = CompactModel(S, W)
    own, shared = [], []
    for t in range(c.steps):
        if cache.needs_roll():
            swa.roll(cache)
            model.roll()
        swa.build_decode_mask(cache, mask)
        model.begin_step(np.zeros(B))
        o1 = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=dev)
        o2 = torch.empty_like(o1)
        swa.decode(cache, 0, c.dec_q[t, 0].to(dev), c.dec_k[t, 0].to(dev), c.dec_v[t, 0].to(dev), mask, scale,
                   o1, ws)
        swa.decode(cache, 0, q_share[t].to(dev), None, None, mask, scale, o2, ws)
        own.append(o1)
        shared.append(o2)
    torch.cuda.synchronize()
    cache.check()
    # the sharing calls appended nothing: the cache holds exactly the owner's rows
    for b in range(B):
        fk, fv = _full_kv(c, b, c.steps)
        ek = torch.from_numpy(model.expected_cache(fk)).to(torch.bfloat16)
        assert np.array_equal(bits(cache.k[0, b].transpose(0, 1)), bits(ek))
    args = (c.prompt_k[0], c.prompt_v[0], None, c.dec_k[:, 0], c.dec_v[:, 0], S, W, scale, c.valid_start.numpy())
    ro, _ = reference.decode_full(args[0], args[1], c.dec_q[:, 0], *args[3:])
    rs, _ = reference.decode_full(args[0], args[1], q_share, *args[3:])
    assert_close(torch.stack(own), ro, "owner")
    assert_close(torch.stack(shared), rs, "KV-sharing layer")


def test_global_layer_as_unbounded_window(swa):
    """A global (full causal) layer through the same path: a window at least as
    long as every position the job reaches (W >= S + steps); the rolls then
    drop only rows of negative positions."""
    S, T = 150, 130
    c = synth.decode_case(3500, batch=1, q_heads=4, kv_heads=2, head_dim=256, window=S + T, prompt_len=S,
                          steps=T, layers=1)
    _, _, dec_o, dec_l, ref_o, ref_l = run_decode_case(swa, c, check_every_step=False)
    assert_close(dec_o, ref_o, "global-layer decode")
    assert_lse(dec_l, ref_l, "global-layer decode lse")
