"""Pins of the oracle's compact-cache index model (CPU only).

* the hand-derived worked example for the tiny workload (tests/golden);
* the runtime mask admits exactly the positions the full-length decode
  predicate admits, each once (no stale duplicate), at every step;
* compact W+64 attention equals full-cache masked attention bit for bit at
  every step of a 70-step decode over the anchored buffer that crosses one
  roll (the case the Spyre page's Correctness section checks), and over 512
  steps of the
  single-stream shape;
* pad rows and never-written rows get zero weight (bit-identical outputs
  after filling them with large finite values);
* rolls happen exactly every 64 decode steps whatever the prompt length;
* the modular ring (W rows, position p in row p % W) admits the same
  positions as the full-length predicate at every step, never rolls, and its
  decode equals the full-cache decode up to fp64 rounding (its rows come in a
  different order, so the sums differ in their last bits only).
"""

import json
import os

import numpy as np
import pytest

from oracle import masks, reference
from oracle.compact import CompactModel, RingModel
from sliding_window_gqa_swa_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "index_map_s200_w64.json")


def test_worked_example():
    g = json.load(open(GOLDEN))
    m = CompactModel(g["prompt_len"], g["window"])
    assert m.R == g["rows"] and m.origin == g["origin_after_compact"]
    assert m.next_row == g["next_row_after_compact"]
    assert m.held[0] == g["rows_0_63_hold_positions"][0] and m.held[63] == g["rows_0_63_hold_positions"][1]
    assert np.all(m.held[64:] == -1)
    want = {s["step"]: s for s in g["steps"]}
    rolls = []
    for t in range(70):
        if m.needs_roll():
            rolls.append(t)
            m.roll()
        mask = m.begin_step([0])[0]
        if t in want:
            s = want[t]
            assert m.query_position() == s["query_position"]
            assert m.cur_row == s["cur_row"] and m.origin == s["origin"]
            lo, hi = s["allowed_rows"]
            assert np.flatnonzero(mask).tolist() == list(range(lo, hi + 1))
    assert rolls == g["roll_before_steps"]


@pytest.mark.parametrize("prompt_len,window,vs", [(200, 64, 0), (200, 64, 150), (40, 64, 0), (40, 64, 7),
                                                   (1000, 128, 900), (129, 128, 3), (64, 64, 0)])
def test_mask_admits_exactly_the_window(prompt_len, window, vs):
    m = CompactModel(prompt_len, window)
    for t in range(300):
        if m.needs_roll():
            m.roll()
        mask = m.begin_step([vs])[0]
        p = m.query_position()
        got = sorted(m.held[mask].tolist())
        pos = np.arange(0, p + 1)
        exp = pos[masks.decode_mask_full(p, window, vs, pos)].tolist()
        assert got == exp, (t, got[:5], exp[:5])
        # the rows the mask admits hold exactly origin + r
        r = np.flatnonzero(mask)
        assert np.all(m.held[r] == m.origin + r)


@pytest.mark.parametrize("prompt_len", [1, 63, 64, 65, 200, 1023, 8192])
def test_rolls_every_64_steps(prompt_len):
    m = CompactModel(prompt_len, 64)
    rolls = []
    for t in range(260):
        if m.needs_roll():
            rolls.append(t)
            m.roll()
        m.begin_step([0])
    assert rolls == [64, 128, 192, 256]


def test_compact_equals_full_70_steps_across_roll():
    c = synth.workload1()
    args = (c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0], c.dec_v[:, 0], c.prompt_len,
            c.window, c.head_dim ** -0.5, c.valid_start)
    o_full, l_full = reference.decode_full(*args)
    o_cmp, l_cmp = reference.decode_compact(*args)
    assert np.array_equal(o_full, o_cmp) and np.array_equal(l_full, l_cmp)
    assert np.all(np.isfinite(o_full))


def test_compact_equals_full_with_padding_and_short_prompt():
    c = synth.decode_case(77, batch=3, q_heads=4, kv_heads=2, head_dim=16, window=64, prompt_len=40,
                          steps=150, layers=1)
    vs = np.array([0, 5, 39])
    args = (c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0], c.dec_v[:, 0], c.prompt_len,
            c.window, 0.25, vs)
    o_full, l_full = reference.decode_full(*args)
    o_cmp, l_cmp = reference.decode_compact(*args)
    assert np.array_equal(o_full, o_cmp) and np.array_equal(l_full, l_cmp)


@pytest.mark.slow
def test_compact_equals_full_single_stream_512_steps():
    # the single-stream decode shape (one layer, last 1024 prompt rows suffice)
    c = synth.decode_case(2002, batch=1, q_heads=4, kv_heads=2, head_dim=256, window=1024,
                          prompt_len=8192, prompt_rows=1024, steps=512, layers=1)
    args = (c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0], c.dec_v[:, 0], c.prompt_len,
            c.window, c.head_dim ** -0.5, c.valid_start)
    o_full, l_full = reference.decode_full(*args)
    o_cmp, l_cmp = reference.decode_compact(*args)
    assert np.array_equal(o_full, o_cmp) and np.array_equal(l_full, l_cmp)


def test_pad_and_unwritten_rows_get_zero_weight():
    c = synth.decode_case(78, batch=2, q_heads=2, kv_heads=1, head_dim=8, window=64, prompt_len=30,
                          steps=80, layers=1)
    vs = np.array([4, 11])
    args = [c.prompt_k[0].double().numpy(), c.prompt_v[0].double().numpy(), c.dec_q[:, 0], c.dec_k[:, 0],
            c.dec_v[:, 0], c.prompt_len, c.window, 0.5, vs]
    o1, l1 = reference.decode_compact(*args)
    pk, pv = args[0].copy(), args[1].copy()
    for b in range(2):
        pk[b, :vs[b]] = 1e6
        pv[b, :vs[b]] = -1e6
    args[0], args[1] = pk, pv
    o2, l2 = reference.decode_compact(*args)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # never-written rows (negative positions) are zero in the model and masked
    m = CompactModel(30, 64)
    assert np.all(m.held[:34] == -1) and m.held[34] == 0


def test_roll_requires_full_cache():
    m = CompactModel(100, 64)
    with pytest.raises(RuntimeError):
        m.roll()
    for _ in range(64):
        m.begin_step([0])
    with pytest.raises(RuntimeError):
        m.begin_step([0])
    m.roll()
    assert m.origin == 100 and m.next_row == 64


@pytest.mark.parametrize("prompt_len,window,vs", [(200, 64, 0), (200, 64, 150), (40, 64, 0), (40, 64, 7),
                                                   (1000, 128, 900), (129, 128, 3), (64, 64, 0), (5, 3, 1)])
def test_ring_mask_admits_exactly_the_window(prompt_len, window, vs):
    m = RingModel(prompt_len, window)
    for t in range(300):
        assert not m.needs_roll()
        mask = m.begin_step([vs])[0]
        p = m.query_position()
        got = sorted(m.held[mask].tolist())
        pos = np.arange(0, p + 1)
        exp = pos[masks.decode_mask_full(p, window, vs, pos)].tolist()
        assert got == exp, (t, got[:5], exp[:5])
        # every written row holds a position congruent to its index, the
        # current one in row p % W
        w = m.held >= 0
        assert np.all(m.held[w] % window == np.flatnonzero(w))
        assert m.cur_row == p % window and m.held[m.cur_row] == p


def test_ring_equals_full_with_padding_and_short_prompt():
    c = synth.decode_case(78, batch=3, q_heads=4, kv_heads=2, head_dim=16, window=64, prompt_len=40,
                          steps=150, layers=1)
    vs = np.array([0, 5, 39])
    args = (c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0], c.dec_v[:, 0], c.prompt_len,
            c.window, 0.25, vs)
    o_full, l_full = reference.decode_full(*args)
    o_ring, l_ring = reference.decode_compact(*args, ring=True)
    assert np.allclose(o_ring, o_full, rtol=1e-12, atol=1e-12)
    assert np.allclose(l_ring, l_full, rtol=1e-12, atol=1e-12)


def test_ring_equals_full_70_steps():
    c = synth.workload1()
    args = (c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0], c.dec_v[:, 0], c.prompt_len,
            c.window, c.head_dim ** -0.5, c.valid_start)
    o_full, l_full = reference.decode_full(*args)
    o_ring, l_ring = reference.decode_compact(*args, ring=True)
    assert np.allclose(o_ring, o_full, rtol=1e-12, atol=1e-12)
    assert np.allclose(l_ring, l_full, rtol=1e-12, atol=1e-12)
