"""Seeded synthetic inputs with the shapes of the five workloads.

This module only draws random numbers and lays out integer metadata (lengths,
pads, image blocks, document boundaries); it holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle can take their inputs
from it.  Everything is drawn on the CPU with ``torch.Generator`` so both
sides see the same bf16 bits.

Recipe (seed = 1000 + workload number, draws in the order listed):

1. tiny causal SWA: B=1, Hq=4, Hkv=2, D=256, W=64, S=200, 70 decode steps.
   prompt q, k, v ~ N(0,1); decode q, k, v ~ N(0,1).
2. single-stream decode: B=1, Hq=4, Hkv=2, D=256, W=1024, S=8192, 26 layers,
   512 decode steps. prompt q, k, v [L, B, S, H, D]; decode q, k, v
   [T, L, B, H, D]; all N(0,1).
3. batched decode: B=64, Hq=16, Hkv=8, D=256, W=1024, 256 decode steps.
   prompt k, v for the last W positions [B, W, Hkv, D]; decode q, k, v;
   then lengths ~ U{16..8192}, S = max(lengths), pad_b = S - len_b; then
   "finite garbage" (100 x N(0,1)) written into the prompt rows of pad
   positions, which must receive zero weight.
4. chunked prefill + VLM: B=4, S=8192 (chunks of 2048), Hq=8, Hkv=4, D=256,
   W=1024. q, k, v ~ N(0,1); then pad_b ~ U{0..512}; sequence 1 carries
   image blocks at padded positions [1536,1792), [2560,2816), [5120,5376),
   [5376,5632) with ids 0..3 (the last two are adjacent, distinct ids).
5. packed varlen forward: 4 documents of 4096 tokens (T=16384), Hq=16, Hkv=8,
   D=512, W=4096; q, k ~ N(0, std 1/sqrt(D)), v ~ N(0,1).

Backward (training) cases add an upstream gradient dout ~ N(0,1) of the
output's shape, drawn from its own generator (seed + 500) so the forward
inputs stay the same draws.

Normal draws are float32 ``torch.randn`` rounded to bf16 (round to nearest
even).  The same generators build smaller cases for the parity tests.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

SEED_BASE = 1000


def _normal(gen: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(tuple(shape), generator=gen, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


@dataclass
class DecodeCase:
    """A prompt already in the cache followed by ``steps`` decode tokens."""
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    window: int
    prompt_len: int            # S (padded)
    steps: int
    layers: int
    prompt_k: torch.Tensor     # [L, B, P, Hkv, D], positions [S-P, S)
    prompt_v: torch.Tensor
    dec_q: torch.Tensor        # [T, L, B, Hq, D]
    dec_k: torch.Tensor        # [T, L, B, Hkv, D]
    dec_v: torch.Tensor
    valid_start: torch.Tensor  # [B] int32
    prompt_q: Optional[torch.Tensor] = None   # [L, B, S, Hq, D] when the prompt is prefilled too


@dataclass
class PrefillCase:
    """A left-padded batch prefilled in chunks (cache mode)."""
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    window: int
    seq_len: int
    chunk: int
    q: torch.Tensor            # [B, S, Hq, D]
    k: torch.Tensor            # [B, S, Hkv, D]
    v: torch.Tensor
    valid_start: torch.Tensor  # [B] int32
    img_id: Optional[torch.Tensor] = None   # [B, S] int32, -1 = text


@dataclass
class VarlenCase:
    """Packed documents (no cache)."""
    q_heads: int
    kv_heads: int
    head_dim: int
    window: int
    q: torch.Tensor            # [T, Hq, D]
    k: torch.Tensor            # [T, Hkv, D]
    v: torch.Tensor
    cu_seqlens: torch.Tensor   # [docs + 1] int32
    extra: dict = field(default_factory=dict)


# --------------------------------------------------------------------------- decode
def decode_case(seed: int, *, batch: int, q_heads: int, kv_heads: int, head_dim: int,
                window: int, prompt_len: int, steps: int, layers: int = 1,
                with_prompt_q: bool = False, prompt_rows: Optional[int] = None,
                lengths: Optional[tuple] = None, garbage: float = 0.0) -> DecodeCase:
    """Generic decode workload.

    ``prompt_rows`` (default: the whole prompt) limits the stored prompt to
    its last rows; ``lengths=(lo, hi)`` draws per-sequence lengths uniformly
    and pads on the left up to ``prompt_len`` (or to the largest length when
    ``prompt_len`` is 0); ``garbage`` > 0 overwrites pad positions of the
    stored prompt with ``garbage * N(0,1)``.
    """
    gen = torch.Generator().manual_seed(seed)
    p_rows = prompt_len if prompt_rows is None else prompt_rows
    pq = None
    if with_prompt_q:
        pq = _normal(gen, (layers, batch, prompt_len, q_heads, head_dim))
    pk = _normal(gen, (layers, batch, p_rows, kv_heads, head_dim))
    pv = _normal(gen, (layers, batch, p_rows, kv_heads, head_dim))
    dq = _normal(gen, (steps, layers, batch, q_heads, head_dim))
    dk = _normal(gen, (steps, layers, batch, kv_heads, head_dim))
    dv = _normal(gen, (steps, layers, batch, kv_heads, head_dim))
    if lengths is not None:
        lens = torch.randint(lengths[0], lengths[1] + 1, (batch,), generator=gen, dtype=torch.int64)
        s = prompt_len if prompt_len > 0 else int(lens.max())
        vs = (s - lens).to(torch.int32)
        prompt_len = s
    else:
        vs = torch.zeros(batch, dtype=torch.int32)
    if prompt_rows is None:
        p_rows = prompt_len
    if garbage > 0.0:
        gk = _normal(gen, pk.shape, garbage)
        gv = _normal(gen, pv.shape, garbage)
        start = prompt_len - p_rows
        pos = start + torch.arange(p_rows)
        for b in range(batch):
            pad = pos < int(vs[b])
            pk[:, b, pad] = gk[:, b, pad]
            pv[:, b, pad] = gv[:, b, pad]
    return DecodeCase(batch, q_heads, kv_heads, head_dim, window, prompt_len, steps, layers,
                      pk, pv, dq, dk, dv, vs, pq)


def workload1() -> DecodeCase:
    """Tiny causal SWA: prefill S=200 then 70 decode steps across one roll."""
    return decode_case(SEED_BASE + 1, batch=1, q_heads=4, kv_heads=2, head_dim=256, window=64,
                       prompt_len=200, steps=70, layers=1, with_prompt_q=True)


def workload2(layers: int = 26, steps: int = 512, with_prompt_q: bool = True) -> DecodeCase:
    """Gemma-like single-stream decode: prompt 8192, positions 8192..8703, 26 layers."""
    return decode_case(SEED_BASE + 2, batch=1, q_heads=4, kv_heads=2, head_dim=256, window=1024,
                       prompt_len=8192, steps=steps, layers=layers, with_prompt_q=with_prompt_q)


def workload3(steps: int = 256) -> DecodeCase:
    """Batched serving decode: 64 left-padded sequences, lengths U{16..8192}."""
    return decode_case(SEED_BASE + 3, batch=64, q_heads=16, kv_heads=8, head_dim=256, window=1024,
                       prompt_len=0, steps=steps, layers=1, prompt_rows=1024,
                       lengths=(16, 8192), garbage=100.0)


# --------------------------------------------------------------------------- prefill
def prefill_case(seed: int, *, batch: int, q_heads: int, kv_heads: int, head_dim: int,
                 window: int, seq_len: int, chunk: int, max_pad: int = 0,
                 images: Optional[dict] = None) -> PrefillCase:
    """Generic chunked-prefill workload; ``images`` maps a sequence to its
    list of (start, end) image blocks (ids are assigned 0, 1, ... in order)."""
    gen = torch.Generator().manual_seed(seed)
    q = _normal(gen, (batch, seq_len, q_heads, head_dim))
    k = _normal(gen, (batch, seq_len, kv_heads, head_dim))
    v = _normal(gen, (batch, seq_len, kv_heads, head_dim))
    if max_pad > 0:
        vs = torch.randint(0, max_pad + 1, (batch,), generator=gen, dtype=torch.int64).to(torch.int32)
    else:
        vs = torch.zeros(batch, dtype=torch.int32)
    img = None
    if images:
        img = torch.full((batch, seq_len), -1, dtype=torch.int32)
        for b, blocks in images.items():
            for i, (s0, s1) in enumerate(blocks):
                img[b, s0:s1] = i
    return PrefillCase(batch, q_heads, kv_heads, head_dim, window, seq_len, chunk, q, k, v, vs, img)


WORKLOAD4_IMAGES = {1: [(1536, 1792), (2560, 2816), (5120, 5376), (5376, 5632)]}


def workload4() -> PrefillCase:
    """Chunked causal prefill plus VLM mask (generic plan)."""
    return prefill_case(SEED_BASE + 4, batch=4, q_heads=8, kv_heads=4, head_dim=256, window=1024,
                        seq_len=8192, chunk=2048, max_pad=512, images=WORKLOAD4_IMAGES)


def varlen_case(seed: int, *, doc_lens, q_heads: int, kv_heads: int, head_dim: int,
                window: int, qk_std: Optional[float] = None) -> VarlenCase:
    gen = torch.Generator().manual_seed(seed)
    total = int(sum(doc_lens))
    std = head_dim ** -0.5 if qk_std is None else qk_std
    q = _normal(gen, (total, q_heads, head_dim), std)
    k = _normal(gen, (total, kv_heads, head_dim), std)
    v = _normal(gen, (total, kv_heads, head_dim))
    cu = [0]
    for n in doc_lens:
        cu.append(cu[-1] + int(n))
    return VarlenCase(q_heads, kv_heads, head_dim, window, q, k, v, torch.tensor(cu, dtype=torch.int32))


def upstream_grad(seed: int, shape) -> torch.Tensor:
    """dL/dout for a backward case: N(0,1) in bf16 from generator seed + 500."""
    return _normal(torch.Generator().manual_seed(seed + 500), shape)


def workload5() -> VarlenCase:
    """Packed varlen forward, training shape: 4 x 4096 tokens, D=512, W=4096."""
    return varlen_case(SEED_BASE + 5, doc_lens=[4096] * 4, q_heads=16, kv_heads=8, head_dim=512,
                       window=4096)
