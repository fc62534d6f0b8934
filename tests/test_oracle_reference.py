"""Pins of the oracle's workload drivers (CPU only).

* packed documents (cu_seqlens, document-causal mask) equal running every
  document as its own sequence -- cross-document pairs excluded by structure
  instead of by mask, the nested formulation of "Add SDPA attention
  implementation", Summary;
* selected rows equal the same rows of the whole-batch prefill;
* the full-length decode loop equals a prefill over prompt + decode tokens
  read at the decode rows (a decode token is a text query at the next
  position of the same sequence).
"""

import numpy as np

from oracle import reference
from sliding_window_gqa_swa_gb300 import synth


def test_varlen_equals_documents_run_separately():
    c = synth.varlen_case(91, doc_lens=[5, 9, 1, 12], q_heads=4, kv_heads=2, head_dim=8, window=6)
    rows = list(range(int(c.cu_seqlens[-1])))
    o, lse = reference.varlen_rows(c.q, c.k, c.v, c.cu_seqlens.tolist(), c.window, 0.3, rows)
    cu = c.cu_seqlens.tolist()
    for d in range(len(cu) - 1):
        a, b = cu[d], cu[d + 1]
        od, ld = reference.prefill(c.q[None, a:b], c.k[None, a:b], c.v[None, a:b], c.window, 0.3)
        assert np.array_equal(o[a:b], od[0]) and np.array_equal(lse[a:b], ld[0])


def test_rows_equal_whole_prefill():
    c = synth.prefill_case(92, batch=2, q_heads=4, kv_heads=1, head_dim=8, window=5, seq_len=24, chunk=8,
                           max_pad=6, images={1: [(10, 14), (14, 17)]})
    o, lse = reference.prefill(c.q, c.k, c.v, c.window, 0.5, c.valid_start, c.img_id)
    for b in range(2):
        rows = [0, 3, 11, 15, 23]
        ob, lb = reference.prefill_rows(c.q, c.k, c.v, c.window, 0.5, b, rows, c.valid_start, c.img_id)
        assert np.array_equal(ob, o[b, rows]) and np.array_equal(lb, lse[b, rows])


def test_decode_equals_prefill_rows():
    c = synth.decode_case(93, batch=2, q_heads=4, kv_heads=2, head_dim=8, window=7, prompt_len=12,
                          steps=9, layers=1)
    vs = np.array([0, 4])
    o, lse = reference.decode_full(c.prompt_k[0], c.prompt_v[0], c.dec_q[:, 0], c.dec_k[:, 0], c.dec_v[:, 0],
                                   c.prompt_len, c.window, 0.4, vs)
    import torch
    for b in range(2):
        k = torch.cat([c.prompt_k[0, b], c.dec_k[:, 0, b]])[None]
        v = torch.cat([c.prompt_v[0, b], c.dec_v[:, 0, b]])[None]
        q = torch.cat([torch.zeros(12, 4, 8, dtype=c.dec_q.dtype), c.dec_q[:, 0, b]])[None]
        rows = list(range(12, 21))
        ob, lb = reference.prefill_rows(q, k, v, c.window, 0.4, 0, rows, [int(vs[b])])
        assert np.array_equal(ob, o[:, b]) and np.array_equal(lb, lse[:, b])
