"""Plain fp64 CPU oracle for sliding-window grouped-query attention.

TEST INFRASTRUCTURE ONLY. This package is what the CUDA path is checked
against. Only the test suite, the package smoke check and the CPU-baseline leg
of the benchmark may import it; the library itself never does, and it shares
no code, table or helper with the CUDA sources.

What it computes, and where each rule comes from:

* ``masks``     -- the sliding-layer mask predicate, written out literally
                   (window AND (causal OR same image block), document
                   boundaries, left padding), plus the decode-time mask over a
                   full-length cache.
* ``attention`` -- masked softmax attention in float64 over an explicit key
                   set, with query heads sharing key/value heads (GQA).
* ``backward``  -- the gradients of that attention with respect to q, k and v
                   (the derivative of the forward definition, written out).
* ``compact``   -- an integer model of the anchored W+64-row compact cache:
                   the compaction at first decode, the row written by each
                   decode step, the runtime decode mask, and the roll every 64
                   decode tokens.
* ``reference`` -- whole-workload drivers (prefill of a batch, the decode loop)
                   built from the three modules above.

Page citations use the page title and section:
  [SPYRE]   "Enable compact sliding-window attention for Gemma 3 and Gemma 4
            variants" (torch-spyre/hf-adapters pull request 496).
  [BONSAI]  "Gemma3 Local Attention Cache" (jax-ml/bonsai issue 124).
  [FASTLLM] "Add SDPA attention implementation" (ServiceNow/Fast-LLM pull
            request 512).

Parity pins: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (literal matrices, brute force, a library routine,
closed forms, invariants).  Three conventions are readings the pages leave open
and are therefore "parity unpinned" by the pages themselves (the tests pin the
code to the stated reading, not the reading to the pages): the window width
(0 <= q - k < W), the right-aligned anchoring of the compact cache
(origin = S - W), and the softmax scale (an argument, default 1/sqrt(D)).
"""

from . import masks, attention, backward, compact, reference  # noqa: F401
