"""The benchmark's single-stream job computes the same thing however its
steps are staged.

The job stages each decode step's q / k_new / v_new into one of two buffer
sets on a copy stream while the previous step's graph runs, and copies each
step's outputs out the same way; end to end the copies are host uploads and
downloads.  Three runs of a small job must give bit-identical outputs at
every (step, layer): host buffers with the overlapped copies, device buffers
with the overlapped copies, and the in-line staging (one buffer set, the copy
before each step) that the L2-flushed variant uses.  The last step's
outputs of the first and last layer are also checked against the oracle.
"""

import pytest
import torch

import bench
from oracle import reference
from sliding_window_gqa_swa_gb300 import synth
from tests._gpu import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def swa():
    from tests._lib import ensure_built
    ensure_built()
    from sliding_window_gqa_swa_gb300 import swa as mod
    return mod


def test_staging_modes_agree_and_match_oracle(swa):
    dev = torch.device("cuda")
    case = synth.workload2(layers=3, steps=70)  # one roll
    outs = []
    for kw in ({"e2e": True}, {}, {"l2_flush": torch.empty(1 << 20, dtype=torch.uint8, device=dev)}):
        job = bench.SingleStreamJob(swa, case, dev, **kw)
        for _ in range(2):  # the first run captures the step graphs
            job.run(job.make_events())
        torch.cuda.synchronize()
        outs.append(job.outs.cpu())
        del job
    for name, o in zip(("device buffers, overlapped", "in-line staging"), outs[1:]):
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16)), f"{name} differs from host buffers"
    W, S, T = case.window, case.prompt_len, case.steps
    for layer in (0, case.layers - 1):
        ro, _ = reference.decode_full(case.prompt_k[layer][:, -W:], case.prompt_v[layer][:, -W:],
                                      case.dec_q[:, layer], case.dec_k[:, layer], case.dec_v[:, layer],
                                      S, W, case.head_dim ** -0.5, None, steps=[T - 1])
        assert_close(outs[0][T - 1, layer], ro[T - 1], f"layer {layer}, last step")
