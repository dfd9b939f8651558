"""Failure handling on the GPU without a fault: a bounded wait that runs out.

Every pipeline wait of the library (TMA stages, MMA completion, softmax
hand-offs) is bounded; when one gives up, the kernel records an error word
and returns instead of hanging.  te_selftest_wait_timeout runs the same
bounded wait on a barrier nothing arrives at, with a short limit.  The host
must then see TE_EDEVICE from te_check, the error must clear, and the context
must stay usable for ordinary work.
"""
import numpy as np
import pytest

import transformer_encoder_forward_gb300 as te
from oracle import encoder as O
from tests.gpu_util import bf16_input, rel_frob, to_dev, to_np
from transformer_encoder_forward_gb300 import synth

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    import torch
    te.check()                                   # nothing pending before
    te.selftest_wait_timeout(2000)               # 2 ms limit
    with pytest.raises(te.TEError) as ei:
        te.check()
    assert ei.value.status == te.TE_EDEVICE
    assert "bounded wait gave up" in str(ei.value)
    te.check()                                   # the error word was cleared
    # ordinary work still runs and is correct afterwards
    rng = np.random.default_rng(3)
    m, k, n = 97, 256, 128
    x, x64 = bf16_input(rng, (m, k))
    w = synth.draw_q8(rng, n, k, True, False)
    y = torch.empty(m, n, dtype=torch.float32, device="cuda")
    te.q8_linear(x, [{"w": te.q8w(to_dev(w["q"]), to_dev(w["s"])), "y": y, "ldy": n}])
    te.check()
    assert rel_frob(to_np(y), O.q8_linear(x64, w["q"], w["s"])) < 1e-3


def test_selftest_rejects_bad_limits():
    with pytest.raises(te.TEError):
        te.selftest_wait_timeout(0)
