"""Every pipeline barrier wait in the library's kernels is bounded: a wait that
never completes gives up after its limit, sets GQA_DEVERR_WAIT_TIMEOUT in the
device error word and lets the kernel return, so a stalled pipeline reports an
error instead of hanging the GPU.  gqa_check_wait_limit runs that same wait on
an mbarrier nothing arrives on; this test checks the status it leaves and that
the context is still usable afterwards.  Nothing here faults or hangs the GPU:
the wait ends by its own limit (about 2 s)."""
import time

import numpy as np
import pytest
import torch

import oracle
from long_context_causal_gqa_gb300 import inputs

pytestmark = pytest.mark.gpu

MAX_ABS, REL_L2 = 1e-3, 1e-2   # the pages' FP16 envelope


def test_a_stalled_wait_reports_a_timeout_and_the_context_stays_usable(cuda_lib):
    cuda_lib.device_error()                      # start from a clear error word
    t0 = time.monotonic()
    cuda_lib.check_wait_limit()
    err = cuda_lib.device_error()                # synchronises the stream
    elapsed = time.monotonic() - t0
    assert err & cuda_lib.DEVERR_WAIT_TIMEOUT
    assert 1.0 < elapsed < 60.0, elapsed
    # The context is usable: a prefill afterwards matches the oracle and
    # leaves no error.
    dev = torch.device("cuda")
    d = inputs.dense_inputs(64, 300, seed=11)
    out = cuda_lib.prefill(d.q.to(dev), d.k.to(dev), d.v.to(dev), d.scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_error() == 0
    g = out.float().cpu().numpy().astype(np.float64)
    ref = oracle.dense(d.q, d.k, d.v, d.scale)
    assert np.abs(g - ref).max() <= MAX_ABS
    assert np.linalg.norm(g - ref) / np.linalg.norm(ref) <= REL_L2
