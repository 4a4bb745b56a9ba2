"""Failure detection on the GPU without a fault: a bounded pipeline wait that
nothing completes gives up after its limit and reports DUALKV_ERR_TIMEOUT and
its site through the device error word.  The kernel returns normally, so the
context stays usable and the next call runs clean."""
import time

import pytest
import torch

from shared_prompt_exact_dualkv_gb300 import synthetic

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    assert D.dualkv_last_device_error() == (D.DUALKV_OK, 0)
    t0 = time.perf_counter()
    D.dualkv_selftest_wait_timeout(20_000_000, 4242)      # 20 ms limit
    st, site = D.dualkv_last_device_error()                # synchronises
    elapsed = time.perf_counter() - t0
    assert (st, site) == (D.DUALKV_ERR_TIMEOUT, 4242)
    assert 0.02 <= elapsed < 5.0
    # reading the word cleared it
    assert D.dualkv_last_device_error() == (D.DUALKV_OK, 0)
    # the context is intact: a real forward + backward runs and is clean
    w = synthetic.WORKLOADS["tiny"]
    x = synthetic.make_inputs(w, 0)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    out, lse = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    D.backward(q, k, v, out, do, lse, w.P, w.R_lens, w.scale)
    assert D.dualkv_last_device_error() == (D.DUALKV_OK, 0)
    assert torch.isfinite(out.float()).all()
