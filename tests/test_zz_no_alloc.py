"""The backward entry point that allocates nothing (dualkv_bwd_static_workspace).

Callers that cannot allocate device memory while they run the backward pass
(a framework whose memory manager owns the whole device, code that must not
risk the implicit synchronisation of cudaMalloc/cudaFree, or a plain-C host
without an allocator) use this entry point: it runs the same backward pass
with the library's fixed 16 MiB device scratch in place of a caller workspace.

This test calls it through the C ABI twice in a row and checks each result
against the regular dualkv_bwd (caller-allocated workspace) within the
gradient tolerance the parity tests use.  This file is named so that pytest
collects it last; it needs no state from the other tests.
"""
import ctypes

import pytest
import torch

from shared_prompt_exact_dualkv_gb300 import synthetic
from tests.parity_util import check_grads

pytestmark = pytest.mark.gpu


def _inputs(w, seed):
    x = synthetic.make_inputs(w, seed)
    return [t.cuda() for t in (x.q, x.k, x.v, x.dout)]


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "deterministic"])
def test_static_workspace_matches_regular_backward(deterministic):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    w = synthetic.make_workload("noalloc", 4, 2, 128, 300, (200, 0, 131, 128))
    assert D.dualkv_bwd_workspace_bytes(w.P, w.R_lens, w.Hq, w.Hkv, w.d, deterministic) <= D.STATIC_SCRATCH_BYTES
    q, k, v, do = _inputs(w, seed=11)
    out, lse = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    ref = D.backward(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, deterministic=deterministic)
    torch.cuda.synchronize()
    for call in range(2):
        dq, dk, dv = torch.full_like(q, float("nan")), torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
        st = D.dualkv_bwd_static_workspace(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, deterministic, dq, dk, dv,
                                           check=False)
        assert st == D.DUALKV_OK, D.dualkv_status_string(st)
        est, site = D.dualkv_last_device_error()
        assert est == 0, (est, site)
        check_grads({"dq": (dq.float().cpu().numpy(), ref[0].float().cpu().numpy()),
                     "dk": (dk.float().cpu().numpy(), ref[1].float().cpu().numpy()),
                     "dv": (dv.float().cpu().numpy(), ref[2].float().cpu().numpy())}, f"static call {call}")
        if deterministic:
            for a, b in zip((dq, dk, dv), ref):
                assert torch.equal(a, b)


def test_static_workspace_rejects_oversize_shape():
    """A shape whose workspace exceeds the fixed scratch is refused before any launch."""
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    R = (ctypes.c_int32 * 1)(0)
    st = D.lib.dualkv_bwd_static_workspace(None, None, None, None, None, None, 65536, 1, R, 32, 8, 128, 0.088,
                                           0, 0, None, None, None, None)
    assert st == D.DUALKV_ERR_WORKSPACE


def test_static_workspace_limit_is_the_library_constant():
    """The Python constant STATIC_SCRATCH_BYTES is the library's own limit: a
    shape whose workspace is the largest at or below it is accepted, and the
    next larger shape (one more prompt row) is refused with
    DUALKV_ERR_WORKSPACE before any launch (null data pointers: nothing runs)."""
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    R = (ctypes.c_int32 * 1)(0)

    def need(P):
        return D.lib.dualkv_bwd_workspace_bytes(P, 1, R, 1, 1, 64, 0, 0)

    lo, hi = 1, 1 << 20                      # need(lo) <= limit < need(hi)
    assert need(lo) <= D.STATIC_SCRATCH_BYTES < need(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if need(mid) <= D.STATIC_SCRATCH_BYTES else (lo, mid)
    call = lambda P: D.lib.dualkv_bwd_static_workspace(None, None, None, None, None, None, P, 1, R, 1, 1, 64,
                                                       0.125, 0, 0, None, None, None, None)
    assert call(hi) == D.DUALKV_ERR_WORKSPACE
    assert call(lo) == D.DUALKV_ERR_INVALID_ARG   # accepted size; the null pointers are refused next
