"""Full-size parity: the five large workloads, run through the C ABI exactly
as bench.py runs them (all heads, both dK/dV modes), checked against the fp64
oracle on sampled outputs it can compute one at a time, plus identities that
hold at any size.

* O, LSE and dQ of sampled query rows (prompt start/end, 128-row tile
  boundaries, first/last rows of several responses) of two q-heads in
  different kv groups: the oracle's row-wise function.
* dK and dV of sampled key rows of kv-head 0 -- prompt keys in the last two
  prompt tiles (seen by every response) and response keys -- summed over the
  group's q-heads and every query row that sees them.
* sum_k dV[k] = sum over the group's rows of dO and sum_k dK[k] = 0 per
  kv-head (each softmax row sums to 1, each dS row to 0), over all rows.
"""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

from oracle import attention as ora
from shared_prompt_exact_dualkv_gb300 import synthetic
from tests.parity_util import GRAD_REL_L2, LSE_MAX_ABS, OUT_MAX_ABS, OUT_REL_L2, max_abs, rel_l2

pytestmark = pytest.mark.gpu

NAMES = ["qwen3_8b", "p32k", "ragged_30b_a3b", "edge_p64k", "edge_n4"]


def sample_rows(w):
    rows = set()
    P, off = w.P, w.offsets
    for r in (0, 1, 127, 128, P // 2, P - 129, P - 1):
        if 0 <= r < P:
            rows.add(r)
    for i in sorted({0, w.N // 2, w.N - 1}):
        for r in (off[i], off[i] + 1, off[i] + 127, off[i] + 128, off[i + 1] - 1):
            if off[i] <= r < off[i + 1]:
                rows.add(r)
    return sorted(rows)


def sample_keys(w):
    keys = set()
    P, off = w.P, w.offsets
    for r in (P - 1, P - 128, P - 129, P - 200):
        if 0 <= r < P:
            keys.add(r)
    for i in sorted({0, w.N - 1}):
        for r in (off[i], off[i] + 129, off[i + 1] - 1):
            if off[i] <= r < off[i + 1]:
                keys.add(r)
    return sorted(keys)


def oracle_keys(q64, k64, v64, do64, w, keys):
    """dK/dV of `keys` for kv-head 0; one q-head per thread, summed in head order."""
    g = w.Hq // w.Hkv

    def one(h):
        return ora.keys_dkdv(q64[:, h:h + 1], k64, v64, do64[:, h:h + 1], w.P, w.R_lens, w.scale, 0, keys,
                             row_block=256)

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(g, os.cpu_count() or 1)) as ex:
        parts = list(ex.map(one, range(g)))
    return sum(p[0] for p in parts), sum(p[1] for p in parts)


@pytest.mark.parametrize("name", NAMES)
def test_fullsize_sampled_parity(name):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    w = synthetic.WORKLOADS[name]
    x = synthetic.make_inputs(w, seed=0)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    out, lse = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    grads = {det: D.backward(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, deterministic=det)
             for det in (False, True)}
    st, site = D.dualkv_last_device_error()
    assert st == 0, (st, site)

    g = w.Hq // w.Hkv
    rows = sample_rows(w)
    heads = [0, w.Hq - 1]
    q64 = synthetic.to_f64(x.q[:, heads])
    do64 = synthetic.to_f64(x.dout[:, heads])
    kv_heads = [0, w.Hkv - 1]
    k64 = synthetic.to_f64(x.k[:, kv_heads])
    v64 = synthetic.to_f64(x.v[:, kv_heads])
    # sliced arrays: q-head heads[a] reads kv-head kv_heads[a] (1:1 in the slice)
    ref = ora.rows_forward_backward(q64, k64, v64, do64, w.P, w.R_lens, w.scale, [0, 1], rows)
    got_o = out[rows][:, heads].float().cpu().numpy().transpose(1, 0, 2)
    got_l = lse[heads][:, rows].cpu().numpy()
    assert max_abs(got_o, ref["o"]) <= OUT_MAX_ABS
    assert rel_l2(got_o, ref["o"]) <= OUT_REL_L2
    assert max_abs(got_l, ref["lse"]) <= LSE_MAX_ABS
    for det, (dq, dk, dv) in grads.items():
        got_dq = dq[rows][:, heads].float().cpu().numpy().transpose(1, 0, 2)
        assert rel_l2(got_dq, ref["dq"]) <= GRAD_REL_L2, (det, rel_l2(got_dq, ref["dq"]))

    keys = sample_keys(w)
    qg = synthetic.to_f64(x.q[:, 0:g])
    dog = synthetic.to_f64(x.dout[:, 0:g])
    kk = synthetic.to_f64(x.k[:, 0:1])
    vv = synthetic.to_f64(x.v[:, 0:1])
    rdk, rdv = oracle_keys(qg, kk, vv, dog, w, keys)
    for det, (dq, dk, dv) in grads.items():
        gdk = dk[keys, 0].float().cpu().numpy()
        gdv = dv[keys, 0].float().cpu().numpy()
        assert rel_l2(gdk, rdk) <= GRAD_REL_L2, (det, "dk", rel_l2(gdk, rdk))
        assert rel_l2(gdv, rdv) <= GRAD_REL_L2, (det, "dv", rel_l2(gdv, rdv))

        # identities over all rows, per kv-head
        sdv = dv.float().sum(0).double().cpu().numpy()                                   # [Hkv, d]
        sdo = do.float().view(w.T, w.Hkv, g, w.d).sum((0, 2)).double().cpu().numpy()    # [Hkv, d]
        assert rel_l2(sdv, sdo) <= GRAD_REL_L2, (det, "sum dV", rel_l2(sdv, sdo))
        sdk = dk.float().sum(0).double().cpu().numpy()
        scale_dk = dk.float().abs().sum(0).double().cpu().numpy()
        assert np.all(np.abs(sdk) <= 1e-2 * scale_dk + 1e-3), (det, "sum dK")
    if name == "p32k":
        # both modes agree closely (they differ only in the order of fp32 sums)
        a, b = grads[False], grads[True]
        assert torch.equal(a[0], b[0])
        for x_, y_ in zip(a[1:], b[1:]):
            assert rel_l2(x_.float().cpu().numpy(), y_.float().cpu().numpy()) <= 1e-3
