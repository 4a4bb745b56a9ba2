"""Full-size parity: the five large workloads, run through the C ABI exactly
as bench.py runs them (all heads, the library's split choice, both dK/dV
modes), compared element by element with the fp64 oracle.

Heads are independent, so the oracle runs on whole kv-head groups (the
q-heads that read one kv-head) and the comparison is exact for those heads:

* every workload: every row of O, LSE and dQ of the q-heads of kv-head 0, and
  every row of that kv-head's dK and dV;
* Qwen3-8B, ragged 30B-A3B and edge case (b): the same for the last kv-head;
* P32K and edge case (a) P64K, last kv-head: complete 128-row query tiles
  (O, LSE, dQ) -- the first, middle and last prompt tile and the first and
  last tile of responses 0, N/2 and N-1.

Tolerances are the ones the parity tests use everywhere (out max-abs <= 1e-2
and rel-L2 <= 5e-3; LSE max-abs <= 1e-3; dQ, dK, dV rel-L2 <= 1e-2), taken
over the whole compared set.  Two identities over all heads and rows close
the gap to the heads the oracle does not run: sum_k dV[k] equals the sum of
dO over the group's rows, and sum_k dK[k] = 0 per kv-head (each softmax row
sums to one, each dS row to zero).
"""
import os

import numpy as np
import pytest
import torch

from oracle import kvgroup as okg
from shared_prompt_exact_dualkv_gb300 import synthetic
from tests.parity_util import GRAD_REL_L2, LSE_MAX_ABS, OUT_MAX_ABS, OUT_REL_L2, max_abs, rel_l2

pytestmark = pytest.mark.gpu

# workload -> kv-heads compared over all rows; kv-heads compared on complete tiles
PLAN = {
    "qwen3_8b": ("first_last", ()),
    "ragged_30b_a3b": ("first_last", ()),
    "edge_n4": ("first_last", ()),
    "p32k": ("first", ("last",)),
    "edge_p64k": ("first", ("last",)),
}


def _kv_heads(w, which):
    return {"first": [0], "last": [w.Hkv - 1], "first_last": sorted({0, w.Hkv - 1})}[which]


def _group_inputs(x, w, kvh):
    g = w.Hq // w.Hkv
    hs = slice(kvh * g, (kvh + 1) * g)
    f64 = lambda t: t.to(torch.float64).contiguous()  # exact upcast of bf16
    return f64(x.q[:, hs]), f64(x.k[:, kvh]), f64(x.v[:, kvh]), f64(x.dout[:, hs])


def _cpu(t):
    return t.float().cpu().double().numpy()


def _query_tiles(w):
    """Complete 128-row tiles: first, middle and last prompt tile; first and
    last tile of responses 0, N/2 and N-1 (the last one possibly ragged)."""
    tiles = []
    nP = (w.P + 127) // 128
    for t in sorted({0, nP // 2, nP - 1}):
        tiles.append((t * 128, min(t * 128 + 128, w.P)))
    off = w.offsets
    for i in sorted({0, w.N // 2, w.N - 1}):
        n = (w.R_lens[i] + 127) // 128
        for t in sorted({0, n - 1}):
            tiles.append((off[i] + t * 128, min(off[i] + t * 128 + 128, off[i + 1])))
    return tiles


def _check(name, got, ref, kind):
    if kind == "out":
        assert max_abs(got, ref) <= OUT_MAX_ABS, (name, "max-abs", max_abs(got, ref))
        assert rel_l2(got, ref) <= OUT_REL_L2, (name, "rel-L2", rel_l2(got, ref))
    elif kind == "lse":
        assert max_abs(got, ref) <= LSE_MAX_ABS, (name, "max-abs", max_abs(got, ref))
    else:
        assert np.isfinite(got).all(), name
        assert rel_l2(got, ref) <= GRAD_REL_L2, (name, "rel-L2", rel_l2(got, ref))


@pytest.mark.parametrize("name", list(PLAN))
def test_fullsize_parity(name):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    torch.set_num_threads(os.cpu_count() or 1)
    w = synthetic.WORKLOADS[name]
    g = w.Hq // w.Hkv
    x = synthetic.make_inputs(w, seed=0)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    out, lse = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    grads = {det: D.backward(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, deterministic=det)
             for det in (False, True)}
    st, site = D.dualkv_last_device_error()
    assert st == 0, (st, site)

    full, tiled = PLAN[name]
    for kvh in _kv_heads(w, full):
        hs = slice(kvh * g, (kvh + 1) * g)
        ref = okg.kvgroup_forward_backward(*_group_inputs(x, w, kvh), w.P, w.R_lens, w.scale)
        tag = f"{name} kv-head {kvh}"
        _check(tag + " out", _cpu(out[:, hs]), ref["out"].numpy(), "out")
        _check(tag + " lse", lse[hs].cpu().double().numpy(), ref["lse"].numpy(), "lse")
        for det, (dq, dk, dv) in grads.items():
            _check(f"{tag} det={det} dq", _cpu(dq[:, hs]), ref["dq"].numpy(), "grad")
            _check(f"{tag} det={det} dk", _cpu(dk[:, kvh]), ref["dk"].numpy(), "grad")
            _check(f"{tag} det={det} dv", _cpu(dv[:, kvh]), ref["dv"].numpy(), "grad")
        del ref

    for which in tiled:
        for kvh in _kv_heads(w, which):
            hs = slice(kvh * g, (kvh + 1) * g)
            tiles = _query_tiles(w)
            ref = okg.kvgroup_rows(*_group_inputs(x, w, kvh), w.P, w.R_lens, w.scale, tiles)
            tag = f"{name} kv-head {kvh} tiles"
            cat = lambda key: np.concatenate([ref[t][key].numpy() for t in tiles], axis=1)
            rows = torch.as_tensor(np.concatenate([np.arange(a, b) for a, b in tiles]), device="cuda")
            _check(tag + " out", _cpu(out[rows][:, hs]).transpose(1, 0, 2), cat("out"), "out")
            _check(tag + " lse", lse[hs][:, rows].cpu().double().numpy(), cat("lse"), "lse")
            for det, (dq, _, _) in grads.items():
                _check(f"{tag} det={det} dq", _cpu(dq[rows][:, hs]).transpose(1, 0, 2), cat("dq"), "grad")

    for det, (dq, dk, dv) in grads.items():
        # identities over all rows, per kv-head
        sdv = dv.float().sum(0).double().cpu().numpy()                                   # [Hkv, d]
        sdo = do.float().view(w.T, w.Hkv, g, w.d).sum((0, 2)).double().cpu().numpy()    # [Hkv, d]
        assert rel_l2(sdv, sdo) <= GRAD_REL_L2, (det, "sum dV", rel_l2(sdv, sdo))
        sdk = dk.float().sum(0).double().cpu().numpy()
        scale_dk = dk.float().abs().sum(0).double().cpu().numpy()
        assert np.all(np.abs(sdk) <= 1e-2 * scale_dk + 1e-3), (det, "sum dK")
    # both modes agree closely (they differ only in the order of fp32 sums,
    # then one bf16 rounding)
    for x_, y_ in zip(grads[False], grads[True]):
        diff = float(torch.linalg.vector_norm(x_.float() - y_.float()) / torch.linalg.vector_norm(y_.float()))
        assert diff <= 3e-3, diff


def test_head_outer_block_order_parity():
    """The forward and dQ kernels take the heads as the outer block index when
    the prompt's keys and values of all kv-heads exceed half of L2 (P32K and
    P64K do).  Here with a ragged prompt tail, a ragged last response and an
    empty one: every row of the first and last kv-head groups against the
    oracle, both dK/dV modes."""
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    torch.set_num_threads(os.cpu_count() or 1)
    w = synthetic.make_workload("head_outer", 16, 8, 128, 24001, (300, 1000, 0, 129))
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    assert w.P * w.Hkv * w.d * 4 > l2 // 2, "the case must take the head-outer order"
    g = w.Hq // w.Hkv
    x = synthetic.make_inputs(w, seed=3)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    out, lse = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    grads = {det: D.backward(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, deterministic=det)
             for det in (False, True)}
    st, site = D.dualkv_last_device_error()
    assert st == 0, (st, site)
    for kvh in (0, w.Hkv - 1):
        hs = slice(kvh * g, (kvh + 1) * g)
        ref = okg.kvgroup_forward_backward(*_group_inputs(x, w, kvh), w.P, w.R_lens, w.scale)
        tag = f"head-outer kv-head {kvh}"
        _check(tag + " out", _cpu(out[:, hs]), ref["out"].numpy(), "out")
        _check(tag + " lse", lse[hs].cpu().double().numpy(), ref["lse"].numpy(), "lse")
        for det, (dq, dk, dv) in grads.items():
            _check(f"{tag} det={det} dq", _cpu(dq[:, hs]), ref["dq"].numpy(), "grad")
            _check(f"{tag} det={det} dk", _cpu(dk[:, kvh]), ref["dk"].numpy(), "grad")
            _check(f"{tag} det={det} dv", _cpu(dv[:, kvh]), ref["dv"].numpy(), "grad")
