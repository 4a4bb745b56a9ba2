"""GPU checks of the packed decoder layer (include/dualkv_layer.h).

* Parity: the layer through the C ABI against the fp64 layer oracle (which
  runs every replicated sequence and scatters to the packed rows), on the
  same seeded bf16 inputs, element by element over y, dx and every weight
  gradient.
* Packed versus replicated through the same library: the packed layer's rows
  equal the replicated layer's rows (prompt rows of any replica), its dx on a
  prompt row equals the sum over the replicas, and its weight gradients equal
  the replicated ones.

Tolerances: every intermediate (h1, q, k, v, a, x2, h2, gate/up, m) is stored
in bf16 (unit roundoff 2^-8, RMS rounding error about 2^-9/sqrt(3) = 0.11%).
Along the longest chain about ten such roundings add up independently,
which gives about 0.4% RMS in the outputs.  The bounds below leave a factor
2.5-5 for the fp32 sums and GEMM blocking."""
import numpy as np
import pytest
import torch

from oracle import layer as L
from shared_prompt_exact_dualkv_gb300 import synthetic
from tests.parity_util import rel_l2

pytestmark = pytest.mark.gpu

Y_REL_L2 = 1e-2
DX_REL_L2 = 1e-2
GRAD_REL_L2 = 2e-2

GROUPS = [(130, (70, 0, 129)), (0, (50,)), (40, ())]


def _lib():
    from shared_prompt_exact_dualkv_gb300 import dualkv
    return dualkv


def _setup(shape_name, groups, seed):
    D = _lib()
    shape = synthetic.LAYER_SHAPES[shape_name]
    T = synthetic.group_rows(groups)
    w, x, dy = synthetic.make_layer_inputs(shape, T, seed)
    cfg = D.layer_config(**shape)
    wd = {n: t.cuda() for n, t in w.items()}
    return D, shape, cfg, w, wd, x, dy


@pytest.mark.parametrize("shape_name", ["small", "small_d128", "wide"])
def test_layer_parity_against_oracle(shape_name):
    D, shape, cfg, w, wd, x, dy = _setup(shape_name, GROUPS, 0)
    layer = D.PackedLayer(cfg, wd, GROUPS)
    xg, dyg = x.cuda(), dy.cuda()
    y = layer.forward(xg)
    dx, grads = layer.backward(xg, dyg)
    st, site = D.dualkv_last_device_error()
    assert st == 0, (st, site)
    c = L.LayerConfig(**shape)
    W64 = {n: synthetic.to_f64(t) for n, t in w.items()}
    x64, dy64 = synthetic.to_f64(x), synthetic.to_f64(dy)
    ry = L.packed_forward(x64, GROUPS, W64, c)
    rdx, rgrads = L.packed_backward(x64, dy64, GROUPS, W64, c)
    errs = {"y": rel_l2(y.float().cpu().numpy(), ry), "dx": rel_l2(dx.float().cpu().numpy(), rdx)}
    for n in L.WEIGHT_NAMES:
        errs[n] = rel_l2(grads[n].cpu().numpy(), rgrads[n])
    assert errs["y"] <= Y_REL_L2, errs
    assert errs["dx"] <= DX_REL_L2, errs
    for n in L.WEIGHT_NAMES:
        assert errs[n] <= GRAD_REL_L2, (n, errs)


def _replicate(groups, x, dy):
    """Rows of the replicated layout, the replicated dy (prompt rows' dy to
    each group's first sequence) and the bookkeeping to map back."""
    xs, dys, seqs = [], [], []
    a = 0
    for P, R in groups:
        off = a + P
        lens = list(R) if len(R) else [0]
        for i, r in enumerate(lens):
            idx = list(range(a, a + P)) + list(range(off, off + r))
            xs.append(x[idx])
            d = dy[idx].clone()
            if i > 0:
                d[:P] = 0
            dys.append(d)
            seqs.append((a, P, off, r))
            off += r
        a = off
    rep_groups = [(len(t), ()) for t in xs]
    return torch.cat(xs), torch.cat(dys), rep_groups, seqs


def test_packed_layer_equals_replicated_layer():
    groups = [(300, (200, 0, 131, 128)), (64, (257,))]
    D, shape, cfg, w, wd, x, dy = _setup("small", groups, 3)
    xg, dyg = x.cuda(), dy.cuda()
    packed = D.PackedLayer(cfg, wd, groups)
    y = packed.forward(xg)
    dx, grads = packed.backward(xg, dyg)
    xr, dyr, rep_groups, seqs = _replicate(groups, xg, dyg)
    rep = D.PackedLayer(cfg, wd, rep_groups)
    yr = rep.forward(xr)
    dxr, grads_r = rep.backward(xr, dyr)
    st, site = D.dualkv_last_device_error()
    assert st == 0, (st, site)
    # scatter the replicated results back to packed rows
    y_from_rep = torch.zeros_like(y, dtype=torch.float32)
    dx_from_rep = torch.zeros_like(dx, dtype=torch.float32)
    row = 0
    first = set()
    for a, P, off, r in seqs:
        yi, dxi = yr[row:row + P + r].float(), dxr[row:row + P + r].float()
        y_from_rep[off:off + r] = yi[P:]
        dx_from_rep[off:off + r] = dxi[P:]
        if a not in first:
            y_from_rep[a:a + P] = yi[:P]
            first.add(a)
        dx_from_rep[a:a + P] += dxi[:P]
        row += P + r
    assert rel_l2(y.float().cpu().numpy(), y_from_rep.cpu().numpy()) <= Y_REL_L2
    assert rel_l2(dx.float().cpu().numpy(), dx_from_rep.cpu().numpy()) <= DX_REL_L2
    for n in D.LAYER_WEIGHTS:
        assert rel_l2(grads[n].cpu().numpy(), grads_r[n].cpu().numpy()) <= GRAD_REL_L2, n
