"""GPU parity of the multi-group entry points (several prompts per packed
batch, each with its own responses): the CUDA path through the C ABI against
the fp64 group oracle, element by element, and against separate single-group
calls on each group's rows.  The last case holds more work items than one
launch carries, so it also covers the split into several launches."""
import numpy as np
import pytest
import torch

from oracle import attention as ora
from shared_prompt_exact_dualkv_gb300 import synthetic
from tests.parity_util import check_forward, check_grads

pytestmark = pytest.mark.gpu

CASES = [
    # name, Hq, Hkv, d, groups [(P_g, R_lens_g), ...]
    ("mixed_d128", 4, 2, 128, [(300, (200, 0, 131)), (0, (77, 150)), (129, ()), (50, (1, 128))]),
    ("mixed_d64", 2, 1, 64, [(256, (129, 1)), (5, (3,)), (0, (0,)), (140, (40, 260, 7))]),
    ("eight_aligned", 4, 1, 128, [(128, (128, 128))] * 8),
    # 16 groups + 1024 responses = 1040 segments, the per-call limit
    ("max_segments", 2, 1, 64, [(40 + g, tuple((g + i) % 5 for i in range(64))) for g in range(16)]),
]


def _lib():
    from shared_prompt_exact_dualkv_gb300 import dualkv
    return dualkv


def _inputs(case, seed=0):
    _, Hq, Hkv, d, groups = case
    x = synthetic.make_group_inputs(groups, Hq, Hkv, d, seed)
    return x, [t.cuda() for t in (x.q, x.k, x.v, x.dout)]


@pytest.fixture(scope="module")
def oracle_cache():
    return {}


def _oracle(case, x, cache):
    name, Hq, Hkv, d, groups = case
    if name not in cache:
        f64 = [synthetic.to_f64(t) for t in (x.q, x.k, x.v, x.dout)]
        scale = d ** -0.5
        out, lse = ora.dualkv_forward_groups(f64[0], f64[1], f64[2], groups, scale)
        dq, dk, dv = ora.dualkv_backward_groups(*f64, groups, scale)
        cache[name] = (out, lse, dq, dk, dv)
    return cache[name]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_groups_forward_parity(case, oracle_cache):
    D = _lib()
    x, (q, k, v, _) = _inputs(case)
    out, lse = D.forward_groups(q, k, v, case[4])
    st, site = D.dualkv_last_device_error()
    assert st == 0, (st, site)
    ref_out, ref_lse, *_ = _oracle(case, x, oracle_cache)
    check_forward(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, case[0])


@pytest.mark.parametrize("deterministic", [False, True], ids=["atomic", "deterministic"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_groups_backward_parity(case, deterministic, oracle_cache):
    D = _lib()
    x, (q, k, v, do) = _inputs(case)
    groups = case[4]
    out, lse = D.forward_groups(q, k, v, groups)
    _, _, rdq, rdk, rdv = _oracle(case, x, oracle_cache)
    for splits in (0, 3):
        dq, dk, dv = D.backward_groups(q, k, v, out, do, lse, groups, deterministic=deterministic,
                                       num_splits=splits)
        st, site = D.dualkv_last_device_error()
        assert st == 0, (st, site)
        check_grads({"dq": (dq.float().cpu().numpy(), rdq), "dk": (dk.float().cpu().numpy(), rdk),
                     "dv": (dv.float().cpu().numpy(), rdv)}, f"{case[0]} splits={splits}")


def _separate(D, q, k, v, do, groups, num_splits):
    """Each group through the single-group calls on its own rows."""
    outs, lses, dqs, dks, dvs = [], [], [], [], []
    a = 0
    for P_g, R_g in groups:
        b = a + P_g + sum(R_g)
        R = tuple(R_g) if len(R_g) else (0,)          # a prompt alone = one empty response
        sl = [t[a:b].contiguous() for t in (q, k, v, do)]
        o, l = D.forward(sl[0], sl[1], sl[2], P_g, R)
        g = D.backward(sl[0], sl[1], sl[2], o, sl[3], l, P_g, R, deterministic=True, num_splits=num_splits)
        outs.append(o)
        lses.append(l)
        dqs.append(g[0])
        dks.append(g[1])
        dvs.append(g[2])
        a = b
    return (torch.cat(outs), torch.cat(lses, dim=1), torch.cat(dqs), torch.cat(dks), torch.cat(dvs))


def _assert_same_as_separate(D, q, k, v, do, groups, num_splits):
    out, lse = D.forward_groups(q, k, v, groups)
    dq, dk, dv = D.backward_groups(q, k, v, out, do, lse, groups, deterministic=True, num_splits=num_splits)
    st, site = D.dualkv_last_device_error()
    assert st == 0, (st, site)
    s_out, s_lse, s_dq, s_dk, s_dv = _separate(D, q, k, v, do, groups, num_splits)
    st, site = D.dualkv_last_device_error()
    assert st == 0, (st, site)
    # every row's arithmetic is the same in both layouts, in the same order
    for name, a, b in (("out", out, s_out), ("lse", lse, s_lse), ("dq", dq, s_dq), ("dk", dk, s_dk),
                       ("dv", dv, s_dv)):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("case", CASES[:2], ids=[c[0] for c in CASES[:2]])
def test_groups_equal_separate_calls(case):
    D = _lib()
    _, (q, k, v, do) = _inputs(case, seed=7)
    _assert_same_as_separate(D, q, k, v, do, case[4], num_splits=1)


def test_long_work_list_is_split_across_launches():
    """8 groups of a 16K prompt and 16 responses of 4K rows: 5120 query tiles
    and more key items than one launch carries, so all three attention
    kernels run in two launches.  The result equals separate single-group
    calls (each of which fits in one launch)."""
    D = _lib()
    groups = [(16384, (4096,) * 16)] * 8
    x = synthetic.make_group_inputs(groups, 2, 1, 64, seed=9)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    D.dualkv_trace_enable(True)
    out, lse = D.forward_groups(q, k, v, groups)
    torch.cuda.synchronize()
    launches = {n: c for n, (_, c) in D.dualkv_trace_read().items()}
    D.dualkv_trace_enable(False)
    assert launches["fwd"] == 2
    _assert_same_as_separate(D, q, k, v, do, groups, num_splits=4)
