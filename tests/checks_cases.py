"""Runs the small parity cases through the library named by DUALKV_LIBRARY
(the checks build, in tests/test_gpu_checks.py) and prints one JSON line per
case: the device error word after the case and the parity errors against the
fp64 oracle.  Test helper; run as a child process so that the checks build is
the only copy of the library in it."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from oracle import attention as ora  # noqa: E402
from shared_prompt_exact_dualkv_gb300 import dualkv as D  # noqa: E402
from shared_prompt_exact_dualkv_gb300 import synthetic  # noqa: E402

CASES = [
    ("tiny", 2, 1, 64, 128, (64, 64, 64, 64)),
    ("ragged_d128", 4, 2, 128, 300, (200, 0, 131, 128, 77)),
    ("no_prompt", 4, 4, 128, 0, (129, 1, 256)),
    ("one_sequence", 2, 1, 64, 257, (300,)),
    ("group4_d64", 8, 2, 64, 384, (5, 250, 128)),
]


def rel(a, b):
    a = a.float().cpu().double().numpy() if torch.is_tensor(a) else a
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def main():
    assert D.lib.dualkv_checks_enabled() == 1, "not the checks build"
    for name, Hq, Hkv, d, P, R in CASES:
        w = synthetic.make_workload(name, Hq, Hkv, d, P, R)
        x = synthetic.make_inputs(w, seed=3)
        q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
        f64 = [synthetic.to_f64(t) for t in (x.q, x.k, x.v, x.dout)]
        ro, rl = ora.dualkv_forward(*f64[:3], w.P, w.R_lens, w.scale)
        rg = ora.dualkv_backward(*f64, w.P, w.R_lens, w.scale)
        out, lse = D.forward(q, k, v, w.P, w.R_lens, w.scale)
        res = {"case": name, "out": rel(out, ro), "lse": float(np.abs(lse.cpu().numpy() - rl).max())}
        for det, splits in ((0, 0), (1, 0), (1, 3), (2, 0)):
            g = D.backward(q, k, v, out, do, lse, w.P, w.R_lens, w.scale, deterministic=det, num_splits=splits)
            res[f"grads_det{int(det)}_s{splits}"] = max(rel(a, b) for a, b in zip(g, rg))
        st, site = D.dualkv_last_device_error()
        res.update(status=st, site=site)
        print(json.dumps(res), flush=True)

    # several prompt groups, one of them without a prompt and one without responses
    groups = [(200, (64, 130)), (0, (100,)), (129, ())]
    Hq, Hkv, d = 4, 2, 128
    x = synthetic.make_group_inputs(groups, Hq, Hkv, d, seed=5)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    f64 = [synthetic.to_f64(t) for t in (x.q, x.k, x.v, x.dout)]
    scale = d ** -0.5
    ro, rl = ora.dualkv_forward_groups(*f64[:3], groups, scale)
    rg = ora.dualkv_backward_groups(*f64, groups, scale)
    out, lse = D.forward_groups(q, k, v, groups, scale)
    g = D.backward_groups(q, k, v, out, do, lse, groups, scale, deterministic=False)
    st, site = D.dualkv_last_device_error()
    print(json.dumps({"case": "groups", "out": rel(out, ro), "lse": float(np.abs(lse.cpu().numpy() - rl).max()),
                      "grads": max(rel(a, b) for a, b in zip(g, rg)), "status": st, "site": site}), flush=True)

    # a rank's part of a sequence-sharded step: prompt query rows [128, 300)
    w = synthetic.make_workload("partial", 4, 2, 128, 300, (200, 0, 131))
    x = synthetic.make_inputs(w, seed=6)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    out, lse = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    ws = torch.empty(D.dualkv_bwd_workspace_bytes(w.P, w.R_lens, w.Hq, w.Hkv, w.d, False), dtype=torch.uint8,
                     device="cuda")
    dq, dk, dv = torch.zeros_like(q), torch.empty_like(k), torch.empty_like(v)
    f32 = [torch.zeros((w.P, h, w.d), device="cuda") for h in (w.Hq, w.Hkv, w.Hkv)]
    D.dualkv_fwd_partial(q, k, v, w.P, w.R_lens, (128, 300), out, lse, w.scale)
    D.dualkv_bwd_partial(q, k, v, out, do, lse, w.P, w.R_lens, (128, 300), w.scale, False, ws, dq, dk, dv, *f32)
    do64 = synthetic.to_f64(x.dout)
    do64[:128] = 0.0
    rq, rk, rv = ora.dualkv_backward(*[synthetic.to_f64(t) for t in (x.q, x.k, x.v)], do64, w.P, w.R_lens, w.scale)
    st, site = D.dualkv_last_device_error()
    print(json.dumps({"case": "partial", "dq": rel(dq[128:], rq[128:]), "dk": rel(dk, rk), "dv": rel(dv, rv),
                      "dk_prompt_f32": rel(f32[1], rk[:w.P]), "status": st, "site": site}), flush=True)

    # a prompt whose keys and values exceed half of L2: the forward and dQ
    # blocks take the heads as their outer index; kv-head 0 against the
    # kv-group oracle (torch fp64)
    from oracle import kvgroup as okg
    w = synthetic.make_workload("head_outer", 8, 8, 128, 20000, (129, 300))
    assert w.P * w.Hkv * w.d * 4 > torch.cuda.get_device_properties(0).L2_cache_size // 2
    x = synthetic.make_inputs(w, seed=7)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    out, lse = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    g = D.backward(q, k, v, out, do, lse, w.P, w.R_lens, w.scale)
    st, site = D.dualkv_last_device_error()
    f64 = lambda t: t.to(torch.float64).contiguous()
    ref = okg.kvgroup_forward_backward(f64(x.q[:, 0:1]), f64(x.k[:, 0]), f64(x.v[:, 0]), f64(x.dout[:, 0:1]),
                                       w.P, w.R_lens, w.scale)
    print(json.dumps({"case": "head_outer", "out": rel(out[:, 0:1], ref["out"].numpy()),
                      "lse": float(np.abs(lse[0:1].cpu().numpy() - ref["lse"].numpy()).max()),
                      "dq": rel(g[0][:, 0:1], ref["dq"].numpy()), "dk": rel(g[1][:, 0], ref["dk"].numpy()),
                      "dv": rel(g[2][:, 0], ref["dv"].numpy()), "status": st, "site": site}), flush=True)

    # the layer's GEMM in all three forms, on the 128-row tile path and the
    # 256-row one (19000 x 2056 has 675 tiles of 256 x 256), against fp64 products
    g = torch.Generator("cpu").manual_seed(8)
    worst = 0.0
    for M, N, K in ((296, 264, 200), (19000, 2056, 200)):   # every row length a multiple of 8
        for kind in (0, 1, 2):
            shapes = {0: ((M, K), (N, K)), 1: ((M, K), (K, N)), 2: ((K, M), (K, N))}[kind]
            A = torch.randn(shapes[0], generator=g).to(torch.bfloat16)
            B = torch.randn(shapes[1], generator=g).to(torch.bfloat16)
            ref = {0: lambda: A.double() @ B.double().T, 1: lambda: A.double() @ B.double(),
                   2: lambda: A.double().T @ B.double()}[kind]()
            Y = torch.full((M, N), float("nan"), dtype=torch.float32 if kind == 2 else torch.bfloat16, device="cuda")
            D.dualkv_gemm(kind, A.cuda(), B.cuda(), Y)
            worst = max(worst, rel(Y, ref.numpy()))
    st, site = D.dualkv_last_device_error()
    print(json.dumps({"case": "gemm", "gemm": worst, "status": st, "site": site}), flush=True)


if __name__ == "__main__":
    main()
