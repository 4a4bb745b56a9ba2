"""Sequence-sharded backward (shared_prompt_exact_dualkv_gb300/sharded.py).

CPU tests run 2 gloo ranks with the fp64 oracle standing in for the
kernels.  They check the response split, the local packing and the
all-reduce of the prompt rows against the unsharded oracle.  The GPU test
runs 2 processes on one GPU with the real library; the exchange is a gloo
all-reduce staged through the host, so no kernel of one rank waits on the
other.  It compares the assembled result with the fp64 oracle and with an
unsharded run."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import attention as ora
from shared_prompt_exact_dualkv_gb300 import sharded, synthetic
from tests.parity_util import check_grads

SHARES = (0.25, 0.75)   # each rank's share of the prompt rows' dO


def test_shard_bounds_cover_every_response_once():
    for N in (1, 2, 5, 16, 17):
        for world in (1, 2, 3, 8):
            spans = [sharded.shard_bounds(N, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == N
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        sharded.shard_bounds(4, 2, 2)


def test_local_rows():
    idx = sharded.local_rows(3, [2, 1, 4], 1, 3)
    assert idx.tolist() == [0, 1, 2, 5, 6, 7, 8, 9]


def _oracle_fwd(q, k, v, P, R, scale):
    o, l = ora.dualkv_forward(q.numpy(), k.numpy(), v.numpy(), P, R, scale)
    return torch.from_numpy(o), torch.from_numpy(l)


def _oracle_bwd(q, k, v, out, dout, lse, P, R, scale):
    g = ora.dualkv_backward(q.numpy(), k.numpy(), v.numpy(), dout.numpy(), P, R, scale)
    return tuple(torch.from_numpy(x) for x in g)


def _case():
    P, R = 37, [5, 0, 19, 1, 40]
    w = synthetic.make_workload("shard", 4, 2, 8, P, R)
    x = synthetic.make_inputs(w, seed=4)
    return w, [synthetic.to_f64(t) for t in (x.q, x.k, x.v, x.dout)]


def _cpu_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, (Q, K, V, DO) = _case()
    lo, hi = sharded.shard_bounds(w.N, world, rank)
    idx = sharded.local_rows(w.P, w.R_lens, lo, hi).numpy()
    t = [torch.from_numpy(a[idx].copy()) for a in (Q, K, V, DO)]
    t[3][:w.P] *= SHARES[rank]
    R_local = list(w.R_lens[lo:hi])
    out, lse = sharded.sharded_forward(t[0], t[1], t[2], w.P, R_local, w.scale, fwd_fn=_oracle_fwd)
    dq, dk, dv = sharded.sharded_backward(t[0], t[1], t[2], out, t[3], lse, w.P, R_local, w.scale,
                                          bwd_fn=_oracle_bwd)
    q.put((rank, idx, out.numpy(), lse.numpy(), dq.numpy(), dk.numpy(), dv.numpy()))
    dist.destroy_process_group()


def _run_ranks(target, world, timeout=300):
    port = 29600 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=target, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=timeout) for _ in range(world)]
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    return sorted(res, key=lambda r: r[0])


def _assemble(res, T, Hq, Hkv, d, P):
    out = np.zeros((T, Hq, d)); lse = np.zeros((Hq, T))
    dq = np.zeros((T, Hq, d)); dk = np.zeros((T, Hkv, d)); dv = np.zeros((T, Hkv, d))
    for rank, idx, o, l, a, b, c in res:
        out[idx] = o; lse[:, idx] = l; dq[idx] = a; dk[idx] = b; dv[idx] = c
        # every rank holds the same prompt rows after the exchange
        np.testing.assert_array_equal(a[:P], res[0][4][:P])
        np.testing.assert_array_equal(b[:P], res[0][5][:P])
    return out, lse, dq, dk, dv


def test_two_cpu_ranks_match_unsharded_oracle():
    w, (Q, K, V, DO) = _case()
    res = _run_ranks(_cpu_rank, 2)
    out, lse, dq, dk, dv = _assemble(res, w.T, w.Hq, w.Hkv, w.d, w.P)
    ro, rl = ora.dualkv_forward(Q, K, V, w.P, w.R_lens, w.scale)
    rdq, rdk, rdv = ora.dualkv_backward(Q, K, V, DO, w.P, w.R_lens, w.scale)
    np.testing.assert_allclose(out, ro, atol=1e-12)
    np.testing.assert_allclose(lse, rl, atol=1e-12)
    # the exchange runs in fp32
    for a, b in ((dq, rdq), (dk, rdk), (dv, rdv)):
        np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-5)


def _gpu_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synthetic.make_workload("shard_gpu", 4, 2, 128, 300, (200, 0, 131, 128, 77))
    x = synthetic.make_inputs(w, seed=6)
    lo, hi = sharded.shard_bounds(w.N, world, rank)
    idx = sharded.local_rows(w.P, w.R_lens, lo, hi)
    t = [a[idx].contiguous().cuda() for a in (x.q, x.k, x.v, x.dout)]
    t[3][:w.P] = (t[3][:w.P].float() * SHARES[rank]).to(torch.bfloat16)
    R_local = list(w.R_lens[lo:hi])
    out, lse = sharded.sharded_forward(t[0], t[1], t[2], w.P, R_local, w.scale)
    dq, dk, dv = sharded.sharded_backward(t[0], t[1], t[2], out, t[3], lse, w.P, R_local, w.scale)
    torch.cuda.synchronize()
    q.put((rank, idx.numpy(), out.float().cpu().numpy(), lse.cpu().numpy(), dq.float().cpu().numpy(),
           dk.float().cpu().numpy(), dv.float().cpu().numpy()))
    dist.destroy_process_group()


@pytest.mark.gpu
def test_two_gpu_processes_match_oracle_and_unsharded_run():
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    w = synthetic.make_workload("shard_gpu", 4, 2, 128, 300, (200, 0, 131, 128, 77))
    x = synthetic.make_inputs(w, seed=6)
    res = _run_ranks(_gpu_rank, 2)
    out, lse, dq, dk, dv = _assemble(res, w.T, w.Hq, w.Hkv, w.d, w.P)
    # the dO each rank saw, summed: the prompt shares add up to the packed dO
    full_do = x.dout.clone()
    full_do[:w.P] = sum((x.dout[:w.P].float() * s).to(torch.bfloat16).float() for s in SHARES).to(torch.bfloat16)
    f64 = [synthetic.to_f64(t) for t in (x.q, x.k, x.v)]
    rdq, rdk, rdv = ora.dualkv_backward(*f64, synthetic.to_f64(full_do), w.P, w.R_lens, w.scale)
    check_grads({"dq": (dq, rdq), "dk": (dk, rdk), "dv": (dv, rdv)}, "sharded")
    # response rows and the forward are the unsharded run's, bit for bit
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, full_do))
    uo, ul = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    udq, udk, udv = D.backward(q, k, v, uo, do, ul, w.P, w.R_lens, w.scale)
    np.testing.assert_array_equal(out, uo.float().cpu().numpy())
    np.testing.assert_array_equal(lse, ul.cpu().numpy())
    for a, b in ((dq, udq), (dk, udk), (dv, udv)):
        np.testing.assert_array_equal(a[w.P:], b.float().cpu().numpy()[w.P:])
