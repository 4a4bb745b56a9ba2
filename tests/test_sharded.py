"""Sharded DualKV attention (shared_prompt_exact_dualkv_gb300/sharded.py) and
the partial entry points it runs on (dualkv_fwd_partial / dualkv_bwd_partial).

CPU tests run 2 gloo ranks with the fp64 oracle standing in for the kernels.
They check the splits, the local packing and the exchanges against the
unsharded oracle, for the sequence split (prompt rows divided, or repeated on
every rank) and for the kv-head split.  GPU tests run 2 processes on one GPU
with the real library; every exchange is a gloo collective staged through the
host, so no kernel of one rank waits on the other.  They compare the
assembled result with the fp64 oracle and with an unsharded run.  Single-GPU
tests hold the partial entry points to the regular ones and to the oracle."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import attention as ora
from shared_prompt_exact_dualkv_gb300 import sharded, synthetic
from tests.parity_util import check_forward, check_grads

SHARES = (0.25, 0.75)   # each rank's share of the prompt rows' dO


# --------------------------------------------------------------------------- host logic

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


@pytest.mark.parametrize("P", [0, 1, 127, 128, 300, 4096, 32768, 32769])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_prompt_bounds_tile_and_balance(P, world):
    spans = [sharded.prompt_bounds(P, world, r) for r in range(world)]
    assert spans[0][0] == 0 and spans[-1][1] == P
    assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    for lo, hi in spans:
        assert (lo % 128 == 0 or lo == P) and (hi % 128 == 0 or hi == P) and lo <= hi
    n = (P + 127) // 128
    if n >= 8 * world:   # causal work (tile t walks t + 1 key tiles) within one tile's worth of even
        work = [sum(t + 1 for t in range(lo // 128, (hi + 127) // 128)) for lo, hi in spans]
        assert max(work) - min(work) <= 2 * n


def test_local_rows():
    idx = sharded.local_rows(3, [2, 1, 4], 1, 3)
    assert idx.tolist() == [0, 1, 2, 5, 6, 7, 8, 9]


# --------------------------------------------------------------------------- oracle stand-ins

def _oracle_fwd(q, k, v, P, R, scale, prompt_rows):
    """The partial forward's contract on the oracle: prompt rows outside
    [lo, hi) are not written (zero here)."""
    lo, hi = prompt_rows
    o, l = ora.dualkv_forward(q.numpy(), k.numpy(), v.numpy(), P, R, scale)
    o[:lo] = o[hi:P] = 0.0
    l[:, :lo] = l[:, hi:P] = 0.0
    return torch.from_numpy(o), torch.from_numpy(l)


def _oracle_bwd(q, k, v, out, dout, lse, P, R, scale, prompt_rows, deterministic=False):
    """The partial backward's contract on the oracle: prompt rows outside
    [lo, hi) act as rows with zero dO, their dQ is not written; the prompt
    rows' gradients are also returned unrounded."""
    lo, hi = prompt_rows
    do = dout.numpy().copy()
    do[:lo] = do[hi:P] = 0.0
    dq, dk, dv = ora.dualkv_backward(q.numpy(), k.numpy(), v.numpy(), do, P, R, scale)
    dq[:lo] = dq[hi:P] = 0.0
    t = [torch.from_numpy(x) for x in (dq, dk, dv)]
    return t[0], t[1], t[2], t[0][:P].clone(), t[1][:P].clone(), t[2][:P].clone()


def _case():
    P, R = 300, [5, 0, 19, 1, 40]
    w = synthetic.make_workload("shard", 4, 2, 8, P, R)
    x = synthetic.make_inputs(w, seed=4)
    return w, [synthetic.to_f64(t) for t in (x.q, x.k, x.v, x.dout)]


def _run_ranks(target, world, extra=(), timeout=300):
    port = 29600 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + tuple(extra)) for r in range(world)]
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
        # every rank holds the same prompt rows after the exchanges
        np.testing.assert_array_equal(o[:P], res[0][2][:P])
        np.testing.assert_array_equal(a[:P], res[0][4][:P])
        np.testing.assert_array_equal(b[:P], res[0][5][:P])
    return out, lse, dq, dk, dv


# --------------------------------------------------------------------------- sequence split on CPU ranks

def _cpu_rank(rank, world, port, q, divide):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, (Q, K, V, DO) = _case()
    lo, hi = sharded.shard_bounds(w.N, world, rank)
    idx = sharded.local_rows(w.P, w.R_lens, lo, hi).numpy()
    t = [torch.from_numpy(a[idx].copy()) for a in (Q, K, V, DO)]
    t[3][:w.P] *= SHARES[rank]
    R_local = list(w.R_lens[lo:hi])
    rows = sharded.prompt_bounds(w.P, world, rank) if divide else None
    out, lse = sharded.sharded_forward(t[0], t[1], t[2], w.P, R_local, w.scale, prompt_rows=rows, fwd_fn=_oracle_fwd)
    dq, dk, dv = sharded.sharded_backward(t[0], t[1], t[2], out, t[3], lse, w.P, R_local, w.scale, prompt_rows=rows,
                                          bwd_fn=_oracle_bwd)
    q.put((rank, idx, out.numpy(), lse.numpy(), dq.numpy(), dk.numpy(), dv.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("divide", [True, False], ids=["prompt_divided", "prompt_on_every_rank"])
def test_two_cpu_ranks_match_unsharded_oracle(divide):
    w, (Q, K, V, DO) = _case()
    res = _run_ranks(_cpu_rank, 2, (divide,))
    out, lse, dq, dk, dv = _assemble(res, w.T, w.Hq, w.Hkv, w.d, w.P)
    ro, rl = ora.dualkv_forward(Q, K, V, w.P, w.R_lens, w.scale)
    rdq, rdk, rdv = ora.dualkv_backward(Q, K, V, DO, w.P, w.R_lens, w.scale)
    # the forward's exchange carries fp32 values of fp64 results
    np.testing.assert_allclose(out, ro, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(lse, rl, rtol=1e-6, atol=1e-6)
    # the gradient exchange runs in fp32
    for a, b in ((dq, rdq), (dk, rdk), (dv, rdv)):
        np.testing.assert_allclose(a, b, rtol=1e-5, atol=1e-5)


# --------------------------------------------------------------------------- kv-head split on CPU ranks

def test_head_bounds_cover_every_head_once():
    for Hkv in (1, 4, 8):
        for world in (1, 2, 4):
            spans = [sharded.head_bounds(Hkv, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == Hkv
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))


def _cpu_head_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, arrs = _case()
    Q, K, V, DO = (torch.from_numpy(a) for a in arrs)
    g = w.Hq // w.Hkv
    lo, hi = sharded.head_bounds(w.Hkv, world, rank)
    out, lse = sharded.heads_forward(Q, K, V, w.P, w.R_lens, w.scale, (lo, hi), fwd_fn=_oracle_fwd)
    dq, dk, dv = sharded.heads_backward(Q, K, V, out, DO, lse, w.P, w.R_lens, w.scale, (lo, hi), bwd_fn=_oracle_bwd)
    full = [sharded.gather_heads(out, w.Hq, lo * g, 1), sharded.gather_heads(lse, w.Hq, lo * g, 0),
            sharded.gather_heads(dq, w.Hq, lo * g, 1), sharded.gather_heads(dk, w.Hkv, lo, 1),
            sharded.gather_heads(dv, w.Hkv, lo, 1)]
    q.put((rank, np.arange(w.T)) + tuple(t.numpy() for t in full))
    dist.destroy_process_group()


def test_kv_head_split_on_two_cpu_ranks_matches_oracle():
    w, (Q, K, V, DO) = _case()
    res = _run_ranks(_cpu_head_rank, 2)
    ro, rl = ora.dualkv_forward(Q, K, V, w.P, w.R_lens, w.scale)
    rdq, rdk, rdv = ora.dualkv_backward(Q, K, V, DO, w.P, w.R_lens, w.scale)
    for r in res:
        # no gradient exchange: each head's values are its owner's, unchanged
        # up to the fp32 representation of the gather
        for a, b in zip(r[2:], (ro, rl, rdq, rdk, rdv)):
            np.testing.assert_allclose(a, b, rtol=1e-6, atol=1e-6)


# --------------------------------------------------------------------------- GPU: partial entry points

def _gpu_case():
    w = synthetic.make_workload("shard_gpu", 4, 2, 128, 300, (200, 0, 131, 128, 77))
    return w, synthetic.make_inputs(w, seed=6)


@pytest.mark.gpu
@pytest.mark.parametrize("det", [0, 1, 2], ids=["atomic", "deterministic", "atomic_fused_dq"])
def test_partial_entry_points_whole_prompt_equal_regular_calls(det):
    """(lo, hi) = (0, P): bf16 outputs are those of dualkv_fwd/dualkv_bwd bit
    for bit (to fp32 summation order where dQ is summed with atomics), and the
    fp32 prompt rows round (RNE) to the bf16 prompt rows."""
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    w, x = _gpu_case()
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    ro, rl = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    rdq, rdk, rdv = D.backward(q, k, v, ro, do, rl, w.P, w.R_lens, w.scale, deterministic=det)
    out, lse = torch.empty_like(ro), torch.empty_like(rl)
    D.dualkv_fwd_partial(q, k, v, w.P, w.R_lens, (0, w.P), out, lse, w.scale)
    ws = torch.empty(D.dualkv_bwd_workspace_bytes(w.P, w.R_lens, w.Hq, w.Hkv, w.d, det), dtype=torch.uint8,
                     device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    f32 = [torch.full((w.P, h, w.d), float("nan"), device="cuda") for h in (w.Hq, w.Hkv, w.Hkv)]
    D.dualkv_bwd_partial(q, k, v, out, do, lse, w.P, w.R_lens, (0, w.P), w.scale, det, ws, dq, dk, dv, *f32)
    assert D.dualkv_last_device_error()[0] == 0
    assert torch.equal(out, ro) and torch.equal(lse, rl)
    for a, b in ((dq, rdq), (dk, rdk), (dv, rdv)):
        if det == 2:   # dQ summed with atomics: the order varies from run to run
            assert ((a.float() - b.float()).norm() / b.float().norm()).item() <= 3e-3
        else:
            assert torch.equal(a, b)
    for a, b in zip(f32, (dq, dk, dv)):
        assert torch.equal(a.to(torch.bfloat16), b[:w.P])


@pytest.mark.gpu
@pytest.mark.parametrize("rows", [(0, 128), (128, 300), (256, 300), (128, 128)])
def test_partial_entry_points_prompt_part_matches_oracle(rows):
    """A part of the prompt's query rows: out/lse/dq of the other prompt rows
    are left untouched, and every output equals the oracle run with zero dO on
    the prompt rows outside the part."""
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    w, x = _gpu_case()
    lo, hi = rows
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.Hq, w.T), float("nan"), device="cuda")
    D.dualkv_fwd_partial(q, k, v, w.P, w.R_lens, rows, out, lse, w.scale)
    ref_o, ref_l = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    keep = torch.ones(w.T, dtype=torch.bool)
    keep[:lo] = False
    keep[hi:w.P] = False
    assert torch.isnan(out[~keep.cuda()].float()).all() and torch.isnan(lse[:, ~keep.cuda()]).all()
    assert torch.equal(out[keep.cuda()], ref_o[keep.cuda()]) and torch.equal(lse[:, keep.cuda()], ref_l[:, keep.cuda()])
    out[~keep.cuda()] = ref_o[~keep.cuda()]   # as the other ranks would supply
    lse[:, ~keep.cuda()] = ref_l[:, ~keep.cuda()]
    ws = torch.empty(D.dualkv_bwd_workspace_bytes(w.P, w.R_lens, w.Hq, w.Hkv, w.d, False), dtype=torch.uint8,
                     device="cuda")
    dq = torch.full_like(q, float("nan"))
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    dq_p = torch.full((w.P, w.Hq, w.d), float("nan"), device="cuda")
    dk_p, dv_p = (torch.empty((w.P, w.Hkv, w.d), device="cuda") for _ in range(2))
    D.dualkv_bwd_partial(q, k, v, out, do, lse, w.P, w.R_lens, rows, w.scale, False, ws, dq, dk, dv, dq_p, dk_p, dv_p)
    assert D.dualkv_last_device_error()[0] == 0
    assert torch.isnan(dq[~keep.cuda()].float()).all() and torch.isnan(dq_p[:lo]).all() and torch.isnan(dq_p[hi:]).all()
    do64 = synthetic.to_f64(x.dout)
    do64[:lo] = 0.0
    do64[hi:w.P] = 0.0
    f64 = [synthetic.to_f64(t) for t in (x.q, x.k, x.v)]
    rdq, rdk, rdv = ora.dualkv_backward(*f64, do64, w.P, w.R_lens, w.scale)
    k_np = keep.numpy()
    check_grads({"dq": (dq.float().cpu().numpy()[k_np], rdq[k_np]), "dk": (dk.float().cpu().numpy(), rdk),
                 "dv": (dv.float().cpu().numpy(), rdv)}, f"partial {rows}")
    if hi > lo:
        check_grads({"dq_p": (dq_p[lo:hi].cpu().numpy(), rdq[lo:hi])}, f"partial {rows} fp32")
    check_grads({"dk_p": (dk_p.cpu().numpy(), rdk[:w.P]), "dv_p": (dv_p.cpu().numpy(), rdv[:w.P])},
                f"partial {rows} fp32")
    check_forward(out.float().cpu().numpy(), lse.cpu().numpy(), *ora.dualkv_forward(*f64, w.P, w.R_lens, w.scale))


# --------------------------------------------------------------------------- GPU: two processes on one GPU

def _gpu_rank(rank, world, port, q, divide):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, x = _gpu_case()
    lo, hi = sharded.shard_bounds(w.N, world, rank)
    idx = sharded.local_rows(w.P, w.R_lens, lo, hi)
    t = [a[idx].contiguous().cuda() for a in (x.q, x.k, x.v, x.dout)]
    t[3][:w.P] = (t[3][:w.P].float() * SHARES[rank]).to(torch.bfloat16)
    R_local = list(w.R_lens[lo:hi])
    rows = sharded.prompt_bounds(w.P, world, rank) if divide else None
    out, lse = sharded.sharded_forward(t[0], t[1], t[2], w.P, R_local, w.scale, prompt_rows=rows)
    dq, dk, dv = sharded.sharded_backward(t[0], t[1], t[2], out, t[3], lse, w.P, R_local, w.scale, prompt_rows=rows,
                                          deterministic=True)
    torch.cuda.synchronize()
    q.put((rank, idx.numpy(), out.float().cpu().numpy(), lse.cpu().numpy(), dq.float().cpu().numpy(),
           dk.float().cpu().numpy(), dv.float().cpu().numpy()))
    dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("divide", [True, False], ids=["prompt_divided", "prompt_on_every_rank"])
def test_two_gpu_processes_match_oracle_and_unsharded_run(divide):
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    w, x = _gpu_case()
    res = _run_ranks(_gpu_rank, 2, (divide,))
    out, lse, dq, dk, dv = _assemble(res, w.T, w.Hq, w.Hkv, w.d, w.P)
    # the prompt rows' dO: the ranks' shares summed in fp32 and rounded once
    full_do = x.dout.clone()
    full_do[:w.P] = sum((x.dout[:w.P].float() * s).to(torch.bfloat16).float() for s in SHARES).to(torch.bfloat16)
    f64 = [synthetic.to_f64(t) for t in (x.q, x.k, x.v)]
    rdq, rdk, rdv = ora.dualkv_backward(*f64, synthetic.to_f64(full_do), w.P, w.R_lens, w.scale)
    check_grads({"dq": (dq, rdq), "dk": (dk, rdk), "dv": (dv, rdv)}, "sharded")
    # the forward, and the backward's response rows, are the unsharded run's, bit for bit
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, full_do))
    uo, ul = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    udq, udk, udv = D.backward(q, k, v, uo, do, ul, w.P, w.R_lens, w.scale, deterministic=True)
    np.testing.assert_array_equal(out, uo.float().cpu().numpy())
    np.testing.assert_array_equal(lse, ul.cpu().numpy())
    for a, b in ((dq, udq), (dk, udk), (dv, udv)):
        np.testing.assert_array_equal(a[w.P:], b.float().cpu().numpy()[w.P:])
    # prompt rows against the unsharded run's own.  With the prompt divided,
    # both runs see the same bf16 dO (the shares' fp32 sum rounded once) and
    # differ by the fp32 summation order; with the prompt on every rank, each
    # rank runs on its own bf16 share and the unsharded run on the rounded sum,
    # a dO difference of up to one bf16 rounding (about 2^-9 relative).
    bound = 3e-3 if divide else 1e-2
    for a, b in ((dq, udq), (dk, udk), (dv, udv)):
        bb = b.float().cpu().numpy()[:w.P]
        assert np.linalg.norm(a[:w.P] - bb) <= bound * np.linalg.norm(bb)


def _gpu_head_rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, x = _gpu_case()
    g = w.Hq // w.Hkv
    Q, K, V, DO = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    lo, hi = sharded.head_bounds(w.Hkv, world, rank)
    out, lse = sharded.heads_forward(Q, K, V, w.P, w.R_lens, w.scale, (lo, hi))
    dq, dk, dv = sharded.heads_backward(Q, K, V, out, DO, lse, w.P, w.R_lens, w.scale, (lo, hi), deterministic=True)
    torch.cuda.synchronize()
    full = [sharded.gather_heads(out.cpu(), w.Hq, lo * g, 1), sharded.gather_heads(lse.cpu(), w.Hq, lo * g, 0),
            sharded.gather_heads(dq.cpu(), w.Hq, lo * g, 1), sharded.gather_heads(dk.cpu(), w.Hkv, lo, 1),
            sharded.gather_heads(dv.cpu(), w.Hkv, lo, 1)]
    q.put((rank, None) + tuple(t.float().numpy() for t in full))
    dist.destroy_process_group()


@pytest.mark.gpu
def test_kv_head_split_on_two_gpu_processes_matches_unsharded_run():
    from shared_prompt_exact_dualkv_gb300 import dualkv as D
    w, x = _gpu_case()
    res = _run_ranks(_gpu_head_rank, 2)
    q, k, v, do = (t.cuda() for t in (x.q, x.k, x.v, x.dout))
    uo, ul = D.forward(q, k, v, w.P, w.R_lens, w.scale)
    ug = D.backward(q, k, v, uo, do, ul, w.P, w.R_lens, w.scale, deterministic=True)
    f64 = [synthetic.to_f64(t) for t in (x.q, x.k, x.v, x.dout)]
    rdq, rdk, rdv = ora.dualkv_backward(*f64, w.P, w.R_lens, w.scale)
    for r in res:
        out, lse, dq, dk, dv = r[2:]
        # each head is computed by the same kernels on the same rows
        np.testing.assert_array_equal(out, uo.float().cpu().numpy())
        np.testing.assert_array_equal(lse, ul.cpu().numpy())
        np.testing.assert_array_equal(dq, ug[0].float().cpu().numpy())
        check_grads({"dq": (dq, rdq), "dk": (dk, rdk), "dv": (dv, rdv)}, "kv-head split")
