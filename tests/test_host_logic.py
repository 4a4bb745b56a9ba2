"""Host-side logic without a GPU: workload arithmetic (packed token and pair
counts, rho, useful flops), the seeded generator, and the benchmark's
multi-rank timing reduction on 2 gloo ranks."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from shared_prompt_exact_dualkv_gb300 import synthetic

W = synthetic.WORKLOADS


def test_ragged_lengths_recipe():
    assert W["ragged_30b_a3b"].R_lens == (7045, 5404, 4438, 2584, 2876, 826, 1089, 638, 1858, 6758, 5500, 7522,
                                          4380, 5171, 7968, 6115)


@pytest.mark.parametrize("name,T,Trep,tflop,tflop_rep", [
    ("tiny", 384, 768, 8.81e-5, 1.328e-4),
    ("qwen3_8b", 135168, 262144, 46.66, 61.58),
    ("p32k", 65536, 557056, 94.29, 556.09),
    ("ragged_30b_a3b", 78364, 201244, 46.32, 75.18),
    ("edge_p64k", 81920, 1064960, 185.20, 2032.4),
    ("edge_n4", 40960, 65536, 25.02, 30.79),
])
def test_workload_sizes(name, T, Trep, tflop, tflop_rep):
    w = W[name]
    assert w.T == T and w.T_replicated == Trep
    assert w.useful_flops() / 1e12 == pytest.approx(tflop, rel=6e-3)
    assert w.replicated().useful_flops() / 1e12 == pytest.approx(tflop_rep, rel=6e-3)
    assert w.rho_tokens() == pytest.approx(Trep / T)


def test_pairs_brute_force():
    w = synthetic.make_workload("x", 1, 1, 64, 5, (3, 0, 2))
    off = w.offsets
    n = 0
    for t in range(w.T):
        if t < w.P:
            n += t + 1
        else:
            i = max(a for a in range(w.N) if off[a] <= t)
            n += w.P + (t - off[i] + 1)
    assert w.pairs_per_head() == n


def test_generator_is_seeded_bf16():
    w = W["tiny"]
    a = synthetic.make_inputs(w, 0)
    b = synthetic.make_inputs(w, 0)
    assert a.q.dtype == torch.bfloat16 and a.q.shape == (w.T, w.Hq, w.d) and a.k.shape == (w.T, w.Hkv, w.d)
    assert torch.equal(a.q, b.q) and torch.equal(a.dout, b.dout)
    assert not torch.equal(a.q, synthetic.make_inputs(w, 1).q)
    x = synthetic.to_f64(a.v)
    assert x.dtype == np.float64 and abs(x.std() - 1) < 0.05


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    mx = bench.max_over_ranks(10.0 + rank, world)
    val = bench.weak_scaling_value(1e12, mx, world)
    q.put((rank, mx, val))
    dist.destroy_process_group()


def test_bench_rank_reduction_gloo():
    """Two ranks: the step time is the slowest rank's and the value counts the
    work of both ranks (weak scaling)."""
    world = 2
    port = 29500 + os.getpid() % 1000
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, mx, val in res:
        assert mx == 11.0
        assert val == pytest.approx(2 * 1e12 / 11e-3 / 1e12)
