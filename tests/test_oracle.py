"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: a worked example
derived by hand, brute force over the packed-row definition, finite
differences, closed forms, invariants of the method (prompt rows identical
across sequences; linearity of the prompt-row gradient), and an independent
library routine (torch's fp64 scaled_dot_product_attention with autograd on the
replicated sequences).  The mutation tests at the end plant plausible mistakes
in copies of the oracle and check that a pin catches each one.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as ora

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(P, R_lens, Hq, Hkv, d, seed=0):
    rng = np.random.default_rng(seed)
    T = P + sum(R_lens)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    do = rng.standard_normal((T, Hq, d))
    return q, k, v, do


# --------------------------------------------------------------------------- golden

def test_hand_worked_example():
    """Values derived by hand (tests/golden/hand_example.json)."""
    g = json.load(open(os.path.join(GOLDEN, "hand_example.json")))
    q, k, v, do = (np.array(g[n], dtype=np.float64) for n in ("q", "k", "v", "dout"))
    out, lse = ora.dualkv_forward(q, k, v, g["P"], g["R_lens"], g["scale"])
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, g["P"], g["R_lens"], g["scale"])
    e = g["expected"]
    np.testing.assert_allclose(out, e["out"], atol=1e-12)
    np.testing.assert_allclose(lse, e["lse"], atol=1e-12)
    np.testing.assert_allclose(dq, e["dq"], atol=1e-12)
    np.testing.assert_allclose(dk, e["dk"], atol=1e-12)
    np.testing.assert_allclose(dv, e["dv"], atol=1e-12)


# --------------------------------------------------------------------------- brute force

def brute_force_forward(q, k, v, P, R_lens, scale):
    """Scalar loops over the packed-row definition: a prompt row t sees keys
    j <= t; a row of response i sees every prompt key and its own response's
    keys up to itself."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    off = [P]
    for r in R_lens:
        off.append(off[-1] + r)
    out = np.zeros((T, Hq, d))
    lse = np.zeros((Hq, T))
    for h in range(Hq):
        for t in range(T):
            if t < P:
                vis = list(range(t + 1))
            else:
                i = max(a for a in range(len(R_lens)) if off[a] <= t)
                vis = list(range(P)) + list(range(off[i], t + 1))
            sc = []
            for j in vis:
                acc = 0.0
                for c in range(d):
                    acc += q[t, h, c] * k[j, h // g, c]
                sc.append(scale * acc)
            m = max(sc)
            den = sum(math.exp(s - m) for s in sc)
            lse[h, t] = m + math.log(den)
            for c in range(d):
                out[t, h, c] = sum(math.exp(s - m) / den * v[j, h // g, c] for s, j in zip(sc, vis))
    return out, lse


@pytest.mark.parametrize("P,R_lens,Hq,Hkv,d", [(2, [1, 2], 1, 1, 4), (3, [0, 4, 2], 2, 1, 3), (0, [3, 2], 2, 2, 2)])
def test_brute_force_forward(P, R_lens, Hq, Hkv, d):
    q, k, v, _ = rand_case(P, R_lens, Hq, Hkv, d, seed=1)
    scale = 1 / math.sqrt(d)
    out, lse = ora.dualkv_forward(q, k, v, P, R_lens, scale)
    bo, bl = brute_force_forward(q, k, v, P, R_lens, scale)
    np.testing.assert_allclose(out, bo, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- finite differences

def test_finite_differences():
    """Central differences of L = sum(dO * O(q, k, v)) on the packed inputs
    agree with the oracle's dQ/dK/dV (this also pins the summation of the
    prompt gradients over the N sequences)."""
    P, R_lens, Hq, Hkv, d = 3, [2, 3], 2, 1, 4
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=2)
    scale = 1 / math.sqrt(d)

    def loss(q_, k_, v_):
        return float((ora.dualkv_forward(q_, k_, v_, P, R_lens, scale)[0] * do).sum())

    dq, dk, dv = ora.dualkv_backward(q, k, v, do, P, R_lens, scale)
    h = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}; args_p[name] = xp
            args_m = {"q": q, "k": k, "v": v}; args_m[name] = xm
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"]) -
                       loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=name)


# --------------------------------------------------------------------------- library routine

def sdpa_packed(q, k, v, do, P, R_lens, scale, split="first"):
    """fp64 torch SDPA with autograd on the replicated sequences gathered from
    the packed tensors; the gather sums prompt-row gradients over sequences."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    g = Hq // Hkv
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    off = [P]
    for r in R_lens:
        off.append(off[-1] + r)
    outs = torch.zeros((T, Hq, d), dtype=torch.float64)
    lses = torch.zeros((Hq, T), dtype=torch.float64)
    loss = 0.0
    N = len(R_lens)
    dot = torch.tensor(do)
    for i, R in enumerate(R_lens):
        idx = torch.cat([torch.arange(P), torch.arange(off[i], off[i] + R)])
        L = len(idx)
        qi = qt[idx].permute(1, 0, 2)                      # [Hq, L, d]
        ki = kt[idx].repeat_interleave(g, dim=1).permute(1, 0, 2)
        vi = vt[idx].repeat_interleave(g, dim=1).permute(1, 0, 2)
        mask = torch.ones((L, L), dtype=torch.bool).tril()
        o = torch.nn.functional.scaled_dot_product_attention(qi, ki, vi, attn_mask=mask, scale=scale)
        s = scale * qi @ ki.transpose(-1, -2)
        s = s.masked_fill(~mask, float("-inf"))
        lse = torch.logsumexp(s, dim=-1)
        doi = dot[idx].permute(1, 0, 2).clone()
        if split == "first":
            if i > 0:
                doi[:, :P] = 0
        else:
            doi[:, :P] = doi[:, :P] / N
        loss = loss + (o * doi).sum()
        with torch.no_grad():
            outs[off[i]:off[i] + R] = o[:, P:].permute(1, 0, 2)
            lses[:, off[i]:off[i] + R] = lse[:, P:]
            if i == 0:
                outs[:P] = o[:, :P].permute(1, 0, 2)
                lses[:, :P] = lse[:, :P]
    loss.backward()
    return outs.numpy(), lses.numpy(), qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("P,R_lens,Hq,Hkv,d", [
    (128, [64] * 4, 2, 1, 64),                 # the Tiny shape
    (37, [5, 0, 19, 1], 4, 2, 8),              # ragged, an empty response, GQA 2:1
    (0, [7, 3], 2, 1, 4),                      # P = 0: independent causal sequences
    (11, [6], 3, 1, 4),                        # N = 1: plain causal attention on P+R
])
def test_against_torch_sdpa(P, R_lens, Hq, Hkv, d):
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=3)
    scale = 1 / math.sqrt(d)
    out, lse = ora.dualkv_forward(q, k, v, P, R_lens, scale)
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, P, R_lens, scale)
    for split in ("first", "equal"):
        to, tl, tdq, tdk, tdv = sdpa_packed(q, k, v, do, P, R_lens, scale, split=split)
        np.testing.assert_allclose(out, to, atol=1e-12)
        np.testing.assert_allclose(lse, tl, atol=1e-12)
        np.testing.assert_allclose(dq, tdq, atol=1e-11)
        np.testing.assert_allclose(dk, tdk, atol=1e-11)
        np.testing.assert_allclose(dv, tdv, atol=1e-11)


@pytest.mark.parametrize("scale", [0.3, 0.05, 1.7])
def test_caller_scale_against_torch_sdpa(scale):
    """The scale is the caller's argument: the oracle with a scale other than
    1/sqrt(d) matches torch's SDPA given the same scale, and scaling q instead
    (q -> a*q with the scale divided by a) gives the same out and LSE and a
    times the dQ."""
    P, R_lens, Hq, Hkv, d = 37, [5, 0, 19, 1], 4, 2, 8
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=5)
    out, lse = ora.dualkv_forward(q, k, v, P, R_lens, scale)
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, P, R_lens, scale)
    to, tl, tdq, tdk, tdv = sdpa_packed(q, k, v, do, P, R_lens, scale)
    for a, b in ((out, to), (lse, tl), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, atol=1e-11)
    a = 2.5
    out2, lse2 = ora.dualkv_forward(a * q, k, v, P, R_lens, scale / a)
    dq2, dk2, dv2 = ora.dualkv_backward(a * q, k, v, do, P, R_lens, scale / a)
    np.testing.assert_allclose(out2, out, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, atol=1e-12)
    np.testing.assert_allclose(a * dq2, dq, atol=1e-11)
    np.testing.assert_allclose(dk2, dk, atol=1e-11)
    np.testing.assert_allclose(dv2, dv, atol=1e-11)


@pytest.mark.slow
def test_against_torch_sdpa_midsize():
    """One head group of a mid-size case (P=1024, N=4, R=256)."""
    P, R_lens, Hq, Hkv, d = 1024, [256] * 4, 2, 1, 128
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=4)
    scale = 1 / math.sqrt(d)
    out, lse = ora.dualkv_forward(q, k, v, P, R_lens, scale)
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, P, R_lens, scale)
    to, tl, tdq, tdk, tdv = sdpa_packed(q, k, v, do, P, R_lens, scale)
    for a, b in ((out, to), (lse, tl), (dq, tdq), (dk, tdk), (dv, tdv)):
        np.testing.assert_allclose(a, b, atol=1e-10)


# --------------------------------------------------------------------------- closed forms

def test_zero_queries_give_uniform_attention():
    """Q = 0: every visible key scores 0, so LSE = ln(#visible keys) and O is
    the mean of the visible V rows."""
    P, R_lens, Hq, Hkv, d = 5, [3, 4], 2, 1, 3
    _, k, v, _ = rand_case(P, R_lens, Hq, Hkv, d, seed=5)
    q = np.zeros((P + sum(R_lens), Hq, d))
    out, lse = ora.dualkv_forward(q, k, v, P, R_lens, 0.5)
    off = ora.segment_offsets(P, R_lens)
    for t in range(P + sum(R_lens)):
        if t < P:
            vis = list(range(t + 1))
        else:
            i = max(a for a in range(len(R_lens)) if off[a] <= t)
            vis = list(range(P)) + list(range(off[i], t + 1))
        for h in range(Hq):
            assert abs(lse[h, t] - math.log(len(vis))) < 1e-14
            np.testing.assert_allclose(out[t, h], v[vis, 0].mean(axis=0), atol=1e-14)


def test_constant_values_give_zero_qk_grads():
    """All V rows equal v: O = v for every row, and dQ = dK = 0."""
    P, R_lens, Hq, Hkv, d = 6, [2, 5, 1], 2, 1, 4
    q, k, _, do = rand_case(P, R_lens, Hq, Hkv, d, seed=6)
    v = np.broadcast_to(np.arange(1.0, d + 1), (P + sum(R_lens), Hkv, d)).copy()
    out, _ = ora.dualkv_forward(q, k, v, P, R_lens, 0.5)
    np.testing.assert_allclose(out, np.broadcast_to(v[:1, :1], out.shape), atol=1e-13)
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, P, R_lens, 0.5)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12
    assert np.abs(dv).max() > 0.1


# --------------------------------------------------------------------------- invariants

def test_prompt_rows_identical_across_sequences():
    """Causal masking makes the prompt rows the same in every replicated
    sequence (arXiv abstract page): the oracle raises if they differ; here we
    also check it directly on two sequences with different responses."""
    P, R_lens, Hq, Hkv, d = 300, [40, 300], 2, 1, 16
    q, k, v, _ = rand_case(P, R_lens, Hq, Hkv, d, seed=7)
    off = ora.segment_offsets(P, R_lens)
    res = []
    for i in range(2):
        idx = np.concatenate([np.arange(P), np.arange(off[i], off[i + 1])])
        res.append(ora.causal_attention_fwd(q[idx, 0], k[idx, 0], v[idx, 0], 0.25, split_at=P))
    assert np.array_equal(res[0][0][:P], res[1][0][:P])
    assert np.array_equal(res[0][1][:P], res[1][1][:P])


def test_prompt_dout_split_invariance():
    """Prompt-row gradients are linear in dO: any split of the packed prompt dO
    over the N sequences (summing to it) gives the same dQ/dK/dV."""
    P, R_lens, Hq, Hkv, d = 9, [4, 7, 3], 4, 2, 5
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=8)
    ref = ora.dualkv_backward(q, k, v, do, P, R_lens, 0.4)
    rng = np.random.default_rng(9)
    parts = [rng.standard_normal((P, Hq, d)) for _ in range(len(R_lens) - 1)]
    parts.append(do[:P] - sum(parts))
    for split in (parts, [do[:P] / len(R_lens)] * len(R_lens)):
        got = ora.dualkv_backward(q, k, v, do, P, R_lens, 0.4, prompt_dout_split=split)
        for a, b in zip(ref, got):
            np.testing.assert_allclose(a, b, atol=1e-12)


def test_column_sum_identities():
    """sum_k dV[k] = sum over the group's q-heads and all packed rows of dO
    (each softmax row sums to 1), and sum_k dK[k] = 0 (each dS row sums to 0)."""
    P, R_lens, Hq, Hkv, d = 20, [9, 13], 4, 2, 6
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=10)
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, P, R_lens, 0.3)
    for j in range(Hkv):
        np.testing.assert_allclose(dv[:, j].sum(0), do[:, 2 * j:2 * j + 2].sum((0, 1)), atol=1e-12)
        np.testing.assert_allclose(dk[:, j].sum(0), 0.0, atol=1e-12)


# --------------------------------------------------------------------------- row-sampled oracle

def test_sampled_rows_match_full_oracle():
    P, R_lens, Hq, Hkv, d = 70, [33, 0, 50, 7], 4, 2, 8
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=11)
    scale = 1 / math.sqrt(d)
    out, lse = ora.dualkv_forward(q, k, v, P, R_lens, scale)
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, P, R_lens, scale)
    T = P + sum(R_lens)
    rows = [0, 1, 69, 70, 102, 103, 140, 159, T - 1]
    heads = [0, 3]
    r = ora.rows_forward_backward(q, k, v, do, P, R_lens, scale, heads, rows)
    for a, h in enumerate(heads):
        np.testing.assert_allclose(r["o"][a], out[rows, h], atol=1e-12)
        np.testing.assert_allclose(r["lse"][a], lse[h, rows], atol=1e-12)
        np.testing.assert_allclose(r["dq"][a], dq[rows, h], atol=1e-12)
    for keys in ([0, 5, 69], [70, 100, 130, 159], [3, 69, 80, 150]):
        for j in range(Hkv):
            skd, svd = ora.keys_dkdv(q, k, v, do, P, R_lens, scale, j, keys, row_block=16)
            np.testing.assert_allclose(skd, dk[keys, j], atol=1e-12)
            np.testing.assert_allclose(svd, dv[keys, j], atol=1e-12)


# --------------------------------------------------------------------------- kv-group oracle (torch fp64)

@pytest.mark.parametrize("P,R_lens,Hq,Hkv,d,row_block", [
    (70, [33, 0, 50, 7], 4, 2, 8, 16),      # ragged, an empty response, blocks inside segments
    (0, [40, 17], 2, 1, 8, 16),             # P = 0: independent causal sequences
    (45, [0], 2, 2, 4, 8),                  # a prompt alone
    (33, [64], 6, 2, 8, 64),                # N = 1, group of 3 q-heads
])
def test_kvgroup_oracle_matches_numpy_oracle(P, R_lens, Hq, Hkv, d, row_block):
    """The torch kv-group evaluation (prompt rows once, responses against
    prompt + own keys) equals the replicated NumPy oracle to fp64 rounding,
    for every output, including complete row ranges through kvgroup_rows."""
    from oracle import kvgroup as okg
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=12)
    scale = 1 / math.sqrt(d)
    out, lse = ora.dualkv_forward(q, k, v, P, R_lens, scale)
    dq, dk, dv = ora.dualkv_backward(q, k, v, do, P, R_lens, scale)
    g = Hq // Hkv
    T = P + sum(R_lens)
    off = ora.segment_offsets(P, R_lens)
    ranges = [(a, min(a + 16, b)) for a, b in ([(0, P)] + [(off[i], off[i + 1]) for i in range(len(R_lens))]) if b > a]
    for j in range(Hkv):
        hs = slice(j * g, (j + 1) * g)
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x))
        r = okg.kvgroup_forward_backward(t(q[:, hs]), t(k[:, j]), t(v[:, j]), t(do[:, hs]), P, R_lens, scale,
                                         row_block=row_block)
        np.testing.assert_allclose(r["out"].numpy(), out[:, hs], atol=1e-12)
        np.testing.assert_allclose(r["lse"].numpy(), lse[hs], atol=1e-12)
        np.testing.assert_allclose(r["dq"].numpy(), dq[:, hs], atol=1e-12)
        np.testing.assert_allclose(r["dk"].numpy(), dk[:, j], atol=1e-12)
        np.testing.assert_allclose(r["dv"].numpy(), dv[:, j], atol=1e-12)
        f = okg.kvgroup_forward_backward(t(q[:, hs]), t(k[:, j]), t(v[:, j]), None, P, R_lens, scale)
        np.testing.assert_allclose(f["out"].numpy(), out[:, hs], atol=1e-12)
        rr = okg.kvgroup_rows(t(q[:, hs]), t(k[:, j]), t(v[:, j]), t(do[:, hs]), P, R_lens, scale, ranges,
                              row_block=5)
        for a, b in ranges:
            np.testing.assert_allclose(rr[(a, b)]["out"].numpy(), out[a:b, hs].transpose(1, 0, 2), atol=1e-12)
            np.testing.assert_allclose(rr[(a, b)]["lse"].numpy(), lse[hs, a:b], atol=1e-12)
            np.testing.assert_allclose(rr[(a, b)]["dq"].numpy(), dq[a:b, hs].transpose(1, 0, 2), atol=1e-12)
    assert T == off[-1]


def test_kvgroup_oracle_catches_a_dropped_response_key():
    """A kv-group evaluation that leaves out a response row's own diagonal key
    disagrees with the replicated oracle (the comparison above can fail)."""
    from oracle import kvgroup as okg
    P, R_lens, Hq, Hkv, d = 20, [9, 13], 2, 1, 6
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=13)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x))
    real = okg._block_fwd

    def no_diag(qb, kk, vv, scale, vis, n_open=0):
        b = vis.shape[0]
        vis = vis & ~torch.eye(b, vis.shape[1], dtype=torch.bool, device=vis.device).roll(vis.shape[1] - b, 1)
        return real(qb, kk, vv, scale, vis, n_open)

    out, _ = ora.dualkv_forward(q, k, v, P, R_lens, 0.4)
    okg._block_fwd = no_diag
    try:
        r = okg.kvgroup_forward_backward(t(q), t(k[:, 0]), t(v[:, 0]), None, P, R_lens, 0.4, row_block=4)
    finally:
        okg._block_fwd = real
    assert not np.allclose(r["out"].numpy(), out, atol=1e-3)   # NaN rows (nothing visible) also fail


# --------------------------------------------------------------------------- planted mistakes

def _mutant(monkeypatch, fwd=None, bwd=None):
    if fwd is not None:
        monkeypatch.setattr(ora, "causal_attention_fwd", fwd)
    if bwd is not None:
        monkeypatch.setattr(ora, "causal_attention_bwd", bwd)


def _pins_fail():
    """True if the SDPA cross-check or the hand example rejects the oracle."""
    try:
        test_against_torch_sdpa(37, [5, 0, 19, 1], 4, 2, 8)
        test_hand_worked_example()
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught(monkeypatch):
    real_fwd, real_bwd = ora.causal_attention_fwd, ora.causal_attention_bwd

    def fwd_no_diagonal(q, k, v, scale, split_at=0):
        L = q.shape[0]
        o, lse = real_fwd(q, k, v, scale, split_at)
        # a query that does not see its own key
        s = scale * q @ k.T
        m = np.tril(np.ones((L, L), bool), -1)
        m[0, 0] = True
        s = np.where(m, s, -np.inf)
        lse2 = np.log(np.exp(s - s.max(1, keepdims=True)).sum(1)) + s.max(1)
        return np.exp(s - lse2[:, None]) @ v, lse2

    def bwd_dk_unscaled(q, k, v, o, lse, do, scale, split_at=0):
        dq, dk, dv = real_bwd(q, k, v, o, lse, do, scale, split_at)
        return dq, dk / scale, dv

    def bwd_d_sign(q, k, v, o, lse, do, scale, split_at=0):
        return real_bwd(q, k, v, -o, lse, do, scale, split_at)

    for f, b in ((fwd_no_diagonal, None), (None, bwd_dk_unscaled), (None, bwd_d_sign)):
        with monkeypatch.context() as m:
            _mutant(m, f, b)
            assert _pins_fail()
    assert not _pins_fail()


def test_planted_prompt_grads_not_summed(monkeypatch):
    """An oracle that keeps only sequence 0's prompt dK/dV fails finite differences."""
    real = ora.dualkv_backward

    def first_only(q, k, v, dout, P, R_lens, scale, heads=None, prompt_dout_split=None):
        n0 = P + R_lens[0]
        _, dk0, dv0 = real(q[:n0], k[:n0], v[:n0], dout[:n0], P, R_lens[:1], scale)
        dq, dk, dv = (x.copy() for x in real(q, k, v, dout, P, R_lens, scale))
        dk[:P] = dk0[:P]
        dv[:P] = dv0[:P]
        return dq, dk, dv

    monkeypatch.setattr(ora, "dualkv_backward", first_only)
    with pytest.raises(AssertionError):
        test_finite_differences()


# --------------------------------------------------------------------------- several prompt groups

def group_mask(groups):
    """Dense [T, T] visibility of the packed multi-group batch, written from
    the rule alone: key j is visible to row t iff both are in the same group
    and j <= t, except that a response row sees only its own response's keys
    besides the group's prompt."""
    seg = []        # per row: (group, response index or -1 for the prompt)
    for gi, (P_g, R_g) in enumerate(groups):
        seg += [(gi, -1)] * P_g
        for i, r in enumerate(R_g):
            seg += [(gi, i)] * r
    T = len(seg)
    m = np.zeros((T, T), dtype=bool)
    for t in range(T):
        for j in range(t + 1):
            same_group = seg[j][0] == seg[t][0]
            m[t, j] = same_group and (seg[j][1] == -1 or seg[j][1] == seg[t][1])
    return m


def sdpa_dense(q, k, v, do, mask, scale):
    """fp64 torch SDPA with autograd over the packed rows under a dense mask:
    every packed row appears once, so autograd gives the packed gradient."""
    Hq, Hkv = q.shape[1], k.shape[1]
    g = Hq // Hkv
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    qh = qt.permute(1, 0, 2)
    kh = kt.repeat_interleave(g, dim=1).permute(1, 0, 2)
    vh = vt.repeat_interleave(g, dim=1).permute(1, 0, 2)
    mt = torch.tensor(mask)
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mt, scale=scale)
    s = (scale * qh @ kh.transpose(-1, -2)).masked_fill(~mt, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    (o * torch.tensor(do).permute(1, 0, 2)).sum().backward()
    return (o.detach().permute(1, 0, 2).numpy(), lse.detach().numpy(), qt.grad.numpy(), kt.grad.numpy(),
            vt.grad.numpy())


GROUP_CASES = [
    [(5, [3, 0, 4]), (0, [2, 6]), (7, [1]), (4, [])],     # ragged; P_g = 0; N_g = 1; N_g = 0
    [(9, [2, 2]), (9, [2, 2])],                           # two equal groups
    [(3, [4])],                                           # one group
]


@pytest.mark.parametrize("groups", GROUP_CASES)
def test_groups_against_dense_mask_sdpa(groups):
    T = ora.group_row_starts(groups)[-1]
    Hq, Hkv, d = 4, 2, 8
    rng = np.random.default_rng(11)
    q = rng.standard_normal((T, Hq, d))
    k = rng.standard_normal((T, Hkv, d))
    v = rng.standard_normal((T, Hkv, d))
    do = rng.standard_normal((T, Hq, d))
    scale = 1 / math.sqrt(d)
    out, lse = ora.dualkv_forward_groups(q, k, v, groups, scale)
    dq, dk, dv = ora.dualkv_backward_groups(q, k, v, do, groups, scale)
    to, tl, tdq, tdk, tdv = sdpa_dense(q, k, v, do, group_mask(groups), scale)
    np.testing.assert_allclose(out, to, atol=1e-12)
    np.testing.assert_allclose(lse, tl, atol=1e-12)
    np.testing.assert_allclose(dq, tdq, atol=1e-11)
    np.testing.assert_allclose(dk, tdk, atol=1e-11)
    np.testing.assert_allclose(dv, tdv, atol=1e-11)


def test_group_mask_single_group_matches_replicated_sdpa():
    """The dense-mask formulation agrees with the replicated-sequence one on a
    single group (ties the two library cross-checks together)."""
    P, R_lens, Hq, Hkv, d = 6, [3, 0, 5], 2, 1, 4
    q, k, v, do = rand_case(P, R_lens, Hq, Hkv, d, seed=12)
    a = sdpa_dense(q, k, v, do, group_mask([(P, R_lens)]), 0.5)
    b = sdpa_packed(q, k, v, do, P, R_lens, 0.5)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)


def test_planted_group_leak_is_caught(monkeypatch):
    """A group oracle that shifts the groups' row ranges by one row fails the
    dense-mask pin."""
    real = ora.group_row_starts

    def shifted(groups):
        s = list(real(groups))
        s[1] += 1
        return s

    monkeypatch.setattr(ora, "group_row_starts", shifted)
    with pytest.raises((AssertionError, ValueError)):
        test_groups_against_dense_mask_sdpa(GROUP_CASES[0])
