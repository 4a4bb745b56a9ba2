"""The attention oracle for one kv-head group, evaluated with PyTorch CPU fp64
ops (multi-threaded), for workloads where the NumPy oracle in
``attention.py`` would take hours.

TEST INFRASTRUCTURE ONLY: used by ``tests/`` alone, never by the product
path; it shares no code with the CUDA library.

Definition (the same as ``attention.py``; sources: "DualKV: Shared-Prompt
Flash Attention for Efficient RL Training with Large Rollouts and Long
Contexts", research-map page, section "Approach"; arXiv abstract page; forum
page, "Two changes"): every sequence is X_i = [prompt ; response_i] under
textbook causal softmax attention, in fp64, and the results are scattered
back to the packed rows; prompt-row gradients are summed over the sequences.

Two facts of that definition, both pinned for the NumPy oracle in
``tests/test_oracle.py`` (prompt rows identical across sequences; packed dO
of a prompt row fed to sequence 0 with zeros elsewhere, equivalent to any
split), let this module evaluate it without repeating work:

* the prompt rows of X_i are the same rows, with the same keys, in every
  sequence, so they are computed once;
* with zero dO on the prompt rows of sequences i > 0, those rows have
  D = 0 and dP = 0, hence dS = 0: they add nothing to any gradient.

So the prompt rows are computed once, with the full packed prompt dO, and
each response's rows are computed against the prompt keys followed by the
response's own keys.  ``tests/test_oracle.py`` pins this module against
``attention.py`` to fp64 rounding.

All q-heads of the group are processed together ([g, rows, keys] score
blocks); GQA: they share one kv-head.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

ROW_BLOCK = 256


def _block_fwd(qb, kk, vv, scale, vis, n_open=0):
    """Scores, log-sum-exp, probabilities and outputs of one row block.

    qb [g, b, d]; kk, vv [nk, d]; vis [b, nk - n_open] bool: whether each key
    after the first ``n_open`` (which every row sees) is visible to the row.
    Softmax with the row maximum: p = exp(s - m) / l, l = sum exp(s - m),
    lse = m + log l."""
    s = torch.matmul(qb, kk.T).mul_(scale)                 # [g, b, nk]
    s[:, :, n_open:].masked_fill_(~vis, float("-inf"))
    m = s.amax(dim=2, keepdim=True)
    p = s.sub_(m).exp_()                                  # exp(-inf) = 0 on masked keys
    l = p.sum(dim=2, keepdim=True)
    p.div_(l)
    o = torch.matmul(p, vv)                               # [g, b, d]
    return p, o, (m + torch.log(l)).squeeze(2)


def _block_bwd(qb, kk, vv, p, o, dob, scale):
    """dQ of the block's rows and the block's dK/dV contributions to its keys.

    D = rowsum(dO*O), dV = P^T dO, dP = dO V^T, dS = P*(dP - D),
    dQ = scale dS K, dK = scale dS^T Q (summed over the group's heads)."""
    Dr = (dob * o).sum(dim=2, keepdim=True)               # [g, b, 1]
    dv = torch.matmul(p.transpose(1, 2), dob).sum(dim=0)  # [nk, d]
    dp = torch.matmul(dob, vv.T)                          # [g, b, nk]
    ds = p.mul_(dp.sub_(Dr))                              # p is not used afterwards
    dq = torch.matmul(ds, kk).mul_(scale)                 # [g, b, d]
    dk = torch.matmul(ds.transpose(1, 2), qb).sum(dim=0).mul_(scale)
    return dq, dk, dv


def kvgroup_forward_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: Optional[torch.Tensor],
                             P: int, R_lens: Sequence[int], scale: float, row_block: int = ROW_BLOCK):
    """Packed forward (and backward if ``dout`` is given) of one kv-head group.

    q, dout: [T, g, d] float64 (the g q-heads that read this kv-head);
    k, v: [T, d] float64.  T = P + sum(R_lens); response i is packed rows
    [off_i, off_i + R_i) with off_0 = P.
    Returns a dict with out [T, g, d], lse [g, T] and, with dout, dq [T, g, d],
    dk [T, d], dv [T, d].
    """
    T, g, d = q.shape
    off = [int(P)]
    for r in R_lens:
        off.append(off[-1] + int(r))
    if off[-1] != T or k.shape != (T, d) or v.shape != (T, d):
        raise ValueError("q [T,g,d], k/v [T,d] with T = P + sum(R_lens) expected")
    qh = q.permute(1, 0, 2)                               # [g, T, d] view
    doh = None if dout is None else dout.permute(1, 0, 2)
    out = torch.zeros((g, T, d), dtype=torch.float64)
    lse = torch.zeros((g, T), dtype=torch.float64)
    if dout is not None:
        dq = torch.zeros((g, T, d), dtype=torch.float64)
        dk = torch.zeros((T, d), dtype=torch.float64)
        dv = torch.zeros((T, d), dtype=torch.float64)

    def run(rows0, rows1, kidx_lo, kidx_hi, causal_from):
        # rows [rows0, rows1) see prompt keys [0, kidx_lo) unmasked (kidx_lo = 0
        # for prompt rows) and keys [causal_from, ...) causally up to themselves.
        kk = torch.cat([k[:kidx_lo], k[causal_from:kidx_hi]])
        vv = torch.cat([v[:kidx_lo], v[causal_from:kidx_hi]])
        vis = torch.arange(causal_from, kidx_hi)[None, :] <= torch.arange(rows0, rows1)[:, None]
        p, o, l = _block_fwd(qh[:, rows0:rows1], kk, vv, scale, vis, n_open=kidx_lo)
        out[:, rows0:rows1] = o
        lse[:, rows0:rows1] = l
        if dout is not None:
            bq, bk, bv = _block_bwd(qh[:, rows0:rows1], kk, vv, p, o, doh[:, rows0:rows1], scale)
            dq[:, rows0:rows1] = bq
            n_pre = kidx_lo
            dk[:kidx_lo] += bk[:n_pre]
            dv[:kidx_lo] += bv[:n_pre]
            dk[causal_from:kidx_hi] += bk[n_pre:]
            dv[causal_from:kidx_hi] += bv[n_pre:]

    # prompt rows (once): causal within the prompt
    for r0 in range(0, P, row_block):
        r1 = min(r0 + row_block, P)
        run(r0, r1, 0, r1, 0)
    # response rows: every prompt key, then their own response causally
    for i in range(len(R_lens)):
        for r0 in range(off[i], off[i + 1], row_block):
            r1 = min(r0 + row_block, off[i + 1])
            run(r0, r1, P, r1, off[i])
    res = {"out": out.permute(1, 0, 2), "lse": lse}
    if dout is not None:
        res.update(dq=dq.permute(1, 0, 2), dk=dk, dv=dv)
    return res


def kvgroup_rows(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor, P: int,
                 R_lens: Sequence[int], scale: float, row_ranges: Sequence[tuple], row_block: int = ROW_BLOCK):
    """O, LSE and dQ of selected query rows of one kv-head group.

    ``row_ranges`` lists (first, end) packed-row ranges, each inside one
    segment (the prompt or one response).  Each row's softmax runs over its
    full visible key set.  Returns dicts keyed by the range with out
    [g, n, d], lse [g, n] and dq [g, n, d]."""
    T, g, d = q.shape
    off = [int(P)]
    for r in R_lens:
        off.append(off[-1] + int(r))
    qh = q.permute(1, 0, 2)
    doh = dout.permute(1, 0, 2)
    res = {}
    for a, b in row_ranges:
        if a < P:
            if b > P:
                raise ValueError("a row range must not straddle the prompt end")
            lo, start = 0, 0
        else:
            i = max(j for j in range(len(R_lens)) if off[j] <= a)
            if b > off[i + 1]:
                raise ValueError("a row range must stay inside one response")
            lo, start = P, off[i]
        outs, lses, dqs = [], [], []
        for r0 in range(a, b, row_block):
            r1 = min(r0 + row_block, b)
            kk = torch.cat([k[:lo], k[start:r1]])
            vv = torch.cat([v[:lo], v[start:r1]])
            vis = torch.arange(start, r1)[None, :] <= torch.arange(r0, r1)[:, None]
            p, o, l = _block_fwd(qh[:, r0:r1], kk, vv, scale, vis, n_open=lo)
            bq, _, _ = _block_bwd(qh[:, r0:r1], kk, vv, p, o, doh[:, r0:r1], scale)
            outs.append(o)
            lses.append(l)
            dqs.append(bq)
        res[(a, b)] = {"out": torch.cat(outs, dim=1), "lse": torch.cat(lses, dim=1), "dq": torch.cat(dqs, dim=1)}
    return res
