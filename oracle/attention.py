"""fp64 CPU oracle for exact shared-prompt (DualKV) attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the
CUDA library; both sides are fed by the seeded generators in
``shared_prompt_exact_dualkv_gb300/synthetic.py``.

What it computes (sources: "DualKV: Shared-Prompt Flash Attention for Efficient
RL Training with Large Rollouts and Long Contexts" -- research-map page,
section "Approach"; arXiv abstract page; forum page, "Two changes"):

* A micro-batch of N responses to one prompt is packed as the P prompt rows
  followed by the N responses (P + sum R_i rows).  The method is exact: it
  equals standard causal attention run on each replicated sequence
  X_i = [prompt ; response_i] (abstract: "mathematically equivalent to standard
  attention"; causal masking keeps the prompt rows the same in every sequence).
* So the oracle materialises every X_i, runs textbook causal softmax attention
  on it in fp64, and scatters the results back to the packed layout: response
  rows are copied, prompt rows of O and LSE are taken from sequence 0 after
  checking that all N sequences produced the same bits, and prompt rows of
  dQ/dK/dV are summed over the N sequences (the research-map page, "Approach":
  the shared prompt's gradients are accumulated across sequences).

Readings where the pages are silent:

* LSE is the natural log of sum_j exp(scale * q.k_j) (FlashAttention-2
  convention, the lineage named on the research-map page), layout [Hq, T].
* A query attends to its own key (j <= r).
* Packed dO for a prompt row is the sum of the N sequences' dO for that row
  (the gradient of the one shared hidden state).  Since prompt-row gradients
  are linear in dO, the oracle feeds it to sequence 0 and zeros to the others;
  ``prompt_dout_split`` lets a test spread it differently.
* GQA: q-head h reads kv-head h // (Hq / Hkv); dK/dV of a kv-head sum over
  its q-heads.

Every function here is pinned by ``tests/test_oracle.py`` against brute
force, finite differences, closed forms and an independent library routine
(``torch.nn.functional.scaled_dot_product_attention`` in fp64 with autograd).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np

ROW_BLOCK = 256


def segment_offsets(P: int, R_lens: Sequence[int]) -> list:
    """off_0 = P, off_{i+1} = off_i + R_i: response i is packed rows [off_i, off_i + R_i)."""
    off = [int(P)]
    for r in R_lens:
        off.append(off[-1] + int(r))
    return off


def _row_blocks(L: int, split_at: int):
    """Row blocks of one sequence.  Blocks never straddle ``split_at`` (the
    prompt end), so the prompt rows are computed by the same arithmetic, on
    the same operands, in every replicated sequence."""
    for lo, hi in ((0, min(split_at, L)), (min(split_at, L), L)):
        for r0 in range(lo, hi, ROW_BLOCK):
            yield r0, min(r0 + ROW_BLOCK, hi)


def causal_attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                         split_at: int = 0):
    """Textbook causal softmax attention on one sequence, fp64.

    q, k, v: [L, d].  Returns o [L, d] and lse [L] with
    S = scale * q k^T, key j visible to row r iff j <= r,
    lse_r = log sum_{j<=r} exp(S_rj), o_r = sum_j exp(S_rj - lse_r) v_j.
    """
    L, d = q.shape
    o = np.zeros((L, v.shape[1]), dtype=np.float64)
    lse = np.zeros((L,), dtype=np.float64)
    for r0, r1 in _row_blocks(L, split_at):
        s = scale * (q[r0:r1] @ k[:r1].T)                       # [b, r1]
        rows = np.arange(r0, r1)[:, None]
        cols = np.arange(r1)[None, :]
        s = np.where(cols <= rows, s, -np.inf)
        m = s.max(axis=1)
        l = np.exp(s - m[:, None]).sum(axis=1)
        lse[r0:r1] = m + np.log(l)
        p = np.exp(s - lse[r0:r1, None])
        o[r0:r1] = p @ v[:r1]
    return o, lse


def causal_attention_bwd(q, k, v, o, lse, do, scale: float, split_at: int = 0):
    """Analytic backward of ``causal_attention_fwd`` on one sequence, fp64.

    With Pm = exp(S - lse): D_r = sum_c dO_rc O_rc, dV = Pm^T dO,
    dPm = dO V^T, dS = Pm * (dPm - D), dQ = scale dS K, dK = scale dS^T Q.
    """
    L, d = q.shape
    D = (do * o).sum(axis=1)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for r0, r1 in _row_blocks(L, split_at):
        s = scale * (q[r0:r1] @ k[:r1].T)
        rows = np.arange(r0, r1)[:, None]
        cols = np.arange(r1)[None, :]
        p = np.where(cols <= rows, np.exp(s - lse[r0:r1, None]), 0.0)
        dv[:r1] += p.T @ do[r0:r1]
        dp = do[r0:r1] @ v[:r1].T
        ds = p * (dp - D[r0:r1, None])
        dq[r0:r1] = scale * (ds @ k[:r1])
        dk[:r1] += scale * (ds.T @ q[r0:r1])
    return dq, dk, dv


def _check_shapes(q, k, v, P, R_lens):
    T, Hq, d = q.shape
    Tk, Hkv, dk_ = k.shape
    if v.shape != k.shape or Tk != T or dk_ != d:
        raise ValueError("q [T,Hq,d], k/v [T,Hkv,d] expected")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    off = segment_offsets(P, R_lens)
    if off[-1] != T:
        raise ValueError(f"P + sum(R) = {off[-1]} != T = {T}")
    if len(R_lens) < 1:
        raise ValueError("N >= 1 sequences")
    return T, Hq, Hkv, d, off


def _sequence_rows(P: int, off_i: int, R_i: int) -> np.ndarray:
    """Packed row indices of X_i = [prompt ; response_i]."""
    return np.concatenate([np.arange(P), np.arange(off_i, off_i + R_i)]).astype(np.int64)


def dualkv_forward(q, k, v, P: int, R_lens: Sequence[int], scale: float,
                   heads: Optional[Sequence[int]] = None):
    """Packed forward via replicated per-sequence attention.

    q [T,Hq,d], k/v [T,Hkv,d] float64.  Returns out [T,Hq,d] and lse [Hq,T]
    (rows of heads not in ``heads`` are left at zero).
    """
    T, Hq, Hkv, d, off = _check_shapes(q, k, v, P, R_lens)
    g = Hq // Hkv
    out = np.zeros((T, Hq, d), dtype=np.float64)
    lse = np.zeros((Hq, T), dtype=np.float64)
    for h in (range(Hq) if heads is None else heads):
        j = h // g
        for i, R_i in enumerate(R_lens):
            idx = _sequence_rows(P, off[i], R_i)
            o_i, lse_i = causal_attention_fwd(q[idx, h], k[idx, j], v[idx, j], scale, split_at=P)
            out[off[i]:off[i] + R_i, h] = o_i[P:]
            lse[h, off[i]:off[i] + R_i] = lse_i[P:]
            if i == 0:
                out[:P, h] = o_i[:P]
                lse[h, :P] = lse_i[:P]
            elif not (np.array_equal(out[:P, h], o_i[:P]) and np.array_equal(lse[h, :P], lse_i[:P])):
                raise AssertionError("prompt rows differ between replicated sequences")
    return out, lse


def dualkv_backward(q, k, v, dout, P: int, R_lens: Sequence[int], scale: float,
                    heads: Optional[Sequence[int]] = None,
                    prompt_dout_split: Optional[Sequence[np.ndarray]] = None):
    """Packed backward via replicated per-sequence attention.

    ``dout`` is the packed output gradient [T,Hq,d]; its prompt rows carry the
    gradient of the shared prompt rows.  By default sequence 0 receives them
    and the other sequences get zero; ``prompt_dout_split[i]`` ([P,Hq,d], with
    sum over i equal to dout[:P]) overrides that.  Prompt-row dQ/dK/dV are
    summed over the N sequences.  Returns dq [T,Hq,d], dk, dv [T,Hkv,d];
    with ``heads`` given, only those q-heads contribute.
    """
    T, Hq, Hkv, d, off = _check_shapes(q, k, v, P, R_lens)
    g = Hq // Hkv
    dq = np.zeros((T, Hq, d), dtype=np.float64)
    dk = np.zeros((T, Hkv, d), dtype=np.float64)
    dv = np.zeros((T, Hkv, d), dtype=np.float64)
    for h in (range(Hq) if heads is None else heads):
        j = h // g
        for i, R_i in enumerate(R_lens):
            idx = _sequence_rows(P, off[i], R_i)
            qi, ki, vi = q[idx, h], k[idx, j], v[idx, j]
            doi = dout[idx, h].copy()
            if prompt_dout_split is not None:
                doi[:P] = prompt_dout_split[i][:, h]
            elif i > 0:
                doi[:P] = 0.0
            o_i, lse_i = causal_attention_fwd(qi, ki, vi, scale, split_at=P)
            dq_i, dk_i, dv_i = causal_attention_bwd(qi, ki, vi, o_i, lse_i, doi, scale, split_at=P)
            dq[idx, h] += dq_i
            dk[idx, j] += dk_i
            dv[idx, j] += dv_i
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Several prompt groups in one packed batch (research-map page, "Limitations":
# one shared prefix per micro-batch group; "Key results" quotes a micro-batch
# size, mb=8, that may hold more than one prompt).  Group g occupies its own consecutive rows [prompt_g ; responses_g]
# and no row sees a key of another group, so each group is the single-group
# problem above on its own row range.
# ---------------------------------------------------------------------------

def group_row_starts(groups) -> list:
    """First packed row of each group and, last, the total row count.

    ``groups`` lists (P_g, R_lens_g) in row order."""
    starts = [0]
    for P_g, R_g in groups:
        starts.append(starts[-1] + int(P_g) + sum(int(r) for r in R_g))
    return starts


def dualkv_forward_groups(q, k, v, groups, scale: float, heads: Optional[Sequence[int]] = None):
    """Packed forward over several groups; a group without responses is its
    prompt alone under plain causal attention."""
    T, Hq, d = q.shape
    starts = group_row_starts(groups)
    if starts[-1] != T:
        raise ValueError("row count does not match the groups")
    g = Hq // k.shape[1]
    out = np.zeros((T, Hq, d), dtype=np.float64)
    lse = np.zeros((Hq, T), dtype=np.float64)
    for (P_g, R_g), a, b in zip(groups, starts[:-1], starts[1:]):
        if a == b:
            continue
        if len(R_g) == 0:
            for h in (range(Hq) if heads is None else heads):
                o_h, l_h = causal_attention_fwd(q[a:b, h], k[a:b, h // g], v[a:b, h // g], scale)
                out[a:b, h] = o_h
                lse[h, a:b] = l_h
            continue
        o_g, l_g = dualkv_forward(q[a:b], k[a:b], v[a:b], int(P_g), list(R_g), scale, heads=heads)
        out[a:b] = o_g
        lse[:, a:b] = l_g
    return out, lse


def dualkv_backward_groups(q, k, v, dout, groups, scale: float, heads: Optional[Sequence[int]] = None):
    """Packed backward over several groups (prompt-row gradients summed over
    the group's own responses only)."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    starts = group_row_starts(groups)
    if starts[-1] != T:
        raise ValueError("row count does not match the groups")
    g = Hq // Hkv
    dq = np.zeros((T, Hq, d), dtype=np.float64)
    dk = np.zeros((T, Hkv, d), dtype=np.float64)
    dv = np.zeros((T, Hkv, d), dtype=np.float64)
    for (P_g, R_g), a, b in zip(groups, starts[:-1], starts[1:]):
        if a == b:
            continue
        if len(R_g) == 0:
            for h in (range(Hq) if heads is None else heads):
                j = h // g
                o_h, l_h = causal_attention_fwd(q[a:b, h], k[a:b, j], v[a:b, j], scale)
                dq_h, dk_h, dv_h = causal_attention_bwd(q[a:b, h], k[a:b, j], v[a:b, j], o_h, l_h,
                                                        dout[a:b, h], scale)
                dq[a:b, h] += dq_h
                dk[a:b, j] += dk_h
                dv[a:b, j] += dv_h
            continue
        dq_g, dk_g, dv_g = dualkv_backward(q[a:b], k[a:b], v[a:b], dout[a:b], int(P_g), list(R_g), scale,
                                           heads=heads)
        dq[a:b] = dq_g
        dk[a:b] = dk_g
        dv[a:b] = dv_g
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Row-sampled oracle for full-size workloads.  The same definition, evaluated
# one query row at a time: row t of head h sees keys [0, t] if t is a prompt
# row, and [0, P) plus [off_i, t] if t is in response i.  Used where the
# replicated oracle would take hours; pinned against the functions above.
# ---------------------------------------------------------------------------

def _segment_of(t: int, off: list) -> int:
    """-1 for a prompt row, else the response index i with off_i <= t < off_{i+1}."""
    if t < off[0]:
        return -1
    return int(np.searchsorted(off, t, side="right")) - 1


def _visible_keys(t: int, P: int, off: list) -> np.ndarray:
    i = _segment_of(t, off)
    if i < 0:
        return np.arange(0, t + 1)
    return np.concatenate([np.arange(0, P), np.arange(off[i], t + 1)])


def rows_forward_backward(q, k, v, dout, P: int, R_lens: Sequence[int], scale: float,
                          heads: Sequence[int], rows: Sequence[int]):
    """O, LSE and dQ of the given query rows, one row at a time.

    Returns dict with ``o`` [len(heads), len(rows), d], ``lse`` [len(heads), len(rows)],
    ``dq`` like ``o``.  dO of a prompt row is the packed (summed) gradient.
    """
    T, Hq, Hkv, d, off = _check_shapes(q, k, v, P, R_lens)
    g = Hq // Hkv
    o = np.zeros((len(heads), len(rows), d))
    lse = np.zeros((len(heads), len(rows)))
    dq = np.zeros((len(heads), len(rows), d))
    for a, h in enumerate(heads):
        j = h // g
        for b, t in enumerate(rows):
            keys = _visible_keys(int(t), P, off)
            s = scale * (k[keys, j] @ q[t, h])
            m = s.max()
            lse_t = m + np.log(np.exp(s - m).sum())
            p = np.exp(s - lse_t)
            o_t = p @ v[keys, j]
            D_t = dout[t, h] @ o_t
            dp = v[keys, j] @ dout[t, h]
            ds = p * (dp - D_t)
            o[a, b] = o_t
            lse[a, b] = lse_t
            dq[a, b] = scale * (ds @ k[keys, j])
    return {"o": o, "lse": lse, "dq": dq}


def keys_dkdv(q, k, v, dout, P: int, R_lens: Sequence[int], scale: float,
              kv_head: int, keys: Sequence[int], row_block: int = 512):
    """dK and dV of the given key rows of one kv-head, summed over its q-heads
    and over every query row that sees them (both the prompt's own rows and all
    N responses for a prompt key; the own response's later rows for a response
    key).  Each query row's softmax is taken over its full visible key set.

    Returns dk, dv of shape [len(keys), d].
    """
    T, Hq, Hkv, d, off = _check_shapes(q, k, v, P, R_lens)
    g = Hq // Hkv
    keys = np.asarray(keys, dtype=np.int64)
    dk = np.zeros((len(keys), d))
    dv = np.zeros((len(keys), d))
    N = len(R_lens)
    prompt_keys = keys[keys < P]
    # Query row ranges (segment, first row, end row) that see at least one key.
    ranges = []
    if len(prompt_keys):
        ranges.append((-1, int(prompt_keys.min()), P))
        for i in range(N):
            ranges.append((i, off[i], off[i + 1]))
    else:
        for i in range(N):
            mine = keys[(keys >= off[i]) & (keys < off[i + 1])]
            if len(mine):
                ranges.append((i, int(mine.min()), off[i + 1]))
    for h in range(kv_head * g, kv_head * g + g):
        for seg, t_lo, t_hi in ranges:
            for t0 in range(t_lo, t_hi, row_block):
                t1 = min(t0 + row_block, t_hi)
                if seg < 0:
                    kidx = np.arange(0, t1)
                else:
                    kidx = np.concatenate([np.arange(0, P), np.arange(off[seg], t1)])
                kpos = kidx[None, :]
                rows = np.arange(t0, t1)[:, None]
                # key kidx visible to row t: prompt key (always, for a response row;
                # j <= t for a prompt row) or a response key with j <= t
                vis = (kpos <= rows) if seg < 0 else ((kpos < P) | (kpos <= rows))
                s = scale * (q[t0:t1, h] @ k[kidx, kv_head].T)
                s = np.where(vis, s, -np.inf)
                m = s.max(axis=1)
                lse_t = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
                p = np.where(vis, np.exp(s - lse_t[:, None]), 0.0)
                o_t = p @ v[kidx, kv_head]
                D_t = (dout[t0:t1, h] * o_t).sum(axis=1)
                # columns of the sampled keys inside kidx
                pos = np.searchsorted(kidx, keys)
                present = (pos < len(kidx)) & (kidx[np.minimum(pos, len(kidx) - 1)] == keys)
                if not present.any():
                    continue
                cols = pos[present]
                p_s = p[:, cols]                                   # [rows, ks]
                dp_s = dout[t0:t1, h] @ v[keys[present], kv_head].T
                ds_s = p_s * (dp_s - D_t[:, None])
                dv[present] += p_s.T @ dout[t0:t1, h]
                dk[present] += scale * (ds_s.T @ q[t0:t1, h])
    return dk, dv
