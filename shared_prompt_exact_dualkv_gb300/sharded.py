"""DualKV attention across ranks (one process per GPU): two partitions.

The pages compare DualKV with sequence parallelism (research-map page, "Key
results") but describe no sharded DualKV; the two splits below are the
plainest ones that keep the result exact.

Kv-head split (``head_bounds``, ``heads_forward``, ``heads_backward``).
    Heads are independent: rank r takes kv-heads [lo, hi) and the q-heads that
    read them, on every packed row.  No exchange at all; the caller holds the
    outputs of its own heads (``gather_heads`` assembles them where a test or
    a caller wants every head).

Sequence split (``shard_bounds``, ``prompt_bounds``, ``sharded_forward``,
``sharded_backward``).  The N responses of a prompt group are cut into
contiguous chunks, one per rank.  Every rank holds the whole prompt and its
own responses, packed as [prompt ; its responses].
    * The prompt's own causal attention is divided too: rank r takes the
      prompt query rows ``prompt_bounds(P, world, r)`` (tile-aligned, equal
      causal work) through the library's partial entry points; the other
      ranks' prompt rows of out/lse arrive in one exchange (a sum of
      zero-filled buffers).  Response rows need only the prompt's keys and
      values, which every rank holds.
    * Backward: the packed dO of a prompt row is the sum of the ranks' shares
      (the gradient that reaches the shared row through each rank's
      sequences), so the shares are summed in fp32 and rounded once.  Each
      rank then runs the backward on its prompt rows and responses and keeps
      the prompt rows' dQ/dK/dV in fp32, unrounded; one fp32 all-reduce sums
      them (research-map page, "Approach": the shared prompt's gradients are
      accumulated across sequences in fp32) and they are rounded to bf16 once.
      Response rows need no exchange.
    ``prompt_rows=(0, P)`` on every rank keeps the prompt work on every rank
    instead (no out/dO exchange; the prompt gradients are still summed in fp32).

Bytes exchanged per layer, sequence split: 4*P*Hq*(d+1) forward (prompt
out and lse as fp32); 4*P*Hq*d (dO shares) + 4*P*(Hq + 2*Hkv)*d backward.

The compute calls are injectable (``fwd_fn`` / ``bwd_fn``), so that the
bookkeeping and the exchanges can be tested on CPU ranks with a stand-in.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence, Tuple

import torch
import torch.distributed as dist

TILE = 128


def shard_bounds(N: int, world: int, rank: int) -> Tuple[int, int]:
    """Responses [lo, hi) of ``rank``: contiguous chunks, sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    return (rank * N) // world, ((rank + 1) * N) // world


def prompt_bounds(P: int, world: int, rank: int) -> Tuple[int, int]:
    """Prompt query rows [lo, hi) of ``rank``: 128-row tiles, contiguous, cut
    where the prompt's causal work (tile t walks t + 1 key tiles) is split
    evenly; the last rank's end is P."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    n = (P + TILE - 1) // TILE
    total = n * (n + 1) // 2

    def cut(r):
        if r >= world:
            return n
        goal = r * total / world
        t = 0
        while t < n and t * (t + 1) / 2 < goal:
            t += 1
        return t

    lo, hi = cut(rank), cut(rank + 1)
    return min(lo * TILE, P), min(hi * TILE, P)


def head_bounds(Hkv: int, world: int, rank: int) -> Tuple[int, int]:
    """Kv-heads [lo, hi) of ``rank``: contiguous, sizes differ by at most one."""
    return shard_bounds(Hkv, world, rank)


def local_rows(P: int, R_lens: Sequence[int], lo: int, hi: int) -> torch.Tensor:
    """Packed row indices of the local batch [prompt ; responses lo..hi-1]."""
    off = P + sum(int(r) for r in R_lens[:lo])
    idx = [torch.arange(P)]
    for r in R_lens[lo:hi]:
        idx.append(torch.arange(off, off + int(r)))
        off += int(r)
    return torch.cat(idx).long()


def _active():
    return dist.is_available() and dist.is_initialized()


def _sum_f32(t: torch.Tensor, group) -> torch.Tensor:
    """fp32 all-reduce (sum) of ``t`` over ``group`` (identity on one rank)."""
    t = t.float().contiguous()
    if _active():
        dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return t


# --------------------------------------------------------------------------- library calls

def _library_fwd(q, k, v, P, R_local, scale, prompt_rows):
    from shared_prompt_exact_dualkv_gb300 import dualkv
    out = torch.zeros_like(q)
    lse = torch.zeros((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    dualkv.dualkv_fwd_partial(q, k, v, P, R_local, prompt_rows, out, lse, scale)
    return out, lse


def _library_bwd(q, k, v, out, dout, lse, P, R_local, scale, prompt_rows, deterministic=False):
    """Backward of the local batch; returns bf16 dq, dk, dv and the fp32
    prompt rows dq_p [P,Hq,d] (zero outside prompt_rows), dk_p, dv_p [P,Hkv,d]."""
    from shared_prompt_exact_dualkv_gb300 import dualkv
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    nbytes = dualkv.dualkv_bwd_workspace_bytes(P, R_local, Hq, Hkv, d, deterministic)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.zeros_like(q), torch.empty_like(k), torch.empty_like(v)
    dq_p = torch.zeros((P, Hq, d), dtype=torch.float32, device=q.device)
    dk_p = torch.empty((P, Hkv, d), dtype=torch.float32, device=q.device)
    dv_p = torch.empty((P, Hkv, d), dtype=torch.float32, device=q.device)
    dualkv.dualkv_bwd_partial(q, k, v, out, dout, lse, P, R_local, prompt_rows, scale, deterministic, ws, dq, dk, dv,
                              dq_p if P else None, dk_p if P else None, dv_p if P else None)
    return dq, dk, dv, dq_p, dk_p, dv_p


# --------------------------------------------------------------------------- sequence split

def sharded_forward(q, k, v, P: int, R_local: Sequence[int], scale: float, prompt_rows=None,
                    group: Optional[dist.ProcessGroup] = None, fwd_fn: Optional[Callable] = None):
    """Forward of the local batch [prompt ; local responses].

    ``prompt_rows`` = (lo, hi): the prompt query rows this rank computes
    (``prompt_bounds``); the other prompt rows of out and lse are filled in
    from the ranks that computed them.  None computes every prompt row here."""
    R_local = list(R_local) if len(R_local) else [0]
    lo, hi = (0, P) if prompt_rows is None else prompt_rows
    out, lse = (fwd_fn or _library_fwd)(q, k, v, P, R_local, scale, (lo, hi))
    if prompt_rows is not None and P > 0:
        po = torch.zeros((P,) + tuple(out.shape[1:]), dtype=torch.float32, device=out.device)
        pl = torch.zeros((lse.shape[0], P), dtype=torch.float32, device=lse.device)
        po[lo:hi] = out[lo:hi].float()
        pl[:, lo:hi] = lse[:, lo:hi].float()
        po, pl = _sum_f32(po, group), _sum_f32(pl, group)       # exact: one rank is non-zero per row
        out[:P] = po.to(out.dtype)
        lse[:, :P] = pl.to(lse.dtype)
    return out, lse


def sharded_backward(q, k, v, out, dout, lse, P: int, R_local: Sequence[int], scale: float, prompt_rows=None,
                     group: Optional[dist.ProcessGroup] = None, bwd_fn: Optional[Callable] = None,
                     deterministic: bool = False):
    """Backward of the local batch, then the fp32 sum of the prompt rows of
    dQ, dK and dV over the ranks of ``group``, rounded to bf16 once.

    ``dout`` holds, on its prompt rows, this rank's share of the prompt
    gradient (the gradient that reaches the shared prompt rows through this
    rank's sequences); the shares of all ranks add up to the packed dO.  With
    ``prompt_rows`` given, the shares are summed first (fp32, rounded once)
    and this rank takes the prompt query rows [lo, hi) with the whole dO."""
    R_local = list(R_local) if len(R_local) else [0]
    if prompt_rows is None:
        lo, hi = 0, P
    else:
        lo, hi = prompt_rows
        if P > 0:
            dout = dout.clone()
            dout[:P] = _sum_f32(dout[:P], group).to(dout.dtype)
    dq, dk, dv, dq_p, dk_p, dv_p = (bwd_fn or _library_bwd)(q, k, v, out, dout, lse, P, R_local, scale, (lo, hi),
                                                            deterministic)
    if P > 0:
        nq, nk = dq_p.numel(), dk_p.numel()
        flat = _sum_f32(torch.cat([dq_p.reshape(-1), dk_p.reshape(-1), dv_p.reshape(-1)]), group)
        dq[:P] = flat[:nq].view_as(dq_p).to(dq.dtype)
        dk[:P] = flat[nq:nq + nk].view_as(dk_p).to(dk.dtype)
        dv[:P] = flat[nq + nk:].view_as(dv_p).to(dv.dtype)
    return dq, dk, dv


# --------------------------------------------------------------------------- kv-head split

def _head_slice(t: torch.Tensor, lo: int, hi: int) -> torch.Tensor:
    return t[:, lo:hi].contiguous()


def heads_forward(q, k, v, P: int, R_lens: Sequence[int], scale: float, kv_heads: Tuple[int, int],
                  fwd_fn: Optional[Callable] = None):
    """Forward of kv-heads [lo, hi) and their q-heads on every packed row.
    Returns out [T, g*(hi-lo), d] and lse [g*(hi-lo), T] of those q-heads."""
    g = q.shape[1] // k.shape[1]
    lo, hi = kv_heads
    ql, kl, vl = _head_slice(q, lo * g, hi * g), _head_slice(k, lo, hi), _head_slice(v, lo, hi)
    if fwd_fn is not None:
        return fwd_fn(ql, kl, vl, P, list(R_lens), scale, (0, P))
    from shared_prompt_exact_dualkv_gb300 import dualkv
    return dualkv.forward(ql, kl, vl, P, list(R_lens), scale)


def heads_backward(q, k, v, out_local, dout, lse_local, P: int, R_lens: Sequence[int], scale: float,
                   kv_heads: Tuple[int, int], bwd_fn: Optional[Callable] = None, deterministic: bool = False):
    """Backward of kv-heads [lo, hi): ``out_local``/``lse_local`` come from
    ``heads_forward``; ``dout`` is the full [T, Hq, d] output gradient.
    Returns dq [T, g*(hi-lo), d] and dk, dv [T, hi-lo, d]: final values, no exchange."""
    g = q.shape[1] // k.shape[1]
    lo, hi = kv_heads
    ql, kl, vl = _head_slice(q, lo * g, hi * g), _head_slice(k, lo, hi), _head_slice(v, lo, hi)
    dol = _head_slice(dout, lo * g, hi * g)
    if bwd_fn is not None:
        return bwd_fn(ql, kl, vl, out_local, dol, lse_local, P, list(R_lens), scale, (0, P), deterministic)[:3]
    from shared_prompt_exact_dualkv_gb300 import dualkv
    return dualkv.backward(ql, kl, vl, out_local, dol, lse_local, P, list(R_lens), scale, deterministic=deterministic)


def gather_heads(local: torch.Tensor, total_heads: int, head_lo: int, dim: int,
                 group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """Every rank's heads in one tensor: each rank places its slice (heads
    [head_lo, head_lo + local.shape[dim])) in a zero tensor, and the ranks'
    tensors are summed in fp32 (exact: one rank is non-zero per head)."""
    shape = list(local.shape)
    shape[dim] = total_heads
    full = torch.zeros(shape, dtype=torch.float32, device=local.device)
    full.narrow(dim, head_lo, local.shape[dim]).copy_(local.float())
    return _sum_f32(full, group).to(local.dtype)
