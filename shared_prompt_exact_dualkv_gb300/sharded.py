"""Sequence-sharded DualKV attention across ranks (one process per GPU).

The N responses of a prompt group are split into contiguous chunks, one per
rank.  Every rank holds the whole prompt and its own responses, packed as
[prompt ; its responses], and runs the library's forward and backward on that
local batch.

* Forward: no exchange.  A prompt row only sees prompt keys, so every rank
  computes the same prompt outputs; response rows are local.
* Backward: the prompt's dQ, dK and dV are sums over all N sequences
  (research-map page, "Approach": the shared prompt's gradients are
  accumulated across sequences).  The backward is linear in dO.  So each rank
  runs it with the prompt rows' dO equal to its own sequences' share of the
  prompt gradient, and the ranks' prompt-row dQ/dK/dV are summed with one
  all-reduce.  The all-reduce runs in fp32, on the prompt rows only.  Response
  rows need no exchange.

Only the prompt rows cross ranks: 4*P*(Hq + 2*Hkv)*d bytes per layer.  The
pages compare against sequence parallelism (research-map page, "Key results")
but do not describe a sharded DualKV; this split is the plainest one that
keeps the result exact.

The compute calls are injectable (``fwd_fn`` / ``bwd_fn``), so that the
bookkeeping and the exchange can be tested on CPU ranks with a stand-in.
"""
from __future__ import annotations

from typing import Callable, Optional, Sequence, Tuple

import torch
import torch.distributed as dist


def shard_bounds(N: int, world: int, rank: int) -> Tuple[int, int]:
    """Responses [lo, hi) of ``rank``: contiguous chunks, sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    return (rank * N) // world, ((rank + 1) * N) // world


def local_rows(P: int, R_lens: Sequence[int], lo: int, hi: int) -> torch.Tensor:
    """Packed row indices of the local batch [prompt ; responses lo..hi-1]."""
    off = P + sum(int(r) for r in R_lens[:lo])
    idx = [torch.arange(P)]
    for r in R_lens[lo:hi]:
        idx.append(torch.arange(off, off + int(r)))
        off += int(r)
    return torch.cat(idx).long()


def _library_fwd(q, k, v, P, R_local, scale):
    from shared_prompt_exact_dualkv_gb300 import dualkv
    return dualkv.forward(q, k, v, P, R_local, scale)


def _library_bwd(q, k, v, out, dout, lse, P, R_local, scale):
    from shared_prompt_exact_dualkv_gb300 import dualkv
    return dualkv.backward(q, k, v, out, dout, lse, P, R_local, scale)


def sharded_forward(q, k, v, P: int, R_local: Sequence[int], scale: float,
                    fwd_fn: Optional[Callable] = None):
    """Forward of the local batch (prompt rows are computed on every rank)."""
    R_local = list(R_local) if len(R_local) else [0]
    return (fwd_fn or _library_fwd)(q, k, v, P, R_local, scale)


def sharded_backward(q, k, v, out, dout, lse, P: int, R_local: Sequence[int], scale: float,
                     group: Optional[dist.ProcessGroup] = None, bwd_fn: Optional[Callable] = None):
    """Backward of the local batch, then the sum of the prompt rows of dQ,
    dK and dV over the ranks of ``group``.

    ``dout`` holds, on its prompt rows, this rank's share of the prompt
    gradient (the gradient that reaches the shared prompt rows through this
    rank's sequences); the shares of all ranks add up to the packed dO."""
    R_local = list(R_local) if len(R_local) else [0]
    dq, dk, dv = (bwd_fn or _library_bwd)(q, k, v, out, dout, lse, P, R_local, scale)
    if P > 0 and dist.is_available() and dist.is_initialized():
        flat = torch.cat([dq[:P].reshape(-1), dk[:P].reshape(-1), dv[:P].reshape(-1)]).float()
        dist.all_reduce(flat, op=dist.ReduceOp.SUM, group=group)
        nq, nk = dq[:P].numel(), dk[:P].numel()
        dq[:P] = flat[:nq].view_as(dq[:P]).to(dq.dtype)
        dk[:P] = flat[nq:nq + nk].view_as(dk[:P]).to(dk.dtype)
        dv[:P] = flat[nq + nk:].view_as(dv[:P]).to(dv.dtype)
    return dq, dk, dv
