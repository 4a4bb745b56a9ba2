"""Seeded synthetic inputs and the named workload shapes.

This module holds no attention arithmetic.  It only draws random numbers and
describes shapes, so that the CUDA path, the tests, the benchmark and the CPU
oracle can all be fed the same bytes.

Recipe (stand-in for the RL micro-batches of the DualKV pages, "Experimental
setup" and "Key results" of the research-map page; their datasets are not used):

* ``torch.Generator('cpu').manual_seed(seed)``; q, k, v, dout drawn in that
  order with ``torch.randn`` in fp32 (N(0, 1)), then rounded to bf16 (RNE).
* Ragged response lengths come from ``numpy.random.default_rng(0)``,
  ``integers(512, 8193, size=16)`` (uniform on [512, 8192]).
* Packed token order: prompt rows ``[0, P)``, then response 1, ..., response N.
* Softmax scale ``1/sqrt(d)``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Sequence

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One packed micro-batch shape: a shared prompt of ``P`` tokens and
    ``N = len(R_lens)`` responses.  Heads are ``Hq`` query heads over ``Hkv``
    key/value heads (grouped-query attention), head size ``d``."""

    name: str
    Hq: int
    Hkv: int
    d: int
    P: int
    R_lens: tuple

    @property
    def N(self) -> int:
        return len(self.R_lens)

    @property
    def T(self) -> int:
        """Packed token count P + sum(R_i)."""
        return self.P + int(sum(self.R_lens))

    @property
    def T_replicated(self) -> int:
        """Token count of the replicated layout sum_i (P + R_i)."""
        return int(sum(self.P + r for r in self.R_lens))

    @property
    def offsets(self) -> List[int]:
        """off_0 = P, off_{i+1} = off_i + R_i; response i is rows [off_i, off_i + R_i)."""
        out = [self.P]
        for r in self.R_lens:
            out.append(out[-1] + int(r))
        return out

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def pairs_per_head(self) -> int:
        """Unmasked (query, key) pairs of one head on the packed layout."""
        P = self.P
        n = P * (P + 1) // 2
        for r in self.R_lens:
            n += r * P + r * (r + 1) // 2
        return n

    def pairs_per_head_replicated(self) -> int:
        return sum((self.P + r) * (self.P + r + 1) // 2 for r in self.R_lens)

    def useful_flops(self, fwd: bool = True, bwd: bool = True) -> float:
        """Useful tensor flops on the packed layout: 4d per pair forward
        (QK^T and PV), 10d per pair backward (five products)."""
        per = (4 if fwd else 0) + (10 if bwd else 0)
        return float(per) * self.d * self.Hq * self.pairs_per_head()

    def rho_tokens(self) -> float:
        """rho = N(P+R)/(P+NR), the token compression factor."""
        return self.T_replicated / self.T

    def rho_pairs(self) -> float:
        return self.pairs_per_head_replicated() / self.pairs_per_head()

    def replicated(self) -> "Workload":
        """The same micro-batch on the replicated layout: no shared prompt,
        N independent causal sequences of P + R_i tokens."""
        return Workload(self.name + "-replicated", self.Hq, self.Hkv, self.d, 0,
                        tuple(self.P + int(r) for r in self.R_lens))


def ragged_lengths(n: int = 16, lo: int = 512, hi: int = 8192, seed: int = 0) -> tuple:
    return tuple(int(x) for x in np.random.default_rng(seed).integers(lo, hi + 1, size=n))


WORKLOADS = {
    "tiny": Workload("tiny", 2, 1, 64, 128, (64,) * 4),
    "qwen3_8b": Workload("qwen3_8b", 32, 8, 128, 4096, (4096,) * 32),
    "p32k": Workload("p32k", 32, 8, 128, 32768, (2048,) * 16),
    "ragged_30b_a3b": Workload("ragged_30b_a3b", 32, 4, 128, 8192, ragged_lengths()),
    "edge_p64k": Workload("edge_p64k", 32, 8, 128, 65536, (1024,) * 16),
    "edge_n4": Workload("edge_n4", 32, 8, 128, 8192, (8192,) * 4),
}


def make_workload(name: str, Hq: int, Hkv: int, d: int, P: int, R_lens: Sequence[int]) -> Workload:
    return Workload(name, int(Hq), int(Hkv), int(d), int(P), tuple(int(r) for r in R_lens))


@dataclasses.dataclass
class Inputs:
    """bf16 CPU tensors in the packed layout: q, dout [T, Hq, d]; k, v [T, Hkv, d]."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dout: torch.Tensor


def draw_inputs(T: int, Hq: int, Hkv: int, d: int, seed: int = 0) -> Inputs:
    """q, k, v, dout of T packed rows, drawn in that order from one seeded stream."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((T, Hq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn((T, Hkv, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((T, Hkv, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    dout = torch.randn((T, Hq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return Inputs(q, k, v, dout)


def make_inputs(w: Workload, seed: int = 0) -> Inputs:
    return draw_inputs(w.T, w.Hq, w.Hkv, w.d, seed)


def group_rows(groups) -> int:
    """Packed rows of several prompt groups [(P_g, R_lens_g), ...]."""
    return int(sum(int(p) + sum(int(r) for r in rs) for p, rs in groups))


def make_group_inputs(groups, Hq: int, Hkv: int, d: int, seed: int = 0) -> Inputs:
    """Inputs of a batch of several prompt groups laid out one after another."""
    return draw_inputs(group_rows(groups), Hq, Hkv, d, seed)


def to_f64(x: torch.Tensor) -> np.ndarray:
    """Exact upcast of a bf16 tensor to a float64 numpy array."""
    return x.detach().to("cpu").to(torch.float64).numpy()


# Decoder-layer shapes: Qwen3-8B (the pages' main model; research-map page,
# "Experimental setup") and a small one the fp64 oracle finishes in seconds.
LAYER_SHAPES = {
    "qwen3_8b": dict(hidden=4096, Hq=32, Hkv=8, d=128, inter=12288, rope_base=1.0e6, eps=1.0e-6),
    "small": dict(hidden=256, Hq=4, Hkv=2, d=64, inter=512, rope_base=1.0e4, eps=1.0e-6),
    "small_d128": dict(hidden=512, Hq=4, Hkv=1, d=128, inter=256, rope_base=1.0e6, eps=1.0e-6),
    "wide": dict(hidden=6144, Hq=2, Hkv=1, d=64, inter=256, rope_base=1.0e4, eps=1.0e-5),
}


def make_layer_inputs(shape: dict, T: int, seed: int = 0):
    """Random-init weights (bf16) and packed activations x, dy [T, hidden] (bf16).

    Norm weights are 1 + 0.1 N(0,1); projection weights N(0,1)/sqrt(fan_in);
    x and dy N(0,1).  Drawn in the order ln1, wqkv, wo, ln2, wgu, wd, x, dy
    from one seeded CPU generator."""
    g = torch.Generator("cpu").manual_seed(seed)
    H, I = shape["hidden"], shape["inter"]
    nq, nk = shape["Hq"] * shape["d"], shape["Hkv"] * shape["d"]
    shapes = {"ln1": (H,), "wqkv": (nq + 2 * nk, H), "wo": (H, nq), "ln2": (H,), "wgu": (2 * I, H), "wd": (H, I)}
    w = {}
    for n, sh in shapes.items():
        r = torch.randn(sh, generator=g, dtype=torch.float32)
        w[n] = (1.0 + 0.1 * r if n.startswith("ln") else r / math.sqrt(sh[1])).to(torch.bfloat16)
    x = torch.randn((T, H), generator=g, dtype=torch.float32).to(torch.bfloat16)
    dy = torch.randn((T, H), generator=g, dtype=torch.float32).to(torch.bfloat16)
    return w, x, dy
