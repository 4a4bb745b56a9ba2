"""fp64 CPU oracle of one decoder layer run on the packed (P + NR) layout.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/`` and ``bench.py``'s CPU legs use it.  It shares no code with
the CUDA library.

What it computes ("DualKV: Shared-Prompt Flash Attention for Efficient RL
Training with Large Rollouts and Long Contexts" -- arXiv abstract page: the
repacking into P + NR tokens "extends the token reduction from attention to the
entire model", because causal masking keeps the prompt's hidden states the same
in every sequence at every layer; forum page, "Two changes", change 2):

* Every replicated sequence X_i = [prompt ; response_i] runs through a
  textbook pre-norm decoder layer with positions 0 .. P+R_i-1:

      h1 = RMSNorm(x) * ln1
      q, k, v = split(h1 @ Wqkv^T),   q, k rotated by RoPE at the positions
      a  = causal softmax attention (GQA)
      x2 = x + a @ Wo^T
      h2 = RMSNorm(x2) * ln2
      g, u = split(h2 @ Wgu^T)
      y  = x2 + (silu(g) * u) @ Wd^T

  The layer follows the Qwen3 family the pages train (Qwen3-8B, research-map
  page, "Experimental setup") minus its per-head q/k RMSNorm, which acts on
  each token alone and so changes nothing about which rows are shared.
* The packed result takes response rows from their own sequence and prompt
  rows from sequence 0 (after checking that every sequence produced the same
  values, to 1e-12: BLAS may block sequences of different lengths differently).  In the backward pass the packed dy of a prompt row is the gradient of
  the one shared row; it is handed to sequence 0 (gradients are linear in dy),
  and prompt-row dx and every weight gradient are summed over the sequences.

Conventions (standard for this model family; the pages do not state them):
RMSNorm r = 1/sqrt(mean(x^2) + eps); RoPE in the rotate-half form with
angle pos * base^(-2i/d) for the feature pair (i, i + d/2); silu(g) = g/(1+e^-g);
Wgu holds the gate rows first, then the up rows.

Pinned by ``tests/test_layer_oracle.py``: torch fp64 autograd of the layer
built from library routines (linear, rms_norm, scaled_dot_product_attention,
silu), RoPE as complex multiplication, RoPE and RMSNorm invariants, finite
differences, and planted mistakes.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Sequence

import numpy as np

from oracle import attention as att


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    hidden: int
    Hq: int
    Hkv: int
    d: int
    inter: int
    rope_base: float = 1.0e6
    eps: float = 1.0e-6


WEIGHT_NAMES = ("ln1", "wqkv", "wo", "ln2", "wgu", "wd")


def weight_shapes(c: LayerConfig) -> Dict[str, tuple]:
    return {"ln1": (c.hidden,), "wqkv": ((c.Hq + 2 * c.Hkv) * c.d, c.hidden), "wo": (c.hidden, c.Hq * c.d),
            "ln2": (c.hidden,), "wgu": (2 * c.inter, c.hidden), "wd": (c.hidden, c.inter)}


# --------------------------------------------------------------------------- ops

def rms_norm(x, w, eps):
    """y = x * r * w with r = 1/sqrt(mean(x^2) + eps) per row; returns (y, r)."""
    r = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    return x * r * w, r


def rms_norm_bwd(dy, x, r, w):
    """dx = r*(w*dy) - (r^3/H) * x * sum(w*dy*x);  dw = sum over rows of dy*x*r."""
    H = x.shape[-1]
    gw = dy * w
    dx = r * gw - (r ** 3 / H) * x * (gw * x).sum(axis=-1, keepdims=True)
    dw = (dy * x * r).sum(axis=0)
    return dx, dw


def rope_angles(pos, d, base):
    """[L, d/2] angles pos * base^(-2i/d)."""
    i = np.arange(d // 2, dtype=np.float64)
    inv = base ** (-2.0 * i / d)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]


def rope(x, ang):
    """Rotate the pair (x_i, x_{i+d/2}) of every head by the row's angle i.
    x [L, H, d], ang [L, d/2]."""
    h = x.shape[-1] // 2
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rope_bwd(dy, ang):
    """Transpose of ``rope``: rotation by the negative angle."""
    return rope(dy, -ang)


def silu(g):
    return g / (1.0 + np.exp(-g))


def swiglu_bwd(dm, g, u):
    sg = 1.0 / (1.0 + np.exp(-g))
    dg = dm * u * sg * (1.0 + g * (1.0 - sg))
    du = dm * g * sg
    return dg, du


# --------------------------------------------------------------------------- one sequence

def sequence_forward(x, W, c: LayerConfig):
    """The layer on one causal sequence x [L, hidden] with positions 0..L-1.
    Returns y and the saved intermediates."""
    L = x.shape[0]
    g = c.Hq // c.Hkv
    h1, r1 = rms_norm(x, W["ln1"], c.eps)
    qkv = h1 @ W["wqkv"].T
    nq, nk = c.Hq * c.d, c.Hkv * c.d
    ang = rope_angles(np.arange(L), c.d, c.rope_base)
    q = rope(qkv[:, :nq].reshape(L, c.Hq, c.d), ang)
    k = rope(qkv[:, nq:nq + nk].reshape(L, c.Hkv, c.d), ang)
    v = qkv[:, nq + nk:].reshape(L, c.Hkv, c.d)
    scale = c.d ** -0.5
    a = np.zeros((L, c.Hq, c.d))
    lse = np.zeros((c.Hq, L))
    for h in range(c.Hq):
        a[:, h], lse[h] = att.causal_attention_fwd(q[:, h], k[:, h // g], v[:, h // g], scale)
    af = a.reshape(L, nq)
    x2 = x + af @ W["wo"].T
    h2, r2 = rms_norm(x2, W["ln2"], c.eps)
    gu = h2 @ W["wgu"].T
    gt, up = gu[:, :c.inter], gu[:, c.inter:]
    m = silu(gt) * up
    y = x2 + m @ W["wd"].T
    saved = dict(x=x, h1=h1, r1=r1, q=q, k=k, v=v, ang=ang, a=a, lse=lse, af=af, x2=x2, h2=h2, r2=r2,
                 gt=gt, up=up, m=m)
    return y, saved


def sequence_backward(dy, W, c: LayerConfig, s):
    """Analytic backward of ``sequence_forward``; returns dx and the weight grads."""
    L = dy.shape[0]
    g = c.Hq // c.Hkv
    nq = c.Hq * c.d
    grads = {}
    dm = dy @ W["wd"]
    grads["wd"] = dy.T @ s["m"]
    dgt, dup = swiglu_bwd(dm, s["gt"], s["up"])
    dgu = np.concatenate([dgt, dup], axis=1)
    grads["wgu"] = dgu.T @ s["h2"]
    dh2 = dgu @ W["wgu"]
    dn2, grads["ln2"] = rms_norm_bwd(dh2, s["x2"], s["r2"], W["ln2"])
    dx2 = dy + dn2
    grads["wo"] = dx2.T @ s["af"]
    da = (dx2 @ W["wo"]).reshape(L, c.Hq, c.d)
    scale = c.d ** -0.5
    dq = np.zeros_like(s["q"])
    dk = np.zeros_like(s["k"])
    dv = np.zeros_like(s["v"])
    for h in range(c.Hq):
        j = h // g
        dq_h, dk_h, dv_h = att.causal_attention_bwd(s["q"][:, h], s["k"][:, j], s["v"][:, j], s["a"][:, h],
                                                    s["lse"][h], da[:, h], scale)
        dq[:, h] = dq_h
        dk[:, j] += dk_h
        dv[:, j] += dv_h
    dqkv = np.concatenate([rope_bwd(dq, s["ang"]).reshape(L, -1), rope_bwd(dk, s["ang"]).reshape(L, -1),
                           dv.reshape(L, -1)], axis=1)
    grads["wqkv"] = dqkv.T @ s["h1"]
    dh1 = dqkv @ W["wqkv"]
    dn1, grads["ln1"] = rms_norm_bwd(dh1, s["x"], s["r1"], W["ln1"])
    return dx2 + dn1, grads


# --------------------------------------------------------------------------- packed groups

def _sequences(groups):
    """(group start, prompt length, response start, response length) per
    replicated sequence; a group without responses is its prompt alone."""
    out = []
    a = 0
    for P_g, R_g in groups:
        P_g = int(P_g)
        off = a + P_g
        if len(R_g) == 0:
            out.append((a, P_g, off, 0))
        for r in R_g:
            out.append((a, P_g, off, int(r)))
            off += int(r)
        a = off
    return out


def _rows(a, P_g, off, R):
    return np.concatenate([np.arange(a, a + P_g), np.arange(off, off + R)]).astype(np.int64)


def packed_forward(x, groups, W, c: LayerConfig):
    """y [T, hidden] of the packed batch via the replicated sequences."""
    y = np.zeros_like(x)
    filled = {}
    for a, P_g, off, R in _sequences(groups):
        idx = _rows(a, P_g, off, R)
        y_i, _ = sequence_forward(x[idx], W, c)
        y[off:off + R] = y_i[P_g:]
        if a not in filled:
            y[a:a + P_g] = y_i[:P_g]
            filled[a] = True
        elif not np.allclose(y[a:a + P_g], y_i[:P_g], rtol=0.0, atol=1e-12):
            # equal up to the BLAS blocking of sequences of different lengths
            raise AssertionError("prompt rows differ between replicated sequences")
    return y


def packed_backward(x, dy, groups, W, c: LayerConfig):
    """dx [T, hidden] and weight grads of the packed batch.  The prompt rows'
    dy goes to each group's first sequence; prompt dx and all weight grads
    are summed over the sequences."""
    dx = np.zeros_like(x)
    grads = {n: np.zeros(sh) for n, sh in weight_shapes(c).items()}
    first = set()
    for a, P_g, off, R in _sequences(groups):
        idx = _rows(a, P_g, off, R)
        dy_i = dy[idx].copy()
        if a in first:
            dy_i[:P_g] = 0.0
        first.add(a)
        _, saved = sequence_forward(x[idx], W, c)
        dx_i, g_i = sequence_backward(dy_i, W, c, saved)
        dx[off:off + R] = dx_i[P_g:]
        dx[a:a + P_g] += dx_i[:P_g]
        for n in grads:
            grads[n] += g_i[n]
    return dx, grads


def packed_positions(groups) -> np.ndarray:
    """Position id of every packed row: prompt rows 0..P_g-1, and response
    rows P_g .. P_g + R - 1 (each response continues its group's prompt)."""
    pos = []
    for P_g, R_g in groups:
        pos += list(range(int(P_g)))
        for r in R_g:
            pos += list(range(int(P_g), int(P_g) + int(r)))
    return np.asarray(pos, dtype=np.int64)
