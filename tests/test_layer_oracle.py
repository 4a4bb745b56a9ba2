"""Pins for the fp64 decoder-layer oracle (CPU only).

The oracle's analytic forward and backward are tied to torch fp64 autograd
of the same layer built from library routines (``linear``, ``rms_norm``,
``scaled_dot_product_attention``, ``silu``).  RoPE there is written as a
complex multiplication, a different computation from the oracle's rotation.
The packed result is tied to a formulation that never replicates anything:
the layer over the whole packed batch with a dense attention mask and the
packed position ids.  Finite differences, closed forms, RoPE invariants
and planted mistakes complete the pins."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import layer as L
from tests.test_oracle import group_mask

CFG = L.LayerConfig(hidden=32, Hq=4, Hkv=2, d=8, inter=48, rope_base=1.0e4, eps=1e-6)


def rand_weights(c, seed=0):
    rng = np.random.default_rng(seed)
    W = {}
    for n, sh in L.weight_shapes(c).items():
        if n.startswith("ln"):
            W[n] = 1.0 + 0.1 * rng.standard_normal(sh)
        else:
            W[n] = rng.standard_normal(sh) / math.sqrt(sh[1])
    return W


def torch_layer(x, W, c, pos, mask):
    """fp64 torch layer on rows x [T, hidden] with positions ``pos`` and a
    boolean attention mask [T, T] (True = visible); autograd-ready."""
    T = x.shape[0]
    nq, nk = c.Hq * c.d, c.Hkv * c.d
    h1 = F.rms_norm(x, (c.hidden,), weight=W["ln1"], eps=c.eps)
    qkv = F.linear(h1, W["wqkv"])
    inv = c.rope_base ** (-2.0 * torch.arange(c.d // 2, dtype=torch.float64) / c.d)
    rot = torch.polar(torch.ones(T, c.d // 2, dtype=torch.float64), pos[:, None] * inv[None, :])

    def rope_c(t, H):
        t = t.reshape(T, H, c.d)
        z = torch.complex(t[..., : c.d // 2], t[..., c.d // 2:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    q = rope_c(qkv[:, :nq], c.Hq)
    k = rope_c(qkv[:, nq:nq + nk], c.Hkv)
    v = qkv[:, nq + nk:].reshape(T, c.Hkv, c.d)
    g = c.Hq // c.Hkv
    qh = q.permute(1, 0, 2)
    kh = k.repeat_interleave(g, dim=1).permute(1, 0, 2)
    vh = v.repeat_interleave(g, dim=1).permute(1, 0, 2)
    a = F.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask, scale=c.d ** -0.5)
    x2 = x + F.linear(a.permute(1, 0, 2).reshape(T, nq), W["wo"])
    h2 = F.rms_norm(x2, (c.hidden,), weight=W["ln2"], eps=c.eps)
    gu = F.linear(h2, W["wgu"])
    return x2 + F.linear(F.silu(gu[:, :c.inter]) * gu[:, c.inter:], W["wd"])


def torch_grads(x, dy, W, c, pos, mask):
    xt = torch.tensor(x, requires_grad=True)
    Wt = {n: torch.tensor(w, requires_grad=True) for n, w in W.items()}
    y = torch_layer(xt, Wt, c, torch.tensor(pos, dtype=torch.float64), torch.tensor(mask))
    (y * torch.tensor(dy)).sum().backward()
    return y.detach().numpy(), xt.grad.numpy(), {n: t.grad.numpy() for n, t in Wt.items()}


def test_sequence_layer_against_torch_autograd():
    Lseq = 11
    rng = np.random.default_rng(1)
    x = rng.standard_normal((Lseq, CFG.hidden))
    dy = rng.standard_normal((Lseq, CFG.hidden))
    W = rand_weights(CFG, 2)
    y, saved = L.sequence_forward(x, W, CFG)
    dx, grads = L.sequence_backward(dy, W, CFG, saved)
    mask = np.tril(np.ones((Lseq, Lseq), dtype=bool))
    ty, tdx, tg = torch_grads(x, dy, W, CFG, np.arange(Lseq), mask)
    np.testing.assert_allclose(y, ty, atol=1e-12)
    np.testing.assert_allclose(dx, tdx, atol=1e-11)
    for n in L.WEIGHT_NAMES:
        np.testing.assert_allclose(grads[n], tg[n], atol=1e-11, err_msg=n)


GROUPS = [[(5, [3, 0, 4]), (0, [2, 6]), (4, [])], [(6, [5])]]


@pytest.mark.parametrize("groups", GROUPS)
def test_packed_layer_against_dense_packed_torch(groups):
    """The replicated-sequence oracle on packed rows equals the layer run once
    over the packed rows (dense group mask, packed positions): the model-wide
    saving of the packed layout is exact."""
    T = sum(p + sum(r) for p, r in groups)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((T, CFG.hidden))
    dy = rng.standard_normal((T, CFG.hidden))
    W = rand_weights(CFG, 4)
    y = L.packed_forward(x, groups, W, CFG)
    dx, grads = L.packed_backward(x, dy, groups, W, CFG)
    ty, tdx, tg = torch_grads(x, dy, W, CFG, L.packed_positions(groups), group_mask(groups))
    np.testing.assert_allclose(y, ty, atol=1e-12)
    np.testing.assert_allclose(dx, tdx, atol=1e-11)
    for n in L.WEIGHT_NAMES:
        np.testing.assert_allclose(grads[n], tg[n], atol=1e-10, err_msg=n)


def test_finite_differences():
    c = L.LayerConfig(hidden=8, Hq=2, Hkv=1, d=4, inter=6, rope_base=100.0, eps=1e-6)
    Lseq = 4
    rng = np.random.default_rng(5)
    x = rng.standard_normal((Lseq, c.hidden))
    dy = rng.standard_normal((Lseq, c.hidden))
    W = rand_weights(c, 6)
    _, saved = L.sequence_forward(x, W, c)
    dx, grads = L.sequence_backward(dy, W, c, saved)

    def loss(x_, W_):
        return float((L.sequence_forward(x_, W_, c)[0] * dy).sum())

    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (loss(xp, W) - loss(xm, W)) / (2 * h)
    np.testing.assert_allclose(dx, fd, rtol=1e-6, atol=1e-8)
    for n in ("ln1", "wqkv", "wgu"):
        fdw = np.zeros_like(W[n])
        for idx in np.ndindex(*W[n].shape):
            Wp = dict(W)
            Wm = dict(W)
            Wp[n] = W[n].copy()
            Wm[n] = W[n].copy()
            Wp[n][idx] += h
            Wm[n][idx] -= h
            fdw[idx] = (loss(x, Wp) - loss(x, Wm)) / (2 * h)
        np.testing.assert_allclose(grads[n], fdw, rtol=1e-6, atol=1e-8, err_msg=n)


def test_rope_invariants():
    d, base = 16, 1.0e4
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    # position 0 is the identity
    np.testing.assert_array_equal(L.rope(q, L.rope_angles([0], d, base)), q)
    # each feature pair keeps its length
    r = L.rope(q, L.rope_angles([37], d, base))
    np.testing.assert_allclose(r[..., :d // 2] ** 2 + r[..., d // 2:] ** 2, q[..., :d // 2] ** 2 + q[..., d // 2:] ** 2)

    # q at m . k at n depends on m - n only
    def dot(m, n):
        return float((L.rope(q, L.rope_angles([m], d, base)) * L.rope(k, L.rope_angles([n], d, base))).sum())

    assert dot(10, 3) == pytest.approx(dot(107, 100), abs=1e-10)
    assert dot(10, 3) != pytest.approx(dot(10, 4), abs=1e-6)
    # backward is the inverse rotation
    ang = L.rope_angles([5, 900], d, base)
    x = rng.standard_normal((2, 3, d))
    np.testing.assert_allclose(L.rope_bwd(L.rope(x, ang), ang), x, atol=1e-12)


def test_rms_norm_closed_forms():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((5, 64)) * 3.0
    y, r = L.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt((y * y).mean(axis=1)), 1.0, rtol=1e-12)
    y2, _ = L.rms_norm(7.5 * x, np.ones(64), 0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-12)


def test_packed_positions():
    assert list(L.packed_positions([(3, [2, 1]), (0, [2]), (2, [])])) == [0, 1, 2, 3, 4, 3, 0, 1, 0, 1]


def _pin_fails():
    try:
        test_sequence_layer_against_torch_autograd()
    except AssertionError:
        return True
    return False


def test_planted_mistakes_are_caught(monkeypatch):
    real_rope, real_norm_bwd, real_swiglu_bwd = L.rope, L.rms_norm_bwd, L.swiglu_bwd

    def rope_sign(x, ang):
        return real_rope(x, -ang)

    def norm_bwd_no_mean_term(dy, x, r, w):
        dx, dw = real_norm_bwd(dy, x, r, w)
        return r * dy * w, dw

    def swiglu_bwd_plain(dm, g, u):
        sg = 1.0 / (1.0 + np.exp(-g))
        return dm * u * sg, dm * g * sg

    for name, fn in (("rope", rope_sign), ("rms_norm_bwd", norm_bwd_no_mean_term),
                     ("swiglu_bwd", swiglu_bwd_plain)):
        with monkeypatch.context() as m:
            m.setattr(L, name, fn)
            assert _pin_fails(), name
    assert not _pin_fails()
