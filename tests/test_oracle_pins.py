"""The float64 oracle against facts that the SANATAN pages and mathematics fix
(closed forms, invariants, brute force, a hand-derived worked example, finite
differences, the pages' memory table) and against torch float64 autograd."""
import math

import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
import oracle_pins as P


@pytest.mark.parametrize("check", P.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check()


def _torch_forward(q, k, v, gamma, omega, phi, pos0, eps):
    """Autograd-able float64 forward of eqs. (2)-(4), (6), (8) at p = 1,
    differentiated by torch's own engine to cross-check the oracle's
    hand-derived backward."""
    B, H, T, d = q.shape
    t = (torch.arange(T, dtype=torch.float64) + pos0).view(1, 1, T, 1)
    g = gamma.view(1, H, 1, 1)
    om = omega.view(1, H, 1, d)
    ph = phi.view(1, H, 1, d)

    def feat(u):
        th = math.pi * u / (1 + u.abs())
        r = torch.tanh(g * (torch.cos(th + om) - torch.sin(th + om)))
        tr = th + t * ph
        c, s = torch.cos(tr), torch.sin(tr)
        return torch.stack([torch.ones_like(c), c, s, r, r * c, r * s], -1).reshape(B, H, T, 6 * d)

    s = feat(q) @ feat(k).transpose(-1, -2)
    s = s * torch.tril(torch.ones(T, T, dtype=torch.float64))
    return (s @ v) / (s.sum(-1, keepdim=True) + eps)


@pytest.mark.parametrize("eps,pos0", [(0.0, 0), (0.5, 7)])
def test_backward_matches_torch_autograd(eps, pos0):
    rng = np.random.default_rng(21)
    B, H, T, d, dv = 2, 2, 10, 3, 4
    arr = dict(q=rng.standard_normal((B, H, T, d)), k=rng.standard_normal((B, H, T, d)),
               v=rng.standard_normal((B, H, T, dv)), gamma=rng.uniform(1, 5, H),
               omega=rng.uniform(-3, 3, (H, d)), phi=rng.uniform(0, 1, (H, d)))
    dO = rng.standard_normal((B, H, T, dv))
    ts = {n: torch.tensor(a, requires_grad=True) for n, a in arr.items()}
    o = _torch_forward(ts["q"], ts["k"], ts["v"], ts["gamma"], ts["omega"], ts["phi"], pos0, eps)
    o_ref, _ = O.attn_quadratic(**arr, pos0=pos0, eps=eps)
    assert np.allclose(o.detach().numpy(), o_ref, rtol=1e-12, atol=1e-12)
    (o * torch.tensor(dO)).sum().backward()
    g = O.attn_backward(**arr, dO=dO, pos0=pos0, eps=eps)
    for n in ("q", "k", "v", "gamma", "omega", "phi"):
        assert np.allclose(g["d" + n], ts[n].grad.numpy(), rtol=1e-10, atol=1e-10), n


def _torch_power_forward(q, k, v, gamma, omega, phi, p, pos0, eps):
    """Eq. (8) at integer p in torch float64 (features as in _torch_forward)."""
    B, H, T, d = q.shape
    t = (torch.arange(T, dtype=torch.float64) + pos0).view(1, 1, T, 1)
    g = gamma.view(1, H, 1, 1)
    om = omega.view(1, H, 1, d)
    ph = phi.view(1, H, 1, d)

    def feat(u):
        th = math.pi * u / (1 + u.abs())
        r = torch.tanh(g * (torch.cos(th + om) - torch.sin(th + om)))
        tr = th + t * ph
        c, s = torch.cos(tr), torch.sin(tr)
        return torch.stack([torch.ones_like(c), c, s, r, r * c, r * s], -1).reshape(B, H, T, 6 * d)

    w = (feat(q) @ feat(k).transpose(-1, -2) / (4.0 * d)) ** p
    w = w * torch.tril(torch.ones(T, T, dtype=torch.float64))
    return (w @ v) / (w.sum(-1, keepdim=True) + eps)


@pytest.mark.parametrize("p,eps,pos0", [(2, 0.0, 0), (4, 0.01, 5)])
def test_power_backward_matches_torch_autograd(p, eps, pos0):
    rng = np.random.default_rng(31 + p)
    B, H, T, d, dv = 1, 2, 9, 3, 2
    arr = dict(q=rng.standard_normal((B, H, T, d)), k=rng.standard_normal((B, H, T, d)),
               v=rng.standard_normal((B, H, T, dv)), gamma=rng.uniform(1, 5, H),
               omega=rng.uniform(-3, 3, (H, d)), phi=rng.uniform(0, 1, (H, d)))
    dO = rng.standard_normal((B, H, T, dv))
    ts = {n: torch.tensor(a, requires_grad=True) for n, a in arr.items()}
    o = _torch_power_forward(ts["q"], ts["k"], ts["v"], ts["gamma"], ts["omega"], ts["phi"], p,
                             pos0, eps)
    o_ref, _ = O.attn_power(**arr, p=p, pos0=pos0, eps=eps)
    assert np.allclose(o.detach().numpy(), o_ref, rtol=1e-12, atol=1e-12)
    (o * torch.tensor(dO)).sum().backward()
    g = O.attn_power_backward(**arr, dO=dO, p=p, pos0=pos0, eps=eps)
    for n in ("q", "k", "v", "gamma", "omega", "phi"):
        assert np.allclose(g["d" + n], ts[n].grad.numpy(), rtol=1e-10, atol=1e-10), n
