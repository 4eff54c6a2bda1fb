"""One decode token through a stack of attention layers (12 heads x 64 per
layer, synthetic projections) against the float64 oracle: the stepped outputs
against the oracle's stepped stack and its parallel form (float32 path with
atomically accumulated projections: <= 1e-4 relative to the output scale)."""
import math

import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from gpu_util import dev, f64

pytestmark = pytest.mark.gpu


def _case(B, L, heads, seed=0):
    g = torch.Generator().manual_seed(seed)
    Dm = heads * 64
    return dict(
        Wqkv=torch.randn(L, Dm, 3 * Dm, generator=g) / math.sqrt(Dm),
        Wo=torch.randn(L, Dm, Dm, generator=g) / math.sqrt(Dm),
        gamma=torch.full((L, heads), 4.0),
        omega=torch.rand(L, heads, 64, generator=g) * 2 * math.pi - math.pi,
        phi=torch.tensor([10000.0 ** (-a / 64) for a in range(64)]).repeat(L, heads, 1).float())


@pytest.mark.parametrize("B,L,heads", [(1, 3, 12), (2, 2, 12), (8, 1, 12), (3, 2, 2), (5, 2, 4)])
def test_stack_steps_match_the_parallel_form(B, L, heads):
    T = 12
    c = _case(B, L, heads)
    Dm = heads * 64
    X = torch.randn(B, T, Dm, generator=torch.Generator().manual_seed(9))
    gd = {n: t.to(dev()).contiguous() for n, t in c.items()}
    Sd = torch.zeros(L, B * heads, 384, 64, device=dev())
    zd = torch.zeros(L, B * heads, 384, device=dev())
    outs = []
    for t in range(T):
        x = X[:, t].contiguous().to(dev())
        pos = torch.full((B * heads,), 40 + t, dtype=torch.int64, device=dev())
        S.sanatan_stack_decode_step(x, gd["Wqkv"], gd["Wo"], Sd, zd, gd["gamma"], gd["omega"],
                                    gd["phi"], pos, eps=0.05)
        outs.append(x)
    Y = torch.stack(outs, 1)
    torch.cuda.synchronize()
    c64 = {n: f64(t) for n, t in c.items()}
    Y_ref = O.stack_parallel(f64(X), c64["Wqkv"], c64["Wo"], c64["gamma"], c64["omega"],
                             c64["phi"], heads, pos0=40, eps=0.05)
    scale = np.abs(Y_ref).max()
    assert np.abs(f64(Y) - Y_ref).max() <= 1e-4 * scale
    S_ref = np.zeros((L, B * heads, 384, 64))
    z_ref = np.zeros((L, B * heads, 384))
    for t in range(T):
        _, S_ref, z_ref = O.stack_decode_step(f64(X)[:, t], c64["Wqkv"], c64["Wo"], S_ref, z_ref,
                                              c64["gamma"], c64["omega"], c64["phi"], heads,
                                              np.full(B, 40 + t), eps=0.05)
    assert np.linalg.norm(f64(Sd) - S_ref) <= 1e-4 * np.linalg.norm(S_ref)


def test_unsupported_batch():
    c = _case(9, 1, 12)
    x = torch.zeros(9, 768, device=dev())
    with pytest.raises(S.SanatanError) as e:
        S.sanatan_stack_decode_step(x, c["Wqkv"].to(dev()), c["Wo"].to(dev()),
                                    torch.zeros(1, 108, 384, 64, device=dev()),
                                    torch.zeros(1, 108, 384, device=dev()), c["gamma"].to(dev()),
                                    c["omega"].to(dev()), c["phi"].to(dev()),
                                    torch.zeros(108, dtype=torch.int64, device=dev()))
    assert e.value.status == 2
