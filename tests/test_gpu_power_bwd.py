"""Gradients of the power-sharpened attention on the tensor cores against the
float64 oracle's chain rule (itself pinned by finite differences and torch
autograd), on the same bf16-rounded inputs.  Bar: per-tensor relative L2
error <= 1e-2 (the gradient bar of the p = 1 backward)."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import f64, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-2


def run(x, p, pos0=0, eps=0.0, dO=None):
    g = to_dev(x)
    o, D = S.sanatan_power_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p,
                               pos0=pos0, eps=eps)
    dO = g["dO"] if dO is None else dO.to(g["q"].device)
    grads = S.sanatan_power_bwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p, o, D,
                                dO, pos0=pos0, eps=eps)
    S.device_status()
    return grads


def check(x, p, pos0=0, eps=0.0, names=("dq", "dk", "dv", "dgamma", "domega", "dphi")):
    grads = run(x, p, pos0=pos0, eps=eps)
    ref = O.attn_power_backward(**ref_args(x), dO=f64(x["dO"]), p=p, pos0=pos0, eps=eps)
    for n in names:
        err = rel_fro(f64(grads[n]), ref[n])
        assert err <= TOL, (p, n, err)


@pytest.mark.parametrize("p", [1, 2, 4])
@pytest.mark.parametrize("T", [1, 100, 128, 129, 300])
def test_short_sequences(p, T):
    # A single token with eps = 0 has o = v whatever q and k are (its gradients
    # in q, k and the parameters vanish); eps > 0 keeps them non-degenerate.
    check(W.make(W.TRAIN, B=1, H=2, T=T, with_grad_out=True), p, eps=0.5 if T == 1 else 0.0)


@pytest.mark.parametrize("p", [1, 2])
def test_single_token_without_eps_is_degenerate(p):
    """T = 1, eps = 0: o = v exactly, so dv = dO and every other gradient is
    zero; the kernel's are rounding noise far below the gradients' scale."""
    x = W.make(W.TRAIN, B=1, H=2, T=1, with_grad_out=True)
    g = run(x, p)
    assert rel_fro(f64(g["dv"]), f64(x["dO"])) <= TOL
    scale = float(np.abs(f64(x["dO"])).max())
    for n in ("dq", "dk", "dgamma", "domega", "dphi"):
        assert float(np.abs(f64(g[n])).max()) <= 1e-2 * scale, n


def test_eps_offset_and_odd_power():
    check(W.make(W.TRAIN, B=2, H=2, T=257, with_grad_out=True), 3, pos0=500, eps=0.5)


def test_f32_upstream_gradient():
    x = W.make(W.TRAIN, B=1, H=2, T=200, with_grad_out=True)
    x["dO"] = x["dO"].float()
    check(x, 2)


def test_power_one_matches_the_p1_backward_with_eps_times_4d():
    x = W.make(W.TRAIN, B=1, H=3, T=390, with_grad_out=True)
    g = to_dev(x)
    a = run(x, 1, eps=0.25)
    o, D, _, _ = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                     eps=0.25 * 4 * 64)
    b = S.sanatan_chunk_bwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], o, D,
                            g["dO"], eps=0.25 * 4 * 64, want_dphi=True)
    for n in ("dq", "dk", "dv", "dgamma", "domega", "dphi"):
        assert rel_fro(f64(a[n]), f64(b[n])) <= 2 * TOL, n


def test_layer_shape_sampled_heads():
    """B=2, H=2, T=2048 (16 key and query chunks): whole heads and the parameter
    gradients against the definition."""
    check(W.make(W.TRAIN, B=2, H=2, T=2048, with_grad_out=True), 2)
