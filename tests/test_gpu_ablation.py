"""The four-channel (clipped) and three-channel (optionally shifted) ablation
kernels on the tensor cores against the float64 oracle, on the same
bf16-rounded inputs.  Bars as for the power-sharpened attention: outputs max
abs <= 5e-3, the denominator relative Frobenius <= 2e-3 * p."""
import math

import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import f64, max_abs, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu

TOL_O = 5e-3


def check(x, p, channels, shift=0.0, pos0=0, eps=0.0):
    g = to_dev(x)
    o, D = S.sanatan_ablation_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p,
                                  channels, shift=shift, pos0=pos0, eps=eps)
    S.device_status()
    o_ref, D_ref = O.attn_ablation(**ref_args(x), p=p, channels=channels, shift=shift, pos0=pos0,
                                   eps=eps)
    err = max_abs(f64(o), o_ref)
    assert err <= TOL_O, (p, channels, shift, err)
    assert rel_fro(f64(D), D_ref) <= 2e-3 * p, (p, channels, rel_fro(f64(D), D_ref))


@pytest.mark.parametrize("channels,shift", [(4, 0.0), (3, 0.0), (3, 64.0)])
@pytest.mark.parametrize("p", [1, 2, 4])
@pytest.mark.parametrize("T", [1, 129, 300])
def test_short_sequences(T, p, channels, shift):
    check(W.make(W.LAYER, B=1, H=2, T=T), p, channels, shift)


def test_eps_offset():
    x = W.make(W.LAYER, B=2, H=2, T=257)
    check(x, 2, 4, pos0=900, eps=0.25)
    check(x, 4, 3, shift=64.0, pos0=33, eps=1e-3)


def test_four_channel_clip_on_the_gpu():
    """Keys whose total four-channel score is negative get weight zero: with
    every dimension's roots opposite (u_k = -u_q, omega = pi/4, a large gamma)
    and angle difference near 0 mod 2 pi, key 1's score for query 1 is about
    -0.98 d, so o_1 = v_0 (key 0 matches query 1)."""
    d, th = 64, math.pi - 0.1
    u = th / (math.pi - th)
    bf = torch.bfloat16
    q = torch.zeros(1, 1, 2, d, dtype=bf)
    k = torch.zeros(1, 1, 2, d, dtype=bf)
    q[..., 0, :] = 0.3
    q[..., 1, :] = u
    k[..., 0, :] = u
    k[..., 1, :] = -u
    v = torch.randn(1, 1, 2, d, generator=torch.Generator().manual_seed(3)).to(bf)
    x = dict(q=q, k=k, v=v, gamma=torch.tensor([100.0]), omega=torch.full((1, d), math.pi / 4),
             phi=torch.zeros(1, d))
    for p in (1, 2, 4):
        check(x, p, 4)
        g = to_dev(x)
        o, _ = S.sanatan_ablation_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p,
                                      4)
        assert max_abs(f64(o)[0, 0, 1], f64(v)[0, 0, 0]) <= TOL_O


def test_layer_shape_sampled_heads():
    """B=4, H=12, T=2048 (16 query and key chunks per sequence) in the launch
    configuration the benchmark times; whole heads checked against the
    definition."""
    x = W.make(W.LAYER, device="cpu")
    g = to_dev(x)
    ra = ref_args(x)
    for channels, shift, p in ((4, 0.0, 2), (3, 64.0, 2), (3, 0.0, 4)):
        o, D = S.sanatan_ablation_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p,
                                      channels, shift=shift)
        S.device_status()
        for b, h in ((0, 0), (3, 11)):
            sl = {n: ra[n][b:b + 1, h:h + 1] for n in ("q", "k", "v")}
            o_ref, D_ref = O.attn_ablation(**sl, gamma=ra["gamma"][h:h + 1],
                                           omega=ra["omega"][h:h + 1], phi=ra["phi"][h:h + 1],
                                           p=p, channels=channels, shift=shift)
            assert max_abs(f64(o)[b, h], o_ref[0, 0]) <= TOL_O, (channels, shift, p, b, h)
            assert rel_fro(f64(D)[b, h], D_ref[0, 0]) <= 2e-3 * p


def test_argument_errors():
    x = W.make(W.LAYER, B=1, H=1, T=8)
    g = to_dev(x)
    a = (g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"])
    for p, ch, sh, status in ((2, 5, 0.0, 1), (2, 4, 1.0, 1), (2, 3, -1.0, 1), (3, 4, 0.0, 2),
                              (0, 3, 0.0, 1)):
        with pytest.raises(S.SanatanError) as e:
            S.sanatan_ablation_fwd(*a, p, ch, shift=sh)
        assert e.value.status == status
