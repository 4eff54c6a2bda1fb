"""Power-sharpened causal attention (eq. (8) at integer p) on the tensor cores
against the float64 oracle, on the same bf16-rounded inputs.

Bars: outputs max abs <= 5e-3 (bf16 features and values, f32 scores and
accumulation, the weights (s/4d)^p entering the tensor cores as a bf16 hi + lo
pair); the denominator sum (s/4d)^p relative Frobenius <= 2e-3 * p (a relative
error e of a score moves its weight by p e)."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import dev, f64, max_abs, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu

TOL_O = 5e-3


def tol_den(p):
    return 2e-3 * p


def run(x, p, **kw):
    g = to_dev(x)
    o, D = S.sanatan_power_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p, **kw)
    S.device_status()
    return f64(o), f64(D)


def check_full(x, p, pos0=0, eps=0.0):
    o, D = run(x, p, pos0=pos0, eps=eps)
    o_ref, D_ref = O.attn_power(**ref_args(x), p=p, pos0=pos0, eps=eps)
    err = max_abs(o, o_ref)
    assert err <= TOL_O, (p, err)
    assert rel_fro(D, D_ref) <= tol_den(p), (p, rel_fro(D, D_ref))
    return err


@pytest.mark.parametrize("p", [1, 2, 4])
@pytest.mark.parametrize("T", [1, 100, 128, 129, 300])
def test_short_sequences(p, T):
    # one chunk, a ragged single chunk, exactly one chunk, one token past it,
    # and three chunks with a ragged tail
    check_full(W.make(W.LAYER, B=1, H=2, T=T), p)


@pytest.mark.parametrize("p", [3, 8])
def test_odd_and_largest_power(p):
    check_full(W.make(W.LAYER, B=2, H=1, T=260), p)


def test_eps_and_position_offset():
    x = W.make(W.LAYER, B=2, H=3, T=257)
    check_full(x, 2, pos0=1000, eps=0.5)
    check_full(x, 4, pos0=77, eps=1e-3)


def test_power_one_is_the_p1_forward_with_eps_times_4d():
    x = W.make(W.LAYER, B=1, H=3, T=700)
    g = to_dev(x)
    eps = 0.25
    o1, D1 = S.sanatan_power_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 1,
                                 eps=eps)
    o2, D2, _, _ = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                       eps=eps * 4 * 64)
    S.device_status()
    assert max_abs(f64(o1), f64(o2)) <= 2 * TOL_O
    assert rel_fro(f64(D1) * 4 * 64, f64(D2)) <= 2e-3


def test_many_sequences_one_chunk_each():
    # more CTAs than SMs in one wave, every CTA on the diagonal
    x = W.make(W.LAYER, B=2, H=96, T=128)
    o, D = run(x, 2)
    ra = ref_args(x)
    for b, h in ((0, 0), (1, 95), (0, 50)):
        sl = {n: ra[n][b:b + 1, h:h + 1] for n in ("q", "k", "v")}
        o_ref, D_ref = O.attn_power(**sl, gamma=ra["gamma"][h:h + 1], omega=ra["omega"][h:h + 1],
                                    phi=ra["phi"][h:h + 1], p=2)
        assert max_abs(o[b, h], o_ref[0, 0]) <= TOL_O
        assert rel_fro(D[b, h], D_ref[0, 0]) <= tol_den(2)


@pytest.mark.parametrize("p", [2, 4])
def test_layer_shape_full_size_sampled_heads(p):
    """B=4, H=12, T=2048 (768 CTAs, 16 key chunks for the last query chunk):
    whole heads checked against the definition."""
    x = W.make(W.LAYER, device="cpu")
    o, D = run(x, p)
    ra = ref_args(x)
    for b, h in ((0, 0), (3, 11), (2, 5)):
        sl = {n: ra[n][b:b + 1, h:h + 1] for n in ("q", "k", "v")}
        o_ref, D_ref = O.attn_power(**sl, gamma=ra["gamma"][h:h + 1], omega=ra["omega"][h:h + 1],
                                    phi=ra["phi"][h:h + 1], p=p)
        assert max_abs(o[b, h], o_ref[0, 0]) <= TOL_O, (b, h)
        assert rel_fro(D[b, h], D_ref[0, 0]) <= tol_den(p), (b, h)


def test_rows_are_convex_combinations_of_values():
    # the weights are non-negative and normalised (eps = 0): every output lies
    # inside the per-column range of the values it averages
    x = W.make(W.LAYER, B=1, H=2, T=1000)
    o, _ = run(x, 4)
    v = f64(x["v"])
    cmax = np.maximum.accumulate(v, axis=2)
    cmin = np.minimum.accumulate(v, axis=2)
    assert (o <= cmax + 1e-3).all() and (o >= cmin - 1e-3).all()


def test_invalid_power_is_rejected():
    x = W.make(W.LAYER, B=1, H=1, T=8)
    g = to_dev(x)
    for p, code in ((0, 1), (9, 2)):
        with pytest.raises(S.SanatanError) as e:
            S.sanatan_power_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p)
        assert f"status {code}" in str(e.value)


def test_empty_inputs_do_nothing():
    """T = 0 and B * H = 0 are valid calls that write nothing."""
    for B, H, T in ((2, 3, 0), (0, 3, 256)):
        x = W.make(W.LAYER, device="cpu", B=max(B, 1), H=H, T=T)
        g = {n: x[n].to(dev()) for n in ("q", "k", "v", "gamma", "omega", "phi")}
        if B == 0:
            for n in ("q", "k", "v"):
                g[n] = g[n][:0]
        o, D = S.sanatan_power_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 2)[:2]
        torch.cuda.synchronize()
        S.device_status()
        assert o.numel() == 0 and (D is None or D.numel() == 0)
