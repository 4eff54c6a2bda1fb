"""Checks that pin the float64 oracle to facts fixed by the SANATAN pages and by
mathematics, independently of the oracle's own code.

Each ``check_*`` function raises AssertionError when the oracle disagrees.
``test_oracle_pins.py`` runs them all; ``test_oracle_mutations.py`` plants
plausible mistakes in the oracle and shows that at least one check fails for
each, so a dropped term, a wrong sign or index, or a transposed operand does
not go unnoticed.
"""
import math
import os

import numpy as np

import oracle.sanatan_oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _small_case(seed=0, B=1, H=2, T=9, d=3, dv=2, phi_scale=0.3):
    g = _rng(seed)
    return dict(
        q=g.standard_normal((B, H, T, d)),
        k=g.standard_normal((B, H, T, d)),
        v=g.standard_normal((B, H, T, dv)),
        gamma=g.uniform(1.0, 5.0, H),
        omega=g.uniform(-math.pi, math.pi, (H, d)),
        phi=g.uniform(0.0, phi_scale, (H, d)),
    )


# --------------------------------------------------------------------------
# eq. (2): angle squash
# --------------------------------------------------------------------------

def check_squash_closed_forms():
    # u = 0, +-1, +-1/3, 3 give 0, +-pi/2, +-pi/4, 3pi/4 (pi*u/(1+|u|) by hand)
    u = np.array([0.0, 1.0, -1.0, 1.0 / 3.0, -1.0 / 3.0, 3.0])
    want = np.array([0.0, math.pi / 2, -math.pi / 2, math.pi / 4, -math.pi / 4, 3 * math.pi / 4])
    assert np.allclose(O.squash(u), want, rtol=0, atol=1e-15), O.squash(u)
    # near the origin the map is pi*u to first order; it stays inside (-pi, pi)
    x = np.array([1e-9, -1e-9])
    assert np.allclose(O.squash(x) / x, math.pi, rtol=1e-8)
    big = np.array([1e6, -1e6, 3e7])
    th = O.squash(big)
    assert np.all(np.abs(th) < math.pi) and np.allclose(np.abs(th), math.pi, rtol=1e-5)
    grid = np.linspace(-20, 20, 4001)
    assert np.all(np.diff(O.squash(grid)) > 0)  # strictly increasing


# --------------------------------------------------------------------------
# eq. (3): soft root label
# --------------------------------------------------------------------------

def check_soft_root_closed_forms():
    th = np.linspace(-3.1, 3.1, 257)
    for gamma in (0.5, 4.0, 10.0):
        # with omega = pi/4 the coefficient is -sqrt(2) sin(theta)
        r = O.soft_root(th, gamma, math.pi / 4)
        assert np.allclose(r, np.tanh(-gamma * math.sqrt(2.0) * np.sin(th)), rtol=0, atol=1e-14)
        # sign of the root is opposite to the sign of a nonzero theta in (-pi, pi)
        nz = np.abs(th) > 1e-3
        assert np.all(np.sign(r[nz]) == -np.sign(th[nz]))
    # the root boundary: theta = pi/4 - omega (mod pi) gives r = 0
    for omega in (-2.0, -0.3, 0.0, 0.7, 2.9):
        for m in (-1, 0, 1):
            b = math.pi / 4 - omega + m * math.pi
            assert abs(O.soft_root(b, 7.0, omega)) < 1e-13
    # omega -> omega + pi swaps every label (r -> -r)
    om = np.linspace(-3, 3, 13)
    a = O.soft_root(0.37, 3.0, om)
    b = O.soft_root(0.37, 3.0, om + math.pi)
    assert np.allclose(a, -b, atol=1e-13)
    # a large gamma makes the root hard (+-1)
    hard = O.soft_root(np.array([0.5, -0.5]), 200.0, math.pi / 4)
    assert np.allclose(hard, [-1.0, 1.0], atol=1e-12)


# --------------------------------------------------------------------------
# eq. (6)-(7): six-channel features and the factorised kernel
# --------------------------------------------------------------------------

def check_feature_channels():
    g = _rng(1)
    th = g.uniform(-7, 7, (5, 4))
    r = g.uniform(-1, 1, (5, 4))
    f = O.features_from_angles(th, r).reshape(5, 4, 6)
    assert np.all(f[..., 0] == 1.0)
    assert np.allclose(f[..., 1], np.cos(th), atol=1e-15)
    assert np.allclose(f[..., 2], np.sin(th), atol=1e-15)
    assert np.allclose(f[..., 3], r, atol=1e-15)
    assert np.allclose(f[..., 4], r * np.cos(th), atol=1e-15)
    assert np.allclose(f[..., 5], r * np.sin(th), atol=1e-15)


def check_factorisation_bruteforce():
    """<Phi_a(q), Phi_a(k)> = (1 + r_q r_k)(1 + cos(th_q - th_k)) summed over a."""
    g = _rng(2)
    for d in (1, 2, 3, 5):
        for _ in range(20):
            tq, tk = g.uniform(-10, 10, d), g.uniform(-10, 10, d)
            rq, rk = g.uniform(-1, 1, d), g.uniform(-1, 1, d)
            fq = O.features_from_angles(tq, rq)
            fk = O.features_from_angles(tk, rk)
            got = float(O.pair_kernel(fq[None], fk[None])[0, 0])
            want = sum((1 + rq[a] * rk[a]) * (1 + math.cos(tq[a] - tk[a])) for a in range(d))
            assert abs(got - want) < 1e-12 * max(1.0, abs(want))
            assert -1e-12 <= got <= 4 * d + 1e-12
    # hard roots: the per-dimension gate is 0 (labels differ) or 2 (labels agree)
    for rq, rk, gate in ((1, 1, 2), (-1, -1, 2), (1, -1, 0), (-1, 1, 0)):
        f1 = O.features_from_angles(np.array([0.4]), np.array([float(rq)]))
        f2 = O.features_from_angles(np.array([0.4]), np.array([float(rk)]))
        assert abs(float(O.pair_kernel(f1[None], f2[None])[0, 0]) - gate * 2.0) < 1e-14


def check_kernel_range_from_inputs():
    c = _small_case(3, H=2, T=40, d=6)
    pq = O.featurize(c["q"], c["gamma"], c["omega"], c["phi"])
    pk = O.featurize(c["k"], c["gamma"], c["omega"], c["phi"])
    for h in range(2):
        s = O.pair_kernel(pq[0, h], pk[0, h])
        assert s.min() >= -1e-12 and s.max() <= 4 * 6 + 1e-12


# --------------------------------------------------------------------------
# A worked example derived by hand from eqs. (2)-(4), (6), (8)-(9)
# --------------------------------------------------------------------------

def worked_example():
    """d = 1, T = 2, gamma = 1, omega = pi/4, phi = pi/2, pos0 = 0.

    u_q = (1/3, 1)   -> theta_q = (pi/4, pi/2)
    u_k = (-1/3, 0)  -> theta_k = (-pi/4, 0)
    roots from the UN-rotated angles, r = tanh(-sqrt(2) sin theta):
      r_q = (tanh(-1), tanh(-sqrt 2)),  r_k = (tanh(1), 0)
    rotated angles theta + t*pi/2: q -> (pi/4, pi), k -> (-pi/4, pi/2)
      s_00 = (1 - tanh(1)^2) (1 + cos(pi/2))            = sech(1)^2
      s_10 = (1 - tanh(sqrt 2) tanh(1)) (1 + cos(5pi/4)) = (1 - th2 th1)(1 - sqrt(2)/2)
      s_11 = (1 + 0) (1 + cos(pi/2))                      = 1
    v = (2, -1):  o_0 = 2,  o_1 = (2 s_10 - s_11) / (s_10 + s_11)
    """
    th1, th2 = math.tanh(1.0), math.tanh(math.sqrt(2.0))
    s00 = 1.0 - th1 * th1
    s10 = (1.0 - th2 * th1) * (1.0 - math.sqrt(2.0) / 2.0)
    s11 = 1.0
    inputs = dict(
        q=np.array([1.0 / 3.0, 1.0]).reshape(1, 1, 2, 1),
        k=np.array([-1.0 / 3.0, 0.0]).reshape(1, 1, 2, 1),
        v=np.array([2.0, -1.0]).reshape(1, 1, 2, 1),
        gamma=np.array([1.0]), omega=np.array([[math.pi / 4]]), phi=np.array([[math.pi / 2]]),
    )
    o = np.array([2.0, (2.0 * s10 - s11) / (s10 + s11)])
    D = np.array([s00, s10 + s11])
    return inputs, o, D, (s00, s10, s11)


def check_worked_example():
    inp, o_want, D_want, (s00, s10, s11) = worked_example()
    pq = O.featurize(inp["q"], inp["gamma"], inp["omega"], inp["phi"])[0, 0]
    pk = O.featurize(inp["k"], inp["gamma"], inp["omega"], inp["phi"])[0, 0]
    s = O.pair_kernel(pq, pk)
    assert abs(s[0, 0] - s00) < 1e-14 and abs(s[1, 0] - s10) < 1e-14 and abs(s[1, 1] - s11) < 1e-14
    for fn in (O.attn_quadratic, O.attn_recurrent):
        res = fn(inp["q"], inp["k"], inp["v"], inp["gamma"], inp["omega"], inp["phi"])
        assert np.allclose(res[0].ravel(), o_want, rtol=0, atol=1e-14), (fn.__name__, res[0].ravel())
        assert np.allclose(res[1].ravel(), D_want, rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# eq. (8)-(9): quadratic form, recurrent form and their invariants
# --------------------------------------------------------------------------

def check_quadratic_equals_recurrent():
    for seed, eps, with_state in ((4, 0.0, False), (5, 0.37, False), (6, 0.0, True)):
        c = _small_case(seed, B=2, H=2, T=11, d=3, dv=2)
        S0 = z0 = None
        if with_state:
            S0, z0 = O.final_state(c["k"] * 0.5 + 0.1, c["v"][:, :, ::-1], c["gamma"], c["omega"],
                                   c["phi"], pos0=-11)
        a = O.attn_quadratic(**c, pos0=3, eps=eps, S0=S0, z0=z0)
        b = O.attn_recurrent(**c, pos0=3, eps=eps, S0=S0, z0=z0)
        assert np.allclose(a[0], b[0], rtol=1e-12, atol=1e-12)
        assert np.allclose(a[1], b[1], rtol=1e-12, atol=1e-12)
        S, z = O.final_state(c["k"], c["v"], c["gamma"], c["omega"], c["phi"], pos0=3, S0=S0, z0=z0)
        assert np.allclose(S, b[2], rtol=1e-12, atol=1e-12) and np.allclose(z, b[3], rtol=1e-12, atol=1e-12)


def check_single_token():
    c = _small_case(7, B=2, H=3, T=1, d=4, dv=3)
    o, D = O.attn_quadratic(**c)
    assert np.allclose(o, c["v"], rtol=0, atol=1e-14)
    o2, _, _, _ = O.attn_recurrent(**c)
    assert np.allclose(o2, c["v"], rtol=0, atol=1e-14)
    assert np.all(D > 0)


def check_constant_values():
    c = _small_case(8, B=1, H=2, T=17, d=3, dv=4)
    c["v"] = np.broadcast_to(np.array([0.5, -2.0, 3.0, 1e-3]), c["v"].shape).copy()
    o, _ = O.attn_quadratic(**c)
    assert np.allclose(o, c["v"], rtol=1e-13, atol=1e-13)


def check_relative_position():
    c = _small_case(9, B=1, H=2, T=13, d=3, dv=2, phi_scale=0.9)
    o_a, D_a = O.attn_quadratic(**c, pos0=0)
    o_b, D_b = O.attn_quadratic(**c, pos0=12345)
    assert np.allclose(o_a, o_b, rtol=1e-9, atol=1e-9) and np.allclose(D_a, D_b, rtol=1e-9, atol=1e-9)
    # the state itself does depend on the absolute position
    S_a, _ = O.final_state(c["k"], c["v"], c["gamma"], c["omega"], c["phi"], pos0=0)
    S_b, _ = O.final_state(c["k"], c["v"], c["gamma"], c["omega"], c["phi"], pos0=12345)
    assert not np.allclose(S_a, S_b)


def check_state_channel_zero():
    c = _small_case(10, B=2, H=2, T=23, d=5, dv=3)
    _, _, S, z = O.attn_recurrent(**c)
    d = 5
    for a in range(d):
        assert np.allclose(S[:, :, 6 * a, :], c["v"].sum(axis=2), rtol=1e-13, atol=1e-13)
        assert np.allclose(z[:, :, 6 * a], 23.0, rtol=0, atol=1e-12)
    # denominator positivity with soft roots
    _, D = O.attn_quadratic(**c)
    assert np.all(D > 0)


def check_rows_and_decode():
    c = _small_case(11, B=1, H=2, T=15, d=3, dv=2)
    o, D = O.attn_quadratic(**c, pos0=5, eps=0.01)
    rows = [0, 3, 14]
    for h in range(2):
        oo, dd = O.attn_rows(c["q"], c["k"], c["v"], c["gamma"], c["omega"], c["phi"], rows,
                             pos0=5, eps=0.01, b=0, h=h)
        assert np.allclose(oo, o[0, h, rows], rtol=1e-12, atol=1e-12)
        assert np.allclose(dd, D[0, h, rows], rtol=1e-12, atol=1e-12)
    # token-by-token decode over the sequence reproduces the recurrent form
    H, F, dv = 2, 18, 2
    S = np.zeros((H, F, dv))
    z = np.zeros((H, F))
    for t in range(15):
        S, z, ot = O.decode_step(S, z, c["q"][0, :, t], c["k"][0, :, t], c["v"][0, :, t],
                                 c["gamma"], c["omega"], c["phi"], np.full(H, 5 + t), eps=0.01)
        assert np.allclose(ot, o[0, :, t], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# Backward: central finite differences in float64
# --------------------------------------------------------------------------

def _loss(c, dO, pos0, eps, S0, z0):
    o, _ = O.attn_quadratic(c["q"], c["k"], c["v"], c["gamma"], c["omega"], c["phi"],
                            pos0=pos0, eps=eps, S0=S0, z0=z0)
    return float((o * dO).sum())


def check_backward_finite_differences():
    c = _small_case(12, B=1, H=2, T=7, d=2, dv=2, phi_scale=0.8)
    g = _rng(13)
    dO = g.standard_normal(c["v"].shape)
    S0, z0 = O.final_state(g.standard_normal(c["k"].shape), g.standard_normal(c["v"].shape),
                           c["gamma"], c["omega"], c["phi"], pos0=-7)
    for pos0, eps, st in ((2, 0.0, False), (0, 0.25, True)):
        S = S0 if st else None
        Z = z0 if st else None
        grads = O.attn_backward(c["q"], c["k"], c["v"], c["gamma"], c["omega"], c["phi"], dO,
                                pos0=pos0, eps=eps, S0=S, z0=Z)
        h = 1e-6
        for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("gamma", "dgamma"),
                            ("omega", "domega"), ("phi", "dphi")):
            x = c[name]
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = _loss(c, dO, pos0, eps, S, Z)
                x[idx] = old - h
                lm = _loss(c, dO, pos0, eps, S, Z)
                x[idx] = old
                num[idx] = (lp - lm) / (2 * h)
            err = np.abs(num - grads[gname]).max() / max(1e-3, np.abs(num).max())
            assert err < 1e-6, (name, err)


# --------------------------------------------------------------------------
# Memory accounting printed by the pages (golden fixture)
# --------------------------------------------------------------------------

def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            out.setdefault(key, []).append([float(x) for x in vals])
    return out


def check_memory_accounting():
    g = read_golden("memory_accounting.txt")
    total = O.state_bytes(12, 12, 64, 64)
    assert total == int(g["state_bytes_total"][0][0])
    assert O.state_bytes(1, 1, 64, 64) == int(g["state_bytes_per_head"][0][0])
    assert round(total / 1e6, 1) == g["state_mb_decimal"][0][0]
    assert O.kv_crossover(12, 12, 64, 64, 768) == int(g["kv_crossover_n"][0][0])
    for n, mb in g["kv_mb"]:
        assert round(O.kv_cache_bytes(int(n), 12, 768) / 1e6, 1) == mb, (n, mb)


# --------------------------------------------------------------------------
# eq. (8) at p > 1: power-sharpened attention (Notes §2.6)
# --------------------------------------------------------------------------

def _tensor_power_features(phi, p):
    """Phi^{(x)p}: the p-fold outer product of each feature vector, flattened."""
    out = phi
    for _ in range(p - 1):
        out = np.einsum("...i,...j->...ij", out, phi).reshape(phi.shape[:-1] + (-1,))
    return out


def check_power_matches_tensor_power_features():
    """The notes' identity (Phi(q).Phi(k))^p = <Phi(q)^(x)p, Phi(k)^(x)p>: build the
    (6d)^p tensor-power features explicitly and run plain linear attention on them."""
    for p, d in ((2, 2), (4, 1), (3, 1)):
        c = _small_case(40 + p, B=1, H=2, T=7, d=d, dv=3)
        o, D = O.attn_power(**c, p=p, eps=0.25)
        pq = O.featurize(c["q"], c["gamma"], c["omega"], c["phi"])
        pk = O.featurize(c["k"], c["gamma"], c["omega"], c["phi"])
        Fq = _tensor_power_features(pq, p) / (4.0 * d) ** p
        Fk = _tensor_power_features(pk, p)
        T = c["q"].shape[2]
        for h in range(2):
            o_ref = np.zeros((T, 3))
            for t in range(T):
                w = np.array([Fq[0, h, t] @ Fk[0, h, j] for j in range(t + 1)])
                o_ref[t] = (w[:, None] * c["v"][0, h, :t + 1]).sum(0) / (w.sum() + 0.25)
                assert abs(D[0, h, t] - w.sum()) <= 1e-12 * max(1.0, w.sum())
            assert np.allclose(o[0, h], o_ref, rtol=1e-11, atol=1e-12)


def check_power_one_is_linear_attention():
    """At p = 1 eq. (8) is the linear attention with the raw-score eps scaled by 4d."""
    c = _small_case(50, B=2, H=2, T=11, d=3, dv=2)
    o1, D1 = O.attn_power(**c, p=1, eps=0.3)
    o2, D2 = O.attn_quadratic(**c, eps=0.3 * 4 * 3)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-13)
    assert np.allclose(D1 * (4 * 3), D2, rtol=1e-12, atol=1e-12)


def check_power_single_token_and_constant_values():
    c = _small_case(51, B=1, H=2, T=1, d=3, dv=2)
    o, _ = O.attn_power(**c, p=2)
    assert np.allclose(o, c["v"], rtol=0, atol=1e-14)
    c = _small_case(52, B=1, H=2, T=9, d=3, dv=3)
    c["v"] = np.broadcast_to(np.array([1.5, -0.25, 4.0]), c["v"].shape).copy()
    o, _ = O.attn_power(**c, p=4)
    assert np.allclose(o, c["v"], rtol=1e-13, atol=1e-13)


def _power_loss(c, dO, p, pos0, eps):
    o, _ = O.attn_power(c["q"], c["k"], c["v"], c["gamma"], c["omega"], c["phi"], p=p,
                        pos0=pos0, eps=eps)
    return float((o * dO).sum())


def check_power_backward_finite_differences():
    """Every gradient of eq. (8) at p = 2 and 3 against central differences of
    the forward."""
    c = _small_case(60, B=1, H=2, T=6, d=2, dv=2, phi_scale=0.8)
    g = _rng(61)
    dO = g.standard_normal(c["v"].shape)
    for p, pos0, eps in ((2, 3, 0.0), (3, 0, 0.05)):
        grads = O.attn_power_backward(c["q"], c["k"], c["v"], c["gamma"], c["omega"], c["phi"],
                                      dO, p=p, pos0=pos0, eps=eps)
        h = 1e-6
        for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("gamma", "dgamma"),
                            ("omega", "domega"), ("phi", "dphi")):
            x = c[name]
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = _power_loss(c, dO, p, pos0, eps)
                x[idx] = old - h
                lm = _power_loss(c, dO, p, pos0, eps)
                x[idx] = old
                num[idx] = (lp - lm) / (2 * h)
            err = np.abs(num - grads[gname]).max() / max(1e-3, np.abs(num).max())
            assert err < 1e-6, (p, name, err)


def check_power_one_backward_is_linear_backward():
    """At p = 1 the gradients are those of the p = 1 attention with eps x 4d."""
    c = _small_case(62, B=2, H=2, T=9, d=3, dv=2)
    dO = _rng(63).standard_normal(c["v"].shape)
    g1 = O.attn_power_backward(**c, dO=dO, p=1, pos0=4, eps=0.2)
    g2 = O.attn_backward(**c, dO=dO, pos0=4, eps=0.2 * 4 * 3)
    for n in ("dq", "dk", "dv", "dgamma", "domega", "dphi"):
        assert np.allclose(g1[n], g2[n], rtol=1e-10, atol=1e-12), n


ALL_CHECKS = [
    check_squash_closed_forms,
    check_soft_root_closed_forms,
    check_feature_channels,
    check_factorisation_bruteforce,
    check_kernel_range_from_inputs,
    check_worked_example,
    check_quadratic_equals_recurrent,
    check_single_token,
    check_constant_values,
    check_relative_position,
    check_state_channel_zero,
    check_rows_and_decode,
    check_backward_finite_differences,
    check_memory_accounting,
    check_power_matches_tensor_power_features,
    check_power_one_is_linear_attention,
    check_power_single_token_and_constant_values,
    check_power_backward_finite_differences,
    check_power_one_backward_is_linear_backward,
]


# --------------------------------------------------------------------------
# Ablation kernels: four channels (Notes §2.5) and three channels (Notes §4.4)
# --------------------------------------------------------------------------

def _angles(c, u, pos0=0):
    """Un-rotated and rotated angles and roots of one head, from the pages'
    formulas typed directly (not through the oracle's feature functions)."""
    th = math.pi * u / (1.0 + np.abs(u))
    t = (np.arange(u.shape[-2]) + pos0)[:, None]
    om, ph, g = c["omega"][0], c["phi"][0], c["gamma"][0]
    r = np.tanh(g * (np.cos(th + om) - np.sin(th + om)))
    return th + t * ph, r


def check_four_channel_kernel_closed_form():
    # Phi4(q).Phi4(k) = sum_a 1 + r_q r_k (1 + cos(dtheta_a)) (Notes §2.5)
    c = _small_case(seed=11, T=7, d=5)
    pq = O.featurize_ablation(c["q"], c["gamma"], c["omega"], c["phi"], 4)[0, 0]
    pk = O.featurize_ablation(c["k"], c["gamma"], c["omega"], c["phi"], 4)[0, 0]
    tq, rq = _angles(c, c["q"][0, 0])
    tk, rk = _angles(c, c["k"][0, 0])
    for i in range(7):
        for j in range(7):
            want = np.sum(1.0 + rq[i] * rk[j] * (1.0 + np.cos(tq[i] - tk[j])))
            assert abs(pq[i] @ pk[j] - want) < 1e-12
    assert pq.shape[-1] == 4 * 5


def check_four_channel_hard_roots():
    # matching hard roots give 2 + cos(dtheta) in [1, 3], mismatched -cos(dtheta)
    # in [-1, 1] (Notes §2.5)
    dth = np.linspace(-math.pi, math.pi, 101)
    for rq, rk, want in ((1.0, 1.0, 2.0 + np.cos(dth)), (-1.0, -1.0, 2.0 + np.cos(dth)),
                         (1.0, -1.0, -np.cos(dth)), (-1.0, 1.0, -np.cos(dth))):
        fq = O.features4_from_angles(dth[:, None] * 0 + dth[:, None], np.full((101, 1), rq))
        fk = O.features4_from_angles(np.zeros((101, 1)), np.full((101, 1), rk))
        got = np.sum(fq * fk, axis=-1)
        assert np.allclose(got, want, atol=1e-14)


def check_four_channel_clip():
    # A key whose total four-channel score is negative gets weight zero (the
    # max(s, 0) before the power, Notes §2.5): query 1 = key 0 (matched roots,
    # score 3d) and key 1 with the opposite root (score about -0.98 d), so
    # o_1 = v_0 exactly.
    d = 4
    th = math.pi - 0.1
    u = th / (math.pi - th)                      # squash(u) = th
    q = np.array([[[[0.3] * d, [u] * d]]])
    k = np.array([[[[u] * d, [-u] * d]]])
    v = np.array([[[[1.0, 2.0], [-5.0, 7.0]]]])
    gamma = np.array([100.0])
    omega = np.full((1, d), math.pi / 4)
    phi = np.zeros((1, d))
    pq = O.featurize_ablation(q, gamma, omega, phi, 4)[0, 0]
    pk = O.featurize_ablation(k, gamma, omega, phi, 4)[0, 0]
    assert pq[1] @ pk[1] < -0.9 * d and abs(pq[1] @ pk[0] - 3 * d) < 1e-6
    for p in (1, 2, 4):
        o, D = O.attn_ablation(q, k, v, gamma, omega, phi, p, 4)
        assert np.allclose(o[0, 0, 1], v[0, 0, 0], atol=1e-12), (p, o[0, 0, 1])
        assert abs(D[0, 0, 1] - 1.0) < 1e-6     # (3d / 3d)^p from key 0 alone


def check_three_channel_score_range_and_shift():
    # s3 = d + sum_a cos(dtheta_a), in [0, 2d] (Notes §4.4, not the [-d, 3d] of
    # the printed comment); the printed ablation adds d and divides by 3d
    c = _small_case(seed=12, T=11, d=6)
    pq = O.featurize_ablation(c["q"], c["gamma"], c["omega"], c["phi"], 3)[0, 0]
    pk = O.featurize_ablation(c["k"], c["gamma"], c["omega"], c["phi"], 3)[0, 0]
    tq, _ = _angles(c, c["q"][0, 0])
    tk, _ = _angles(c, c["k"][0, 0])
    s = pq @ pk.T
    want = 6 + np.cos(tq[:, None, :] - tk[None, :, :]).sum(axis=-1)
    assert np.allclose(s, want, atol=1e-12)
    assert s.min() >= 0 and s.max() <= 12
    o0, D0 = O.attn_ablation(**c, p=2, channels=3)
    o1, D1 = O.attn_ablation(**c, p=2, channels=3, shift=6.0)
    mask = np.tril(np.ones((11, 11)))
    w = ((s + 6.0) / 18.0) ** 2 * mask
    assert np.allclose(D1[0, 0], w.sum(1), atol=1e-12)
    assert np.allclose(o1[0, 0], (w @ c["v"][0, 0]) / w.sum(1)[:, None], atol=1e-12)
    assert not np.allclose(o0, o1, atol=1e-3)    # the shift changes the distribution


def check_three_channel_p1_is_linear_attention():
    # without shift and clip the three-channel p = 1 form is a linear attention
    # over Phi3: the recurrence S += Phi3(k) v^T, z += Phi3(k) gives the same o
    c = _small_case(seed=13, B=2, T=10, d=3)
    o, D = O.attn_ablation(**c, p=1, channels=3, eps=0.7)
    pq = O.featurize_ablation(c["q"], c["gamma"], c["omega"], c["phi"], 3)
    pk = O.featurize_ablation(c["k"], c["gamma"], c["omega"], c["phi"], 3)
    B, H, T, F = pq.shape
    Sx = np.zeros((B, H, F, 2))
    zx = np.zeros((B, H, F))
    for t in range(T):
        Sx += pk[:, :, t, :, None] * c["v"][:, :, t, None, :]
        zx += pk[:, :, t]
        num = np.einsum("bhf,bhfe->bhe", pq[:, :, t], Sx)
        den = np.einsum("bhf,bhf->bh", pq[:, :, t], zx)
        assert np.allclose(o[:, :, t], num / (den + 0.7 * 2 * 3)[..., None], atol=1e-12)
        assert np.allclose(D[:, :, t] * 6, den, atol=1e-12)


def check_ablation_single_token_and_constant_values():
    for ch in (4, 3):
        c = _small_case(seed=14, T=1)
        o, _ = O.attn_ablation(**c, p=2, channels=ch)
        assert np.allclose(o, c["v"], atol=1e-12)
        c = _small_case(seed=15, T=8)
        c["v"] = np.broadcast_to(np.array([0.5, -2.0]), c["v"].shape).copy()
        o, _ = O.attn_ablation(**c, p=3, channels=ch)
        # the four-channel scores of these inputs are positive, so no row is empty
        assert np.allclose(o, c["v"], atol=1e-12)


ALL_CHECKS += [
    check_four_channel_kernel_closed_form,
    check_four_channel_hard_roots,
    check_four_channel_clip,
    check_three_channel_score_range_and_shift,
    check_three_channel_p1_is_linear_attention,
    check_ablation_single_token_and_constant_values,
]


# --------------------------------------------------------------------------
# Rate parameterisation lambda = 0.01 tanh(lambda_raw) (Notes §2.2) and the
# eps scale of the two normalisation conventions (Notes §2.7)
# --------------------------------------------------------------------------

def check_rate_parameterisation():
    x = np.array([0.0, 1e-8, -1e-8, 40.0, -40.0, 0.5493061443340549])  # atanh(0.5) last
    lam = O.rate_from_raw(x)
    assert lam[0] == 0.0 and abs(lam[1] - 1e-10) < 1e-20      # slope 0.01 at the origin
    assert abs(lam[3] - 0.01) < 1e-15 and abs(lam[4] + 0.01) < 1e-15   # saturates at +-0.01
    assert abs(lam[5] - 0.005) < 1e-15
    g = _rng(21)
    raw = g.standard_normal(50)
    dphi = g.standard_normal(50)
    h = 1e-6
    fd = (O.rate_from_raw(raw + h) - O.rate_from_raw(raw - h)) / (2 * h) * dphi
    assert np.allclose(O.rate_from_raw_grad(raw, dphi), fd, rtol=1e-7, atol=1e-14)


def check_eps_conventions():
    # c = 4d + 1e-6 (parallel code) and 4d x 1e-6 (recurrence notebook), d = 64
    assert abs(O.eps_raw(1.0, 64, 0) - 256.000001) < 1e-9
    assert abs(O.eps_raw(1.0, 64, 1) - 2.56e-4) < 1e-16
    # the raw-score form with eps_raw equals the scaled form with eps (p = 1)
    c = _small_case(seed=22, T=6)
    d = c["q"].shape[-1]
    cc = 4.0 * d + 1e-6
    o_raw, _ = O.attn_quadratic(**c, eps=O.eps_raw(0.3, d, 0))
    pq = O.featurize(c["q"], c["gamma"], c["omega"], c["phi"])[0, 0]
    pk = O.featurize(c["k"], c["gamma"], c["omega"], c["phi"])[0, 0]
    w = (pq @ pk.T) / cc * np.tril(np.ones((6, 6)))
    o_scaled = (w @ c["v"][0, 0]) / (w.sum(1) + 0.3)[:, None]
    assert np.allclose(o_raw[0, 0], o_scaled, atol=1e-12)


ALL_CHECKS += [check_rate_parameterisation, check_eps_conventions]


# --------------------------------------------------------------------------
# Harmonic features (Appendix B of the notes)
# --------------------------------------------------------------------------

def check_harmonic_one_is_six_channel():
    c = _small_case(seed=31, T=7, d=4)
    a = O.featurize_harmonic(c["q"], c["gamma"], c["omega"], c["phi"], 1, pos0=5)
    b = O.featurize(c["q"], c["gamma"], c["omega"], c["phi"], pos0=5)
    assert np.allclose(a, b, atol=1e-15)
    assert O.harmonic_channels(1) == 6 and O.harmonic_channels(3) == 14


def check_harmonic_kernel_closed_form():
    # Phi_N(q).Phi_N(k) = sum_a (1 + r_q r_k)(1 + sum_{n<=N} cos(n dtheta_a))
    c = _small_case(seed=32, T=6, d=3)
    for N in (2, 3):
        pq = O.featurize_harmonic(c["q"], c["gamma"], c["omega"], c["phi"], N)[0, 0]
        pk = O.featurize_harmonic(c["k"], c["gamma"], c["omega"], c["phi"], N)[0, 0]
        tq, rq = _angles(c, c["q"][0, 0])
        tk, rk = _angles(c, c["k"][0, 0])
        for i in range(6):
            for j in range(6):
                dth = tq[i] - tk[j]
                ang = 1.0 + sum(np.cos(n * dth) for n in range(1, N + 1))
                want = np.sum((1.0 + rq[i] * rk[j]) * ang)
                assert abs(pq[i] @ pk[j] - want) < 1e-12, (N, i, j)


def check_harmonic_quadratic_equals_recurrent_and_decode():
    c = _small_case(seed=33, B=2, T=9, d=3)
    for N in (2, 3):
        o, D = O.attn_harmonic(**c, N=N, eps=0.4, pos0=3)
        F = O.harmonic_channels(N) * 3
        Sx = np.zeros((2, 2, F, 2))
        zx = np.zeros((2, 2, F))
        for t in range(9):
            g = np.repeat(c["gamma"][None], 2, 0).reshape(-1)
            om = np.repeat(c["omega"][None], 2, 0).reshape(-1, 3)
            ph = np.repeat(c["phi"][None], 2, 0).reshape(-1, 3)
            Sn, zn, on = O.decode_step_harmonic(
                Sx.reshape(4, F, 2), zx.reshape(4, F), c["q"][:, :, t].reshape(4, 3),
                c["k"][:, :, t].reshape(4, 3), c["v"][:, :, t].reshape(4, 2), g, om, ph,
                np.full(4, 3 + t), N, eps=0.4)
            Sx, zx = Sn.reshape(2, 2, F, 2), zn.reshape(2, 2, F)
            assert np.allclose(on.reshape(2, 2, 2), o[:, :, t], atol=1e-12), (N, t)
        S_ref, z_ref = O.final_state_harmonic(c["k"], c["v"], c["gamma"], c["omega"], c["phi"], N,
                                              pos0=3)
        assert np.allclose(Sx, S_ref, atol=1e-12) and np.allclose(zx, z_ref, atol=1e-12)


def check_harmonic_channels_double_angle():
    # the second harmonic channels obey cos 2x = 2 cos^2 x - 1 and sin 2x =
    # 2 sin x cos x in terms of the first ones, and the root block is r times
    # the angle block (channel order [A, r A] per dimension)
    c = _small_case(seed=34, T=5, d=3)
    f = O.featurize_harmonic(c["k"], c["gamma"], c["omega"], c["phi"], 2, pos0=11)
    f = f.reshape(f.shape[:-1] + (3, 10))
    cos1, sin1, cos2, sin2 = f[..., 1], f[..., 2], f[..., 3], f[..., 4]
    assert np.allclose(cos2, 2 * cos1 ** 2 - 1, atol=1e-13)
    assert np.allclose(sin2, 2 * sin1 * cos1, atol=1e-13)
    assert np.allclose(f[..., 0], 1.0)
    r = f[..., 5]
    assert np.allclose(f[..., 5:], r[..., None] * f[..., :5], atol=1e-15)


def check_harmonic_state_size():
    # N = 1 is the paper's 14,376,960 bytes; each harmonic adds 4d features
    assert O.state_bytes_harmonic(12, 12, 64, 64, 1) == 14376960
    assert O.state_bytes_harmonic(12, 12, 64, 64, 2) == 12 * 12 * (640 * 64 + 640) * 4


def _harmonic_loss(c, N, dO, pos0, eps, S0, z0):
    o, _ = O.attn_harmonic(c["q"], c["k"], c["v"], c["gamma"], c["omega"], c["phi"], N,
                           pos0=pos0, eps=eps, S0=S0, z0=z0)
    return float((o * dO).sum())


def check_harmonic_backward_finite_differences():
    # every gradient of the harmonic map's attention against central finite
    # differences of the forward, for N = 2 and 3, with and without a history
    c = _small_case(35, B=1, H=2, T=6, d=2, dv=2, phi_scale=0.8)
    g = _rng(36)
    dO = g.standard_normal(c["v"].shape)
    for N in (2, 3):
        S0, z0 = O.final_state_harmonic(g.standard_normal(c["k"].shape),
                                        g.standard_normal(c["v"].shape), c["gamma"], c["omega"],
                                        c["phi"], N, pos0=-6)
        for pos0, eps, st in ((3, 0.0, False), (0, 0.3, True)):
            S = S0 if st else None
            Z = z0 if st else None
            grads = O.attn_harmonic_backward(c["q"], c["k"], c["v"], c["gamma"], c["omega"],
                                             c["phi"], dO, N, pos0=pos0, eps=eps, S0=S, z0=Z)
            h = 1e-6
            for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("gamma", "dgamma"),
                                ("omega", "domega"), ("phi", "dphi")):
                x = c[name]
                num = np.zeros_like(x)
                for idx in np.ndindex(x.shape):
                    old = x[idx]
                    x[idx] = old + h
                    lp = _harmonic_loss(c, N, dO, pos0, eps, S, Z)
                    x[idx] = old - h
                    lm = _harmonic_loss(c, N, dO, pos0, eps, S, Z)
                    x[idx] = old
                    num[idx] = (lp - lm) / (2 * h)
                err = np.abs(num - grads[gname]).max() / max(1e-3, np.abs(num).max())
                assert err < 1e-6, (N, name, err)


def check_harmonic_one_backward_is_six_channel_backward():
    c = _small_case(37, B=2, H=2, T=8, d=3)
    dO = _rng(38).standard_normal(c["v"].shape)
    a = O.attn_harmonic_backward(**c, dO=dO, N=1, pos0=5, eps=0.2)
    b = O.attn_backward(**c, dO=dO, pos0=5, eps=0.2)
    for key in ("dq", "dk", "dv", "dgamma", "domega", "dphi"):
        assert np.allclose(a[key], b[key], rtol=1e-12, atol=1e-12), key


ALL_CHECKS += [check_harmonic_one_is_six_channel, check_harmonic_kernel_closed_form,
               check_harmonic_quadratic_equals_recurrent_and_decode, check_harmonic_state_size,
               check_harmonic_channels_double_angle, check_harmonic_backward_finite_differences,
               check_harmonic_one_backward_is_six_channel_backward]


# --------------------------------------------------------------------------
# Attention stack: the stepped recurrence through all layers equals the
# parallel form (the pages' parallel-vs-recurrent agreement, Notes §2.7)
# --------------------------------------------------------------------------

def _stack_case(seed=41, B=2, T=6, L=3, heads=2, d=3):
    g = _rng(seed)
    Dm = heads * d
    return dict(X=g.standard_normal((B, T, Dm)),
                Wqkv=g.standard_normal((L, Dm, 3 * Dm)) / math.sqrt(Dm),
                Wo=g.standard_normal((L, Dm, Dm)) / math.sqrt(Dm),
                gamma=g.uniform(1.0, 5.0, (L, heads)),
                omega=g.uniform(-math.pi, math.pi, (L, heads, d)),
                phi=g.uniform(0.0, 0.3, (L, heads, d)), heads=heads)


def check_stack_recurrent_equals_parallel():
    c = _stack_case()
    B, T, Dm = c["X"].shape
    L, heads = c["Wqkv"].shape[0], c["heads"]
    d = Dm // heads
    Y = O.stack_parallel(**c, pos0=7, eps=0.3)
    S = np.zeros((L, B * heads, 6 * d, d))
    z = np.zeros((L, B * heads, 6 * d))
    for t in range(T):
        y, S, z = O.stack_decode_step(c["X"][:, t], c["Wqkv"], c["Wo"], S, z, c["gamma"],
                                      c["omega"], c["phi"], heads, np.full(B, 7 + t), eps=0.3)
        assert np.allclose(y, Y[:, t], atol=1e-12), t


def check_stack_single_layer_is_one_attention():
    # one layer with identity-like projections: x + attention(x) Wo, directly
    c = _stack_case(seed=42, L=1)
    B, T, Dm = c["X"].shape
    heads, d = c["heads"], Dm // c["heads"]
    qkv = c["X"] @ c["Wqkv"][0]
    sp = lambda m: m.reshape(B, T, heads, d).transpose(0, 2, 1, 3)  # noqa: E731
    o, _ = O.attn_recurrent(sp(qkv[..., :Dm]), sp(qkv[..., Dm:2 * Dm]), sp(qkv[..., 2 * Dm:]),
                            c["gamma"][0], c["omega"][0], c["phi"][0])[:2]
    want = c["X"] + o.transpose(0, 2, 1, 3).reshape(B, T, Dm) @ c["Wo"][0]
    assert np.allclose(O.stack_parallel(**c), want, atol=1e-12)


ALL_CHECKS += [check_stack_recurrent_equals_parallel, check_stack_single_layer_is_one_attention]
