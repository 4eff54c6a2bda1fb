"""Plant plausible mistakes in the float64 oracle (on the CPU, through
monkeypatching) and show that the pins of ``oracle_pins`` catch every one.

A pin set that cannot tell the oracle from a subtly wrong variant would not
pin it; each mutation below is a mistake that a transcription of the pages
could plausibly make."""
import numpy as np
import pytest

import oracle.sanatan_oracle as O
import oracle_pins as P

_orig = {n: getattr(O, n) for n in ("squash", "soft_root", "rotate", "features_from_angles",
                                     "attn_quadratic", "attn_recurrent", "attn_backward",
                                     "_feature_vjp", "state_bytes", "featurize", "attn_power",
                                     "attn_power_backward", "attn_ablation",
                                     "features4_from_angles", "ablation_scale",
                                     "features_harmonic_from_angles", "stack_decode_step",
                                     "_feature_vjp_harmonic", "attn_harmonic_backward")}


def m_squash_no_abs(u):
    u = np.asarray(u, dtype=np.float64)
    return np.pi * u / (1.0 + u)


def m_squash_square(u):
    u = np.asarray(u, dtype=np.float64)
    return np.pi * u / (1.0 + u * u)


def m_root_sign(theta, gamma, omega):
    x = np.asarray(theta, dtype=np.float64) + omega
    return np.tanh(gamma * (np.sin(x) - np.cos(x)))


def m_root_no_omega(theta, gamma, omega):
    x = np.asarray(theta, dtype=np.float64)
    return np.tanh(gamma * (np.cos(x) - np.sin(x)))


def m_rotate_minus(theta, t, phi):
    return np.asarray(theta, dtype=np.float64) - np.asarray(t, dtype=np.float64) * phi


def m_rotate_scaled(theta, t, phi):
    return np.asarray(theta, dtype=np.float64) + 2.0 * np.asarray(t, dtype=np.float64) * phi


def m_features_dropped(theta_rot, r):
    c, s = np.cos(theta_rot), np.sin(theta_rot)
    blk = np.stack([np.ones_like(c), c, s, r, r * c, 0.0 * s], axis=-1)
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * 6,))


def m_features_swapped(theta_rot, r):
    c, s = np.cos(theta_rot), np.sin(theta_rot)
    blk = np.stack([np.ones_like(c), s, c, r, r * s, r * c], axis=-1)
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * 6,))


def m_featurize_root_after_rotation(u, gamma, omega, phi, pos0=0):
    u = np.asarray(u, dtype=np.float64)
    B, H, T, d = u.shape
    g = np.asarray(gamma, dtype=np.float64).reshape(1, H, 1, 1)
    om = np.asarray(omega, dtype=np.float64).reshape(1, H, 1, d)
    ph = np.asarray(phi, dtype=np.float64).reshape(1, H, 1, d)
    t = O.positions(T, pos0).astype(np.float64).reshape(1, 1, T, 1)
    th_rot = O.rotate(O.squash(u), t, ph)
    return O.features_from_angles(th_rot, O.soft_root(th_rot, g, om))


def _quadratic_mask(offset):
    def f(q, k, v, gamma, omega, phi, pos0=0, eps=0.0, S0=None, z0=None):
        pq = O.featurize(q, gamma, omega, phi, pos0)
        pk = O.featurize(k, gamma, omega, phi, pos0)
        v = np.asarray(v, dtype=np.float64)
        B, H, T, _ = pq.shape
        mask = np.tril(np.ones((T, T)), offset)
        o = np.zeros(v.shape[:3] + (v.shape[-1],))
        D = np.zeros((B, H, T))
        for b in range(B):
            for h in range(H):
                s = O.pair_kernel(pq[b, h], pk[b, h]) * mask
                num, den = s @ v[b, h], s.sum(1)
                if S0 is not None:
                    num = num + pq[b, h] @ S0[b, h]
                    den = den + pq[b, h] @ z0[b, h]
                o[b, h] = num / (den + eps)[:, None]
                D[b, h] = den
        return o, D
    return f


def m_recurrent_read_first(q, k, v, gamma, omega, phi, pos0=0, eps=0.0, S0=None, z0=None):
    pq = O.featurize(q, gamma, omega, phi, pos0)
    pk = O.featurize(k, gamma, omega, phi, pos0)
    v = np.asarray(v, dtype=np.float64)
    B, H, T, F = pq.shape
    S = np.zeros((B, H, F, v.shape[-1])) if S0 is None else S0.copy()
    z = np.zeros((B, H, F)) if z0 is None else z0.copy()
    o = np.zeros((B, H, T, v.shape[-1]))
    D = np.zeros((B, H, T))
    for t in range(T):
        num = np.einsum("bhf,bhfe->bhe", pq[:, :, t], S)
        den = np.einsum("bhf,bhf->bh", pq[:, :, t], z)
        o[:, :, t] = num / (den + eps + 1e-300)[..., None]
        D[:, :, t] = den
        S = S + pk[:, :, t, :, None] * v[:, :, t, None, :]
        z = z + pk[:, :, t]
    return o, D, S, z


def m_eps_outside(q, k, v, gamma, omega, phi, pos0=0, eps=0.0, S0=None, z0=None):
    o, D = _orig["attn_quadratic"](q, k, v, gamma, omega, phi, pos0, 0.0, S0, z0)
    return o + eps, D


def _vjp_mutant(kind):
    def f(parts, dphi):
        B, H, T, F = dphi.shape
        d = F // 6
        dp = dphi.reshape(B, H, T, d, 6)
        r, c, s = parts["r"], parts["c"], parts["s"]
        dc = dp[..., 1] + r * dp[..., 4]
        ds = dp[..., 2] + r * dp[..., 5]
        dr = dp[..., 3] + c * dp[..., 4] + s * dp[..., 5]
        if kind == "rot_sign":
            dth_rot = s * dc - c * ds
        else:
            dth_rot = -s * dc + c * ds
        sech2 = 1.0 if kind == "no_sech2" else 1.0 - r * r
        dpre = dr * sech2
        dtheta = dth_rot + dpre * parts["g"] * parts["gpx"]
        u = parts["u"]
        if kind == "squash_deriv":
            du = dtheta * np.pi / (1.0 + np.abs(u))
        else:
            du = dtheta * np.pi / (1.0 + np.abs(u)) ** 2
        dgamma = (dpre * parts["gx"]).sum(axis=(0, 2, 3))
        domega = (dpre * parts["g"] * parts["gpx"]).sum(axis=(0, 2))
        dphi_rate = (dth_rot * parts["t"]).sum(axis=(0, 2))
        return du, dgamma, domega, dphi_rate
    return f


def m_backward_sign_error(q, k, v, gamma, omega, phi, dO, pos0=0, eps=0.0, S0=None, z0=None):
    # a sign slip on the upstream gradient everywhere but dv
    g = _orig["attn_backward"](q, k, v, gamma, omega, phi, -np.asarray(dO), pos0, eps, S0, z0)
    g["dv"] = -g["dv"]
    return g


def m_state_bytes_no_z(layers, heads, d, dv, bytes_per_float=4):
    return layers * heads * (6 * d * dv) * bytes_per_float


def _power_mutant(kind):
    def f(q, k, v, gamma, omega, phi, p, pos0=0, eps=0.0):
        if kind == "exponent":
            return _orig["attn_power"](q, k, v, gamma, omega, phi, int(p) + 1, pos0, eps)
        # kind == "no_scale": (s)^p instead of (s / 4d)^p
        pq = O.featurize(q, gamma, omega, phi, pos0)
        pk = O.featurize(k, gamma, omega, phi, pos0)
        v = np.asarray(v, dtype=np.float64)
        B, H, T, _ = pq.shape
        mask = np.tril(np.ones((T, T)))
        o = np.zeros((B, H, T, v.shape[-1]))
        D = np.zeros((B, H, T))
        for b in range(B):
            for h in range(H):
                w = O.pair_kernel(pq[b, h], pk[b, h]) ** int(p) * mask
                den = w.sum(1)
                o[b, h] = (w @ v[b, h]) / (den + eps)[:, None]
                D[b, h] = den
        return o, D
    return f


def _power_bwd_mutant(kind):
    # the gradient of the powered weight taken as if p were 1 (the factor
    # p x^(p-1) dropped), or the value gradient taken with the raw scores
    def f(q, k, v, gamma, omega, phi, dO, p, pos0=0, eps=0.0):
        g = _orig["attn_power_backward"](q, k, v, gamma, omega, phi, dO, p, pos0, eps)
        if kind == "no_chain_factor":
            g1 = _orig["attn_power_backward"](q, k, v, gamma, omega, phi, dO, 1, pos0, eps)
            for n in ("dq", "dk", "dgamma", "domega", "dphi"):
                g[n] = g1[n]
        else:  # "dv_unpowered"
            g1 = _orig["attn_power_backward"](q, k, v, gamma, omega, phi, dO, 1, pos0, eps)
            g["dv"] = g1["dv"]
        return g
    return f


def _ablation_mutant(kind):
    orig = _orig["attn_ablation"]

    def f(q, k, v, gamma, omega, phi, p, channels, shift=0.0, pos0=0, eps=0.0):
        if kind == "no_clip" and channels == 4:
            pq = O.featurize_ablation(q, gamma, omega, phi, 4, pos0)
            pk = O.featurize_ablation(k, gamma, omega, phi, 4, pos0)
            T = pq.shape[2]
            mask = np.tril(np.ones((T, T)))
            o = np.zeros(np.asarray(v).shape)
            D = np.zeros(pq.shape[:3])
            for b in range(pq.shape[0]):
                for h in range(pq.shape[1]):
                    w = ((pq[b, h] @ pk[b, h].T) / (3.0 * (pq.shape[-1] // 4))) ** p * mask
                    D[b, h] = w.sum(1)
                    o[b, h] = (w @ np.asarray(v)[b, h]) / (D[b, h] + eps)[:, None]
            return o, D
        if kind == "shift_ignored":
            return orig(q, k, v, gamma, omega, phi, p, channels, 0.0, pos0, eps)
        return orig(q, k, v, gamma, omega, phi, p, channels, shift, pos0, eps)
    return f


def m_features4_unrooted(theta_rot, r):
    c, s = np.cos(theta_rot), np.sin(theta_rot)
    blk = np.stack([np.ones_like(c), r, c, s], axis=-1)
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * 4,))


def m_ablation_scale_4d(channels, d, shift=0.0):
    return 4.0 * d


def m_harmonic_unrotated_multiple(theta_rot, r, N):
    # a plausible slip: the n-th harmonic of the rotated angle taken as
    # n theta + t phi (rotation not multiplied) -- emulated by using n = 1 rotation
    th = np.asarray(theta_rot, dtype=np.float64)
    ang = [np.ones_like(th)]
    for n in range(1, N + 1):
        ang += [np.cos(th * (1 if n == 1 else n) + (0.1 if n > 1 else 0.0)),
                np.sin(th * (1 if n == 1 else n) + (0.1 if n > 1 else 0.0))]
    A = np.stack(ang, axis=-1)
    blk = np.concatenate([A, np.asarray(r)[..., None] * A], axis=-1)
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * blk.shape[-1],))


def m_harmonic_no_label_block(theta_rot, r, N):
    th = np.asarray(theta_rot, dtype=np.float64)
    ang = [np.ones_like(th)]
    for n in range(1, N + 1):
        ang += [np.cos(n * th), np.sin(n * th)]
    A = np.stack(ang, axis=-1)
    blk = np.concatenate([A, A], axis=-1)
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * blk.shape[-1],))


def _harmonic_vjp_mutant(kind):
    # the harmonic chain rule with one plausible slip, made by handing the
    # correct chain rule a transformed cotangent:
    #   no_multiple:    d(cos n th)/dth taken as -sin n th (the factor n dropped),
    #   no_label_scale: the label block r A_m passed to dA_m without its r
    def vjp(u, gamma, omega, phi, N, pos0, dphi):
        dphi = np.asarray(dphi, dtype=np.float64)
        B, H, T, F = dphi.shape
        kA = 2 * N + 1
        dp = dphi.reshape(B, H, T, F // (2 * kA), 2, kA).copy()
        if kind == "no_multiple":
            for n in range(2, N + 1):
                dp[..., :, 2 * n - 1] /= n
                dp[..., :, 2 * n] /= n
        else:
            r = O._feature_parts(u, gamma, omega, phi, pos0)["r"]
            dp[..., 0, :] += (1.0 - r[..., None]) * dp[..., 1, :]
        return _orig["_feature_vjp_harmonic"](u, gamma, omega, phi, N, pos0,
                                              dp.reshape(dphi.shape))
    return vjp


def m_harmonic_backward_dv_unmasked(q, k, v, gamma, omega, phi, dO, N, pos0=0, eps=0.0, S0=None,
                                    z0=None):
    # dv summed over every query instead of the causal ones t >= j
    g = dict(_orig["attn_harmonic_backward"](q, k, v, gamma, omega, phi, dO, N, pos0, eps, S0,
                                             z0))
    pq = O.featurize_harmonic(q, gamma, omega, phi, N, pos0)
    pk = O.featurize_harmonic(k, gamma, omega, phi, N, pos0)
    o, D = O.attn_harmonic(q, k, v, gamma, omega, phi, N, pos0=pos0, eps=eps, S0=S0, z0=z0)
    dN = np.asarray(dO, dtype=np.float64) / (D + eps)[..., None]
    s = np.matmul(pq, np.swapaxes(pk, -1, -2))
    g["dv"] = np.matmul(np.swapaxes(s, -1, -2), dN)
    return g


def m_stack_no_residual(x, Wqkv, Wo, S, z, gamma, omega, phi, heads, pos, eps=0.0):
    # the residual dropped: x <- a Wo
    x = np.asarray(x, dtype=np.float64)
    B, Dm = x.shape
    d = Dm // heads
    S = np.array(S, dtype=np.float64)
    z = np.array(z, dtype=np.float64)
    sp_ = np.repeat(np.asarray(pos, dtype=np.int64), heads)
    for l in range(np.asarray(Wqkv).shape[0]):
        qkv = x @ Wqkv[l]
        g = np.tile(gamma[l], B)
        om = np.tile(omega[l], (B, 1))
        ph = np.tile(phi[l], (B, 1))
        S[l], z[l], o = O.decode_step(S[l], z[l], qkv[:, :Dm].reshape(-1, d),
                                      qkv[:, Dm:2 * Dm].reshape(-1, d),
                                      qkv[:, 2 * Dm:].reshape(-1, d), g, om, ph, sp_, eps=eps)
        x = o.reshape(B, Dm) @ Wo[l]
    return x, S, z


MUTANTS = {
    "squash_no_abs": ("squash", m_squash_no_abs),
    "squash_square": ("squash", m_squash_square),
    "root_sign": ("soft_root", m_root_sign),
    "root_no_omega": ("soft_root", m_root_no_omega),
    "rotate_minus": ("rotate", m_rotate_minus),
    "rotate_scaled": ("rotate", m_rotate_scaled),
    "features_dropped_channel": ("features_from_angles", m_features_dropped),
    "features_swapped_cos_sin": ("features_from_angles", m_features_swapped),
    "root_from_rotated_angle": ("featurize", m_featurize_root_after_rotation),
    "mask_strict": ("attn_quadratic", _quadratic_mask(-1)),
    "mask_one_future": ("attn_quadratic", _quadratic_mask(1)),
    "recurrent_read_before_write": ("attn_recurrent", m_recurrent_read_first),
    "eps_outside_ratio": ("attn_quadratic", m_eps_outside),
    "vjp_rotation_sign": ("_feature_vjp", _vjp_mutant("rot_sign")),
    "vjp_missing_sech2": ("_feature_vjp", _vjp_mutant("no_sech2")),
    "vjp_squash_derivative": ("_feature_vjp", _vjp_mutant("squash_deriv")),
    "backward_flipped_upstream": ("attn_backward", m_backward_sign_error),
    "state_bytes_without_z": ("state_bytes", m_state_bytes_no_z),
    "power_exponent_off_by_one": ("attn_power", _power_mutant("exponent")),
    "power_without_4d_scale": ("attn_power", _power_mutant("no_scale")),
    "power_backward_no_chain_factor": ("attn_power_backward", _power_bwd_mutant("no_chain_factor")),
    "power_backward_dv_unpowered": ("attn_power_backward", _power_bwd_mutant("dv_unpowered")),
    "four_channel_without_clip": ("attn_ablation", _ablation_mutant("no_clip")),
    "three_channel_shift_ignored": ("attn_ablation", _ablation_mutant("shift_ignored")),
    "four_channel_angles_unrooted": ("features4_from_angles", m_features4_unrooted),
    "ablation_scale_4d": ("ablation_scale", m_ablation_scale_4d),
    "harmonic_phase_slip": ("features_harmonic_from_angles", m_harmonic_unrotated_multiple),
    "harmonic_without_root_label": ("features_harmonic_from_angles", m_harmonic_no_label_block),
    "stack_without_residual": ("stack_decode_step", m_stack_no_residual),
    "harmonic_vjp_without_multiple": ("_feature_vjp_harmonic", _harmonic_vjp_mutant("no_multiple")),
    "harmonic_vjp_label_unscaled": ("_feature_vjp_harmonic",
                                    _harmonic_vjp_mutant("no_label_scale")),
    "harmonic_backward_dv_unmasked": ("attn_harmonic_backward", m_harmonic_backward_dv_unmasked),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutation_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    caught = []
    for check in P.ALL_CHECKS:
        try:
            check()
        except (AssertionError, FloatingPointError, ZeroDivisionError, ValueError):
            caught.append(check.__name__)
    assert caught, f"no pin detects the planted mistake {name}"
