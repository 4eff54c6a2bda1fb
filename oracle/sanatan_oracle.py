"""Float64 CPU oracle for SANATAN root-parity gated angular attention: the
feature map, the p = 1 causal attention in its quadratic and recurrent forms,
the power-sharpened attention of eq. (8) at integer p, and their gradients,
the four- and three-channel ablation kernels, the harmonic feature map, and
the attention stack of several layers (parallel form and decode step).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The product path (the CUDA library and its Python binding) never
imports, links or calls anything here, and this module imports nothing from the
product package: the two share no code.

Every function is a plain, slow restatement of the method's definitions, taken
from "SANATAN: Root-Parity Gated Angular Attention with an Exact Constant-State
Recurrent Form" as summarised by its reading notes (page "SANATAN：根标签门控的
角度核、精确递推与修订后的实验证据", cited below as *Notes*) and by the author's
own post (cited as *Post*).  Section / equation numbers in brackets are those
of the paper as the notes give them.

Conventions (the readings taken where the pages leave a step open):
  * Shapes: q, k [B, H, T, d]; v [B, H, T, dv]; gamma [H]; omega, phi [H, d].
  * Positions are t = pos0 + i for the i-th token of the sequence.
  * Feature index inside Phi is 6*a + c with channel order
    c = 0..5 -> [1, cos th_rot, sin th_rot, r, r cos th_rot, r sin th_rot].
  * The causal mask includes the current token (state update, then read).
  * eps is added to the denominator in raw score units and defaults to 0.
  * omega is shared by q and k of a head; phi (the rotation rate, lambda on
    the pages) is a per-(head, dim) input, so any parameterisation of it
    (0.01 tanh(lambda_raw), 10000^(-a/d), ...) happens before this module.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force, finite differences and an independent
torch float64 autograd).  None is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Feature map: Notes §2.2-§2.3 [paper §§3.1-3.3, eqs. (2)-(6)]
# ---------------------------------------------------------------------------

N_CHANNELS = 6


def squash(u):
    """Angle squash theta = pi*u / (1 + |u|)  (Notes §2.2, eq. (2)).

    Maps every real component into the open interval (-pi, pi); it is close
    to pi*u near 0 and saturates towards +-pi for large |u|.
    """
    u = np.asarray(u, dtype=np.float64)
    return np.pi * u / (1.0 + np.abs(u))


def soft_root(theta, gamma, omega):
    """Soft root label r = tanh(gamma*(cos(theta+omega) - sin(theta+omega)))
    (Notes §2.2, eq. (3)).  ``theta`` is the content angle BEFORE the temporal
    rotation: the label is not recomputed after the rotation (Notes §2.2,
    the remark after eq. (4))."""
    x = np.asarray(theta, dtype=np.float64) + omega
    return np.tanh(gamma * (np.cos(x) - np.sin(x)))


def rotate(theta, t, phi):
    """Temporal rotation theta_rot = theta + t*phi  (Notes §2.2, eq. (4)).

    ``t`` is an integer position, promoted exactly to float64; ``phi`` is the
    per-dimension rate (lambda on the pages)."""
    return np.asarray(theta, dtype=np.float64) + np.asarray(t, dtype=np.float64) * phi


def features_from_angles(theta_rot, r):
    """Six-channel block per dimension (Notes §2.3, eq. (6)):
    [1, cos th_rot, sin th_rot, r, r cos th_rot, r sin th_rot], concatenated
    over the dimensions so that channel c of dimension a sits at 6a + c."""
    c = np.cos(theta_rot)
    s = np.sin(theta_rot)
    one = np.ones_like(c)
    blk = np.stack([one, c, s, r, r * c, r * s], axis=-1)  # [..., d, 6]
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * N_CHANNELS,))


def positions(T, pos0):
    """t = pos0 + i, i = 0..T-1 (integer valued, exact in float64)."""
    return np.arange(T, dtype=np.int64) + np.int64(pos0)


def featurize(u, gamma, omega, phi, pos0=0):
    """Phi(u) for a [B, H, T, d] tensor of query or key components.

    gamma [H], omega [H, d], phi [H, d]; returns float64 [B, H, T, 6d].
    Steps: eq. (2) squash -> eq. (3) soft root from the un-rotated angle ->
    eq. (4) rotation by t*phi -> eq. (6) six channels."""
    u = np.asarray(u, dtype=np.float64)
    B, H, T, d = u.shape
    g = np.asarray(gamma, dtype=np.float64).reshape(1, H, 1, 1)
    om = np.asarray(omega, dtype=np.float64).reshape(1, H, 1, d)
    ph = np.asarray(phi, dtype=np.float64).reshape(1, H, 1, d)
    t = positions(T, pos0).astype(np.float64).reshape(1, 1, T, 1)
    theta = squash(u)
    r = soft_root(theta, g, om)
    th_rot = rotate(theta, t, ph)
    return features_from_angles(th_rot, r)


def pair_kernel(phi_q, phi_k):
    """Score s = <Phi(q), Phi(k)> (Notes §2.3, eq. (7)); the pages show it
    equals sum_a (1 + r_q r_k)(1 + cos(dtheta_a)), so 0 <= s <= 4d."""
    return np.asarray(phi_q) @ np.asarray(phi_k).T


# ---------------------------------------------------------------------------
# p = 1 causal normalised attention: Notes §2.6-§2.7 [paper §§3.4-3.5,
# eqs. (8)-(9)]
# ---------------------------------------------------------------------------


def _heads(x):
    return np.asarray(x, dtype=np.float64)


def attn_quadratic(q, k, v, gamma, omega, phi, pos0=0, eps=0.0, S0=None, z0=None):
    """Parallel (quadratic) causal form at p = 1 (Notes §2.6, eq. (8) with p=1):

        o_t = sum_{j<=t} s_tj v_j / (sum_{j<=t} s_tj + eps),  s_tj = Phi(q_t).Phi(k_j)

    plus, when an initial state (S0 [B,H,6d,dv], z0 [B,H,6d]) is given, the
    history it summarises: Phi(q_t).S0 is added to the numerator and
    Phi(q_t).z0 to the denominator (Notes §2.7: the state is the sum of the
    outer products of all earlier tokens).

    Returns o [B,H,T,dv] and the denominator D [B,H,T] (without eps)."""
    pq = featurize(q, gamma, omega, phi, pos0)
    pk = featurize(k, gamma, omega, phi, pos0)
    v = _heads(v)
    B, H, T, _ = pq.shape
    dv = v.shape[-1]
    mask = np.tril(np.ones((T, T)))
    o = np.zeros((B, H, T, dv))
    D = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            s = pair_kernel(pq[b, h], pk[b, h]) * mask
            num = s @ v[b, h]
            den = s.sum(axis=1)
            if S0 is not None:
                num = num + pq[b, h] @ _heads(S0)[b, h]
                den = den + pq[b, h] @ _heads(z0)[b, h]
            o[b, h] = num / (den + eps)[:, None]
            D[b, h] = den
    return o, D


def attn_power(q, k, v, gamma, omega, phi, p, pos0=0, eps=0.0):
    """Power-sharpened causal attention (Notes §2.6, eq. (8)), the parallel
    quadratic form used for training at p > 1:

        a_tj = (s_tj / 4d)^p / (sum_{l<=t} (s_tl / 4d)^p + eps),   o_t = sum_{j<=t} a_tj v_j

    with s_tj = Phi(q_t).Phi(k_j) and d the key dimension.  p is a positive
    integer; at p = 1 this is attn_quadratic with eps scaled by 4d.
    Returns o [B,H,T,dv] and D [B,H,T] = sum_{l<=t} (s_tl / 4d)^p (without eps)."""
    p = int(p)
    if p < 1:
        raise ValueError("p must be a positive integer")
    pq = featurize(q, gamma, omega, phi, pos0)
    pk = featurize(k, gamma, omega, phi, pos0)
    v = _heads(v)
    B, H, T, F = pq.shape
    d = F // N_CHANNELS
    mask = np.tril(np.ones((T, T)))
    o = np.zeros((B, H, T, v.shape[-1]))
    D = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            w = (pair_kernel(pq[b, h], pk[b, h]) / (4.0 * d)) ** p * mask
            den = w.sum(axis=1)
            o[b, h] = (w @ v[b, h]) / (den + eps)[:, None]
            D[b, h] = den
    return o, D


def attn_recurrent(q, k, v, gamma, omega, phi, pos0=0, eps=0.0, S0=None, z0=None):
    """Constant-state recurrent form (Notes §2.7, eq. (9)):

        S_t = S_{t-1} + Phi(k_t) v_t^T,   z_t = z_{t-1} + Phi(k_t),
        o_t = Phi(q_t)^T S_t / (Phi(q_t)^T z_t + eps)

    starting from zero (or from S0, z0).  The update precedes the read, which
    is the j <= t mask.  Returns o, D, and the final S [B,H,6d,dv], z [B,H,6d].
    """
    pq = featurize(q, gamma, omega, phi, pos0)
    pk = featurize(k, gamma, omega, phi, pos0)
    v = _heads(v)
    B, H, T, F = pq.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, F, dv)) if S0 is None else _heads(S0).copy()
    z = np.zeros((B, H, F)) if z0 is None else _heads(z0).copy()
    o = np.zeros((B, H, T, dv))
    D = np.zeros((B, H, T))
    for t in range(T):
        S += pk[:, :, t, :, None] * v[:, :, t, None, :]
        z += pk[:, :, t, :]
        num = np.einsum("bhf,bhfe->bhe", pq[:, :, t, :], S)
        den = np.einsum("bhf,bhf->bh", pq[:, :, t, :], z)
        o[:, :, t, :] = num / (den + eps)[..., None]
        D[:, :, t] = den
    return o, D, S, z


def final_state(k, v, gamma, omega, phi, pos0=0, S0=None, z0=None):
    """S_T = S0 + sum_t Phi(k_t) v_t^T and z_T = z0 + sum_t Phi(k_t)
    (Notes §2.7: the definition of the state as a sum, written directly)."""
    pk = featurize(k, gamma, omega, phi, pos0)
    S = np.matmul(np.swapaxes(pk, -1, -2), _heads(v))   # sum_t Phi(k_t) v_t^T per head
    z = pk.sum(axis=2)
    if S0 is not None:
        S = S + _heads(S0)
        z = z + _heads(z0)
    return S, z


def attn_rows(q, k, v, gamma, omega, phi, rows, pos0=0, eps=0.0, b=0, h=0):
    """o_t and D_t of one (batch, head) at the selected row indices only,
    each computed straight from the definition of eq. (8) at p = 1 over its
    own causal prefix.  Used to check large problems one output at a time."""
    q1 = _heads(q)[b:b + 1, h:h + 1]
    k1 = _heads(k)[b:b + 1, h:h + 1]
    v1 = _heads(v)[b, h]
    g1 = np.asarray(gamma, dtype=np.float64)[h:h + 1]
    om1 = np.asarray(omega, dtype=np.float64)[h:h + 1]
    ph1 = np.asarray(phi, dtype=np.float64)[h:h + 1]
    pk = featurize(k1, g1, om1, ph1, pos0)[0, 0]
    out_o, out_D = [], []
    for i in rows:
        qi = q1[:, :, i:i + 1, :]
        pqi = featurize(qi, g1, om1, ph1, pos0 + i)[0, 0, 0]
        s = pk[: i + 1] @ pqi
        den = s.sum()
        out_o.append((s @ v1[: i + 1]) / (den + eps))
        out_D.append(den)
    return np.array(out_o), np.array(out_D)


def decode_step(S, z, q, k, v, gamma, omega, phi, pos, eps=0.0):
    """One token of the recurrence of eq. (9) for N independent slots.

    S [N, 6d, dv], z [N, 6d]; q, k [N, d]; v [N, dv]; gamma [N];
    omega, phi [N, d]; pos [N] integer positions.  Returns (S', z', o)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    N, d = q.shape
    g = np.asarray(gamma, dtype=np.float64).reshape(N, 1)
    om = np.asarray(omega, dtype=np.float64)
    ph = np.asarray(phi, dtype=np.float64)
    t = np.asarray(pos, dtype=np.int64).astype(np.float64).reshape(N, 1)

    def phi_of(u):
        th = squash(u)
        return features_from_angles(rotate(th, t, ph), soft_root(th, g, om))

    pq, pk = phi_of(q), phi_of(k)
    S = _heads(S) + pk[:, :, None] * np.asarray(v, dtype=np.float64)[:, None, :]
    z = _heads(z) + pk
    num = np.einsum("nf,nfe->ne", pq, S)
    den = np.einsum("nf,nf->n", pq, z)
    return S, z, num / (den + eps)[:, None]


# ---------------------------------------------------------------------------
# Backward.  The pages give no gradient; this is the chain rule through
# eqs. (2)-(4), (6) and (8) at p = 1, written for the quadratic causal form.
# ---------------------------------------------------------------------------


def _feature_parts(u, gamma, omega, phi, pos0):
    u = np.asarray(u, dtype=np.float64)
    B, H, T, d = u.shape
    g = np.asarray(gamma, dtype=np.float64).reshape(1, H, 1, 1)
    om = np.asarray(omega, dtype=np.float64).reshape(1, H, 1, d)
    ph = np.asarray(phi, dtype=np.float64).reshape(1, H, 1, d)
    t = positions(T, pos0).astype(np.float64).reshape(1, 1, T, 1)
    theta = squash(u)
    x = theta + om
    gx = np.cos(x) - np.sin(x)            # the pre-tanh coefficient of eq. (3)
    gpx = -np.sin(x) - np.cos(x)          # its derivative in theta (and omega)
    r = np.tanh(g * gx)
    th_rot = rotate(theta, t, ph)
    return dict(u=u, g=g, gx=gx, gpx=gpx, r=r, c=np.cos(th_rot), s=np.sin(th_rot), t=t)


def _feature_vjp(parts, dphi):
    """Pull dPhi [B,H,T,6d] back to du and the parameter gradients."""
    B, H, T, F = dphi.shape
    d = F // N_CHANNELS
    dp = dphi.reshape(B, H, T, d, N_CHANNELS)
    r, c, s = parts["r"], parts["c"], parts["s"]
    dc = dp[..., 1] + r * dp[..., 4]
    ds = dp[..., 2] + r * dp[..., 5]
    dr = dp[..., 3] + c * dp[..., 4] + s * dp[..., 5]
    dth_rot = -s * dc + c * ds                       # d/dtheta of (cos, sin)
    sech2 = 1.0 - r * r                              # tanh' = 1 - tanh^2
    dpre = dr * sech2                                # grad of gamma*g(theta+omega)
    dtheta = dth_rot + dpre * parts["g"] * parts["gpx"]
    u = parts["u"]
    du = dtheta * np.pi / (1.0 + np.abs(u)) ** 2     # d squash / du
    dgamma = (dpre * parts["gx"]).sum(axis=(0, 2, 3))
    domega = (dpre * parts["g"] * parts["gpx"]).sum(axis=(0, 2))
    dphi_rate = (dth_rot * parts["t"]).sum(axis=(0, 2))
    return du, dgamma, domega, dphi_rate


def attn_backward(q, k, v, gamma, omega, phi, dO, pos0=0, eps=0.0, S0=None, z0=None):
    """Gradients of sum(o * dO) for the quadratic form of ``attn_quadratic``.

    With N_t = sum_j s_tj v_j (+ Phi(q_t) S0), D_t = sum_j s_tj (+ Phi(q_t) z0),
    Dh_t = D_t + eps and o_t = N_t / Dh_t:
        dN_t = dO_t / Dh_t,          dD_t = -(dO_t . o_t) / Dh_t,
        ds_tj = [j <= t] (dN_t . v_j + dD_t),
        dv_j = sum_t [j <= t] s_tj dN_t,
        dPhi(q_t) = sum_j ds_tj Phi(k_j) (+ S0 dN_t + z0 dD_t),
        dPhi(k_j) = sum_t ds_tj Phi(q_t),
    then through the feature map.  Returns a dict with dq, dk, dv, dgamma,
    domega and dphi (the rate gradient)."""
    pq = featurize(q, gamma, omega, phi, pos0)
    pk = featurize(k, gamma, omega, phi, pos0)
    v = _heads(v)
    dO = _heads(dO)
    B, H, T, F = pq.shape
    mask = np.tril(np.ones((T, T)))
    dpq = np.zeros_like(pq)
    dpk = np.zeros_like(pk)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            s = pair_kernel(pq[b, h], pk[b, h]) * mask
            num = s @ v[b, h]
            den = s.sum(axis=1)
            if S0 is not None:
                num = num + pq[b, h] @ _heads(S0)[b, h]
                den = den + pq[b, h] @ _heads(z0)[b, h]
            dh = den + eps
            o = num / dh[:, None]
            dN = dO[b, h] / dh[:, None]
            dD = -(dO[b, h] * o).sum(axis=1) / dh
            ds = (dN @ v[b, h].T + dD[:, None]) * mask
            dv[b, h] = s.T @ dN
            dpq[b, h] = ds @ pk[b, h]
            if S0 is not None:
                dpq[b, h] += dN @ _heads(S0)[b, h].T + np.outer(dD, _heads(z0)[b, h])
            dpk[b, h] = ds.T @ pq[b, h]
    dq, dg_q, dom_q, dph_q = _feature_vjp(_feature_parts(q, gamma, omega, phi, pos0), dpq)
    dk, dg_k, dom_k, dph_k = _feature_vjp(_feature_parts(k, gamma, omega, phi, pos0), dpk)
    return dict(dq=dq, dk=dk, dv=dv, dgamma=dg_q + dg_k, domega=dom_q + dom_k,
                dphi=dph_q + dph_k)


def attn_power_backward(q, k, v, gamma, omega, phi, dO, p, pos0=0, eps=0.0):
    """Gradients of sum(o * dO) for ``attn_power`` (Notes §2.6, eq. (8)); the
    pages give no gradient, so this is the chain rule.  With
    w_tj = [j <= t] (s_tj / 4d)^p, D_t = sum_j w_tj, Dh_t = D_t + eps and
    o_t = sum_j w_tj v_j / Dh_t:
        dN_t = dO_t / Dh_t,          dD_t = -(dO_t . o_t) / Dh_t,
        dw_tj = [j <= t] (dN_t . v_j + dD_t),
        ds_tj = dw_tj p (s_tj / 4d)^(p-1) / 4d,
        dv_j = sum_t w_tj dN_t,
        dPhi(q_t) = sum_j ds_tj Phi(k_j),    dPhi(k_j) = sum_t ds_tj Phi(q_t),
    then through the feature map.  Returns the dict of ``attn_backward``."""
    p = int(p)
    if p < 1:
        raise ValueError("p must be a positive integer")
    pq = featurize(q, gamma, omega, phi, pos0)
    pk = featurize(k, gamma, omega, phi, pos0)
    v = _heads(v)
    dO = _heads(dO)
    B, H, T, F = pq.shape
    c4d = 4.0 * (F // N_CHANNELS)
    mask = np.tril(np.ones((T, T)))
    dpq = np.zeros_like(pq)
    dpk = np.zeros_like(pk)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            x = pair_kernel(pq[b, h], pk[b, h]) / c4d
            w = x ** p * mask
            dh = w.sum(axis=1) + eps
            o = (w @ v[b, h]) / dh[:, None]
            dN = dO[b, h] / dh[:, None]
            dD = -(dO[b, h] * o).sum(axis=1) / dh
            dw = (dN @ v[b, h].T + dD[:, None]) * mask
            ds = dw * p * x ** (p - 1) / c4d
            dv[b, h] = w.T @ dN
            dpq[b, h] = ds @ pk[b, h]
            dpk[b, h] = ds.T @ pq[b, h]
    dq, dg_q, dom_q, dph_q = _feature_vjp(_feature_parts(q, gamma, omega, phi, pos0), dpq)
    dk, dg_k, dom_k, dph_k = _feature_vjp(_feature_parts(k, gamma, omega, phi, pos0), dpk)
    return dict(dq=dq, dk=dk, dv=dv, dgamma=dg_q + dg_k, domega=dom_q + dom_k,
                dphi=dph_q + dph_k)


# ---------------------------------------------------------------------------
# Ablation kernels: the four-channel map (Notes §2.5, "四通道为什么是另一种核")
# and the three-channel map of the root-ablation (Notes §4.4, the remark on the
# three-channel comparison), both used in the power-sharpened parallel form
# ---------------------------------------------------------------------------


def features4_from_angles(theta_rot, r):
    """Four-channel block per dimension (Notes §2.5): [1, r, r cos th_rot,
    r sin th_rot] -- the six-channel block without the separate cos, sin --
    concatenated so that channel c of dimension a sits at 4a + c."""
    c = np.cos(theta_rot)
    s = np.sin(theta_rot)
    one = np.ones_like(c)
    blk = np.stack([one, r, r * c, r * s], axis=-1)
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * 4,))


def features3_from_angles(theta_rot):
    """Three-channel block per dimension (Notes §4.4): [1, cos th_rot,
    sin th_rot] (no root channel), channel c of dimension a at 3a + c."""
    c = np.cos(theta_rot)
    s = np.sin(theta_rot)
    blk = np.stack([np.ones_like(c), c, s], axis=-1)
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * 3,))


def featurize_ablation(u, gamma, omega, phi, channels, pos0=0):
    """The four- or three-channel features of a [B, H, T, d] tensor, through
    the same squash, soft root (un-rotated angle) and rotation as ``featurize``."""
    u = np.asarray(u, dtype=np.float64)
    B, H, T, d = u.shape
    g = np.asarray(gamma, dtype=np.float64).reshape(1, H, 1, 1)
    om = np.asarray(omega, dtype=np.float64).reshape(1, H, 1, d)
    ph = np.asarray(phi, dtype=np.float64).reshape(1, H, 1, d)
    t = positions(T, pos0).astype(np.float64).reshape(1, 1, T, 1)
    theta = squash(u)
    th_rot = rotate(theta, t, ph)
    if channels == 4:
        return features4_from_angles(th_rot, soft_root(theta, g, om))
    if channels == 3:
        return features3_from_angles(th_rot)
    raise ValueError("channels must be 4 or 3")


def ablation_scale(channels, d, shift=0.0):
    """The score scale c of the ablation weights: the largest score the map
    can give, 3d for the four-channel kernel (each dimension at most
    1 + 1 * 2) and 2d + shift for the three-channel one (d + sum cos <= 2d,
    the printed ablation divides s3 + d by 3d).  It cancels at eps = 0."""
    return 3.0 * d if channels == 4 else 2.0 * d + shift


def attn_ablation(q, k, v, gamma, omega, phi, p, channels, shift=0.0, pos0=0, eps=0.0):
    """Power-sharpened causal attention with an ablation kernel:

        four channels (Notes §2.5): s_tj = Phi4(q_t).Phi4(k_j), which can be
            negative; the total score is clipped, max(s, 0), before the power;
        three channels (Notes §4.4): s_tj = Phi3(q_t).Phi3(k_j) = d + sum_a
            cos(dtheta_a), in [0, 2d], plus ``shift`` (the printed ablation adds
            d; the fair ablation the notes ask for has shift 0);

        w_tj = [j <= t] (max(s_tj + shift, 0) / c)^p,   c = ablation_scale(...),
        o_t = sum_j w_tj v_j / (sum_j w_tj + eps).

    ``shift`` applies to the three-channel kernel only.  Returns o [B,H,T,dv]
    and D [B,H,T] = sum_j w_tj (without eps)."""
    p = int(p)
    if p < 1:
        raise ValueError("p must be a positive integer")
    if channels == 4 and shift != 0.0:
        raise ValueError("the four-channel kernel takes no shift")
    pq = featurize_ablation(q, gamma, omega, phi, channels, pos0)
    pk = featurize_ablation(k, gamma, omega, phi, channels, pos0)
    v = _heads(v)
    B, H, T, F = pq.shape
    c = ablation_scale(channels, F // channels, shift)
    mask = np.tril(np.ones((T, T)))
    o = np.zeros((B, H, T, v.shape[-1]))
    D = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            s = pair_kernel(pq[b, h], pk[b, h]) + shift
            w = (np.maximum(s, 0.0) / c) ** p * mask
            den = w.sum(axis=1)
            o[b, h] = (w @ v[b, h]) / (den + eps)[:, None]
            D[b, h] = den
    return o, D


# ---------------------------------------------------------------------------
# Harmonic features (Notes, "附录 B 的频谱展望": adding cos(n theta), sin(n theta)
# keeps the p = 1 form explicitly expandable, with more features and state)
# ---------------------------------------------------------------------------


def harmonic_channels(N):
    """Channels per dimension of the map with harmonics 1..N: the label block
    [1, r] times the angle block [1, cos th, sin th, ..., cos N th, sin N th]."""
    return 2 * (2 * N + 1)


def features_harmonic_from_angles(theta_rot, r, N):
    """Per dimension [A, r A] with A = [1, cos th, sin th, cos 2th, sin 2th, ...,
    cos N th, sin N th] of the rotated angle (channel l (2N + 1) + m of
    dimension a at index a * 2(2N+1) + l (2N + 1) + m).  N = 1 is the
    six-channel block of eq. (6)."""
    th = np.asarray(theta_rot, dtype=np.float64)
    ang = [np.ones_like(th)]
    for n in range(1, N + 1):
        ang += [np.cos(n * th), np.sin(n * th)]
    A = np.stack(ang, axis=-1)
    blk = np.concatenate([A, np.asarray(r)[..., None] * A], axis=-1)
    return blk.reshape(blk.shape[:-2] + (blk.shape[-2] * blk.shape[-1],))


def featurize_harmonic(u, gamma, omega, phi, N, pos0=0):
    """The harmonic features of a [B, H, T, d] tensor: squash, soft root from
    the un-rotated angle, rotation, then features_harmonic_from_angles."""
    u = np.asarray(u, dtype=np.float64)
    B, H, T, d = u.shape
    g = np.asarray(gamma, dtype=np.float64).reshape(1, H, 1, 1)
    om = np.asarray(omega, dtype=np.float64).reshape(1, H, 1, d)
    ph = np.asarray(phi, dtype=np.float64).reshape(1, H, 1, d)
    t = positions(T, pos0).astype(np.float64).reshape(1, 1, T, 1)
    theta = squash(u)
    return features_harmonic_from_angles(rotate(theta, t, ph), soft_root(theta, g, om), N)


def attn_harmonic(q, k, v, gamma, omega, phi, N, pos0=0, eps=0.0, S0=None, z0=None):
    """Causal normalised attention at p = 1 with the harmonic map (the
    quadratic form of eq. (9)'s attention, s_tj = Phi_N(q_t).Phi_N(k_j)),
    with the history of a state (S0, z0) added as in attn_quadratic."""
    pq = featurize_harmonic(q, gamma, omega, phi, N, pos0)
    pk = featurize_harmonic(k, gamma, omega, phi, N, pos0)
    v = _heads(v)
    B, H, T, _ = pq.shape
    mask = np.tril(np.ones((T, T)))
    o = np.zeros((B, H, T, v.shape[-1]))
    D = np.zeros((B, H, T))
    for b in range(B):
        for h in range(H):
            s = (pq[b, h] @ pk[b, h].T) * mask
            num = s @ v[b, h]
            den = s.sum(axis=1)
            if S0 is not None:
                num = num + pq[b, h] @ _heads(S0)[b, h]
                den = den + pq[b, h] @ _heads(z0)[b, h]
            o[b, h] = num / (den + eps)[:, None]
            D[b, h] = den
    return o, D


def final_state_harmonic(k, v, gamma, omega, phi, N, pos0=0, S0=None, z0=None):
    """S = S0 + sum_t Phi_N(k_t) v_t^T, z = z0 + sum_t Phi_N(k_t)."""
    pk = featurize_harmonic(k, gamma, omega, phi, N, pos0)
    S = np.matmul(np.swapaxes(pk, -1, -2), _heads(v))
    z = pk.sum(axis=2)
    if S0 is not None:
        S = S + _heads(S0)
        z = z + _heads(z0)
    return S, z


def decode_step_harmonic(S, z, q, k, v, gamma, omega, phi, pos, N, eps=0.0):
    """One token of the recurrence with the harmonic map for N slots (the
    arguments of decode_step; S [n, F_N, dv], z [n, F_N])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    n, d = q.shape
    g = np.asarray(gamma, dtype=np.float64).reshape(n, 1)
    om = np.asarray(omega, dtype=np.float64)
    ph = np.asarray(phi, dtype=np.float64)
    t = np.asarray(pos, dtype=np.int64).astype(np.float64).reshape(n, 1)

    def phi_of(u):
        th = squash(u)
        return features_harmonic_from_angles(rotate(th, t, ph), soft_root(th, g, om), N)

    pq, pk = phi_of(q), phi_of(k)
    S = _heads(S) + pk[:, :, None] * np.asarray(v, dtype=np.float64)[:, None, :]
    z = _heads(z) + pk
    num = np.einsum("nf,nfe->ne", pq, S)
    den = np.einsum("nf,nf->n", pq, z)
    return S, z, num / (den + eps)[:, None]


def _feature_vjp_harmonic(u, gamma, omega, phi, N, pos0, dphi):
    """Pull a cotangent dPhi_N [B,H,T,F_N] of featurize_harmonic back to du and
    the parameter gradients.  Per dimension, with the angle block A_m (A_0 = 1,
    A_{2n-1} = cos n th, A_{2n} = sin n th of the rotated angle th) and the
    label block r A_m:
        dA_m  = dPhi[A_m] + r dPhi[r A_m],      dr = sum_m A_m dPhi[r A_m],
        dth   = sum_n n (-sin(n th) dA_{2n-1} + cos(n th) dA_{2n}),
    then through the soft root, the rotation and the squash exactly as the
    six-channel map (which is N = 1)."""
    parts = _feature_parts(u, gamma, omega, phi, pos0)
    B, H, T, F = dphi.shape
    kA = 2 * N + 1
    d = F // (2 * kA)
    dp = np.asarray(dphi, dtype=np.float64).reshape(B, H, T, d, 2, kA)
    th = rotate(squash(parts["u"]), parts["t"], np.asarray(phi, dtype=np.float64).reshape(
        1, H, 1, d))
    r = parts["r"]
    ang = [np.ones_like(th)]
    for n in range(1, N + 1):
        ang += [np.cos(n * th), np.sin(n * th)]
    A = np.stack(ang, axis=-1)
    dA = dp[..., 0, :] + r[..., None] * dp[..., 1, :]
    dr = (A * dp[..., 1, :]).sum(axis=-1)
    dth_rot = np.zeros_like(th)
    for n in range(1, N + 1):
        dth_rot += n * (-np.sin(n * th) * dA[..., 2 * n - 1] + np.cos(n * th) * dA[..., 2 * n])
    dpre = dr * (1.0 - r * r)
    dtheta = dth_rot + dpre * parts["g"] * parts["gpx"]
    du = dtheta * np.pi / (1.0 + np.abs(parts["u"])) ** 2
    dgamma = (dpre * parts["gx"]).sum(axis=(0, 2, 3))
    domega = (dpre * parts["g"] * parts["gpx"]).sum(axis=(0, 2))
    dphi_rate = (dth_rot * parts["t"]).sum(axis=(0, 2))
    return du, dgamma, domega, dphi_rate


def attn_harmonic_backward(q, k, v, gamma, omega, phi, dO, N, pos0=0, eps=0.0, S0=None, z0=None):
    """Gradients of sum(o * dO) for ``attn_harmonic``: the equations of
    ``attn_backward`` with Phi_N in place of Phi (s_tj = Phi_N(q_t).Phi_N(k_j)),
    then through the harmonic map.  Returns the dict of ``attn_backward``."""
    pq = featurize_harmonic(q, gamma, omega, phi, N, pos0)
    pk = featurize_harmonic(k, gamma, omega, phi, N, pos0)
    v = _heads(v)
    dO = _heads(dO)
    B, H, T, F = pq.shape
    mask = np.tril(np.ones((T, T)))
    dpq = np.zeros_like(pq)
    dpk = np.zeros_like(pk)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            s = (pq[b, h] @ pk[b, h].T) * mask
            num = s @ v[b, h]
            den = s.sum(axis=1)
            if S0 is not None:
                num = num + pq[b, h] @ _heads(S0)[b, h]
                den = den + pq[b, h] @ _heads(z0)[b, h]
            dh = den + eps
            o = num / dh[:, None]
            dN = dO[b, h] / dh[:, None]
            dD = -(dO[b, h] * o).sum(axis=1) / dh
            ds = (dN @ v[b, h].T + dD[:, None]) * mask
            dv[b, h] = s.T @ dN
            dpq[b, h] = ds @ pk[b, h]
            if S0 is not None:
                dpq[b, h] += dN @ _heads(S0)[b, h].T + np.outer(dD, _heads(z0)[b, h])
            dpk[b, h] = ds.T @ pq[b, h]
    dq, dg_q, dom_q, dph_q = _feature_vjp_harmonic(q, gamma, omega, phi, N, pos0, dpq)
    dk, dg_k, dom_k, dph_k = _feature_vjp_harmonic(k, gamma, omega, phi, N, pos0, dpk)
    return dict(dq=dq, dk=dk, dv=dv, dgamma=dg_q + dg_k, domega=dom_q + dom_k,
                dphi=dph_q + dph_k)


def state_bytes_harmonic(layers, heads, d, dv, N, bytes_per_float=4):
    """Recurrent state with harmonics 1..N: per head S (F_N x dv) and z (F_N),
    F_N = 2(2N + 1) d (N = 1: the six-channel 6 d^2 + 6 d of Notes §2.7)."""
    F = harmonic_channels(N) * d
    return layers * heads * (F * dv + F) * bytes_per_float


# ---------------------------------------------------------------------------
# Multi-layer attention stack (Notes §2.7: the whole-model recurrence updates
# the layers' states in order, each layer with its own weights, at the same
# positions; §3.1: 12 layers x 12 heads x d = 64).  The attention path only:
# per layer x -> q, k, v = x Wq, x Wk, x Wv, the p = 1 attention of every
# head, x <- x + a Wo (no normalisation layers or MLP).
# ---------------------------------------------------------------------------


def stack_parallel(X, Wqkv, Wo, gamma, omega, phi, heads, pos0=0, eps=0.0):
    """The attention stack over a whole sequence in the parallel form:
    X [B, T, heads*d]; Wqkv [L, heads*d, 3*heads*d] (columns: q | k | v);
    Wo [L, heads*d, heads*d]; gamma [L, heads]; omega, phi [L, heads, d].
    Every layer's attention is attn_quadratic over the whole prefix.
    Returns the last layer's output X [B, T, heads*d]."""
    X = np.asarray(X, dtype=np.float64)
    B, T, Dm = X.shape
    L = np.asarray(Wqkv).shape[0]
    d = Dm // heads
    for l in range(L):
        qkv = X @ np.asarray(Wqkv[l], dtype=np.float64)
        sp = lambda m: m.reshape(B, T, heads, d).transpose(0, 2, 1, 3)  # noqa: E731
        q, k, v = sp(qkv[..., :Dm]), sp(qkv[..., Dm:2 * Dm]), sp(qkv[..., 2 * Dm:])
        o, _ = attn_quadratic(q, k, v, gamma[l], omega[l], phi[l], pos0=pos0, eps=eps)
        A = o.transpose(0, 2, 1, 3).reshape(B, T, Dm)
        X = X + A @ np.asarray(Wo[l], dtype=np.float64)
    return X


def stack_decode_step(x, Wqkv, Wo, S, z, gamma, omega, phi, heads, pos, eps=0.0):
    """One token through the attention stack with the constant-state
    recurrence: x [B, heads*d]; S [L, B*heads, 6d, d], z [L, B*heads, 6d]
    (slot b * heads + h); pos [B] integer positions.  Returns (x, S, z)."""
    x = np.asarray(x, dtype=np.float64)
    B, Dm = x.shape
    L = np.asarray(Wqkv).shape[0]
    d = Dm // heads
    S = np.array(S, dtype=np.float64)
    z = np.array(z, dtype=np.float64)
    slot_pos = np.repeat(np.asarray(pos, dtype=np.int64), heads)
    for l in range(L):
        qkv = x @ np.asarray(Wqkv[l], dtype=np.float64)
        q = qkv[:, :Dm].reshape(B * heads, d)
        k = qkv[:, Dm:2 * Dm].reshape(B * heads, d)
        v = qkv[:, 2 * Dm:].reshape(B * heads, d)
        g = np.tile(np.asarray(gamma[l], dtype=np.float64), B)
        om = np.tile(np.asarray(omega[l], dtype=np.float64), (B, 1))
        ph = np.tile(np.asarray(phi[l], dtype=np.float64), (B, 1))
        S[l], z[l], o = decode_step(S[l], z[l], q, k, v, g, om, ph, slot_pos, eps=eps)
        x = x + o.reshape(B, Dm) @ np.asarray(Wo[l], dtype=np.float64)
    return x, S, z


# ---------------------------------------------------------------------------
# Rate parameterisation (Notes §2.2, eq. (4)) and the eps scale (Notes §2.7)
# ---------------------------------------------------------------------------


def rate_from_raw(lambda_raw, scale=0.01):
    """The rotation rate lambda = 0.01 tanh(lambda_raw) of eq. (4)."""
    return scale * np.tanh(np.asarray(lambda_raw, dtype=np.float64))


def rate_from_raw_grad(lambda_raw, dphi, scale=0.01):
    """d loss / d lambda_raw from d loss / d lambda (chain rule of tanh)."""
    t = np.tanh(np.asarray(lambda_raw, dtype=np.float64))
    return np.asarray(dphi, dtype=np.float64) * scale * (1.0 - t * t)


def eps_raw(eps, d, convention=0):
    """Notes §2.7: a parallel form that divides by c and then adds eps equals
    the raw-score form with eps_raw = c eps; the authors' parallel code uses
    c = 4d + 1e-6 (convention 0), their recurrence notebook 4d * 1e-6 (1)."""
    c = 4.0 * d + 1e-6 if convention == 0 else 4.0 * d * 1e-6
    return c * eps


# ---------------------------------------------------------------------------
# Memory accounting: Notes §4.5 [paper §4.4]
# ---------------------------------------------------------------------------


def state_bytes(layers, heads, d, dv, bytes_per_float=4):
    """Recurrent state of one sequence: per head S (6d x dv) and z (6d)."""
    return layers * heads * (6 * d * dv + 6 * d) * bytes_per_float


def kv_cache_bytes(n, layers, model_dim, bytes_per_float=4):
    """Softmax KV cache for context n: keys and values of every layer."""
    return 2 * n * layers * model_dim * bytes_per_float


def kv_crossover(layers, heads, d, dv, model_dim, bytes_per_float=4):
    """Smallest integer context n whose KV cache is at least the state size."""
    st = state_bytes(layers, heads, d, dv, bytes_per_float)
    per_token = kv_cache_bytes(1, layers, model_dim, bytes_per_float)
    return int(np.ceil(st / per_token))
