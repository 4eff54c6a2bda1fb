"""sanatan_chunk_bwd against the float64 oracle's hand-derived backward
(itself pinned by finite differences and torch autograd).  Gradient bar:
relative L2 error <= 1e-2 per tensor for bf16 operands, <= 1e-4 for f32."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import dev, f64, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu


def _run(x, dO, pos0=0, eps=0.0, S0=None, z0=None):
    g = to_dev(x)
    dOd = dO.to(dev())
    S0d = None if S0 is None else S0.to(dev())
    z0d = None if z0 is None else z0.to(dev())
    o, D, _, _ = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                     pos0=pos0, eps=eps, S0=S0d, z0=z0d)
    gr = S.sanatan_chunk_bwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], o, D, dOd,
                             pos0=pos0, eps=eps, S0=S0d, z0=z0d, want_dphi=True)
    S.device_status()
    return gr


def _compare(gr, ref, tol, names=("dq", "dk", "dv", "dgamma", "domega", "dphi")):
    errs = {n: rel_fro(f64(gr[n]), ref[n]) for n in names}
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, (bad, errs)
    return errs


@pytest.mark.parametrize("T", [1, 33, 70])
def test_f32_small_with_state_eps_offset(T):
    x = W.make(W.TINY, B=2, H=3, T=T)
    x["phi"] = W.rates(3, 64, "geometric")
    rng = np.random.default_rng(T)
    S0, z0 = O.final_state(rng.standard_normal((2, 3, 25, 64)), rng.standard_normal((2, 3, 25, 64)),
                           f64(x["gamma"]), f64(x["omega"]), f64(x["phi"]), pos0=200)
    S0 = torch.tensor(S0, dtype=torch.float32)
    z0 = torch.tensor(z0, dtype=torch.float32)
    dO = torch.randn(2, 3, T, 64, generator=torch.Generator().manual_seed(T))
    gr = _run(x, dO, pos0=225, eps=0.3, S0=S0, z0=z0)
    ref = O.attn_backward(**ref_args(x), dO=f64(dO), pos0=225, eps=0.3, S0=f64(S0), z0=f64(z0))
    _compare(gr, ref, 1e-4)


def test_bf16_multi_chunk():
    x = W.make(W.TRAIN, B=2, H=2, T=300, with_grad_out=True)
    gr = _run(x, x["dO"])
    ref = O.attn_backward(**ref_args(x), dO=f64(x["dO"]))
    _compare(gr, ref, 1e-2)


@pytest.mark.parametrize("T", [1, 127, 600, 1500])
def test_bf16_with_state_eps_offset_segments(T):
    """bf16 operands with an initial state, eps and a position offset; B*H = 3
    splits T >= 256 into several segments (the per-segment sums of both time
    directions are exercised)."""
    x = W.make(W.TRAIN, B=1, H=3, T=T, with_grad_out=True)
    x["phi"] = W.rates(3, 64, "geometric")
    rng = np.random.default_rng(T + 1)
    S0, z0 = O.final_state(rng.standard_normal((1, 3, 40, 64)), rng.standard_normal((1, 3, 40, 64)),
                           f64(x["gamma"]), f64(x["omega"]), f64(x["phi"]), pos0=60)
    S0 = torch.tensor(S0, dtype=torch.float32)
    z0 = torch.tensor(z0, dtype=torch.float32)
    gr = _run(x, x["dO"], pos0=100, eps=0.3, S0=S0, z0=z0)
    ref = O.attn_backward(**ref_args(x), dO=f64(x["dO"]), pos0=100, eps=0.3, S0=f64(S0),
                          z0=f64(z0))
    _compare(gr, ref, 1e-2)


def test_bf16_grad_dtype_f32_upstream():
    x = W.make(W.TRAIN, B=1, H=2, T=129, with_grad_out=True)
    gr = _run(x, x["dO"].float())
    ref = O.attn_backward(**ref_args(x), dO=f64(x["dO"]))
    _compare(gr, ref, 1e-2)


def test_autograd_function_matches_oracle():
    x = W.make(W.TRAIN, B=1, H=2, T=96, with_grad_out=True)
    g = to_dev(x)
    leaves = {n: g[n].clone().requires_grad_(True) for n in ("q", "k", "v", "gamma", "omega", "phi")}
    o = S.SanatanAttention.apply(leaves["q"], leaves["k"], leaves["v"], leaves["gamma"],
                                 leaves["omega"], leaves["phi"])
    (o * g["dO"].float()).sum().backward()
    ref = O.attn_backward(**ref_args(x), dO=f64(x["dO"]))
    for n in ("q", "k", "v", "gamma", "omega", "phi"):
        assert rel_fro(f64(leaves[n].grad), ref["d" + n]) <= 1e-2, n


def test_training_workload_full_size_all_sequences():
    """B=8, H=12, T=4096 (bf16 q, k, v, dO; three segments per sequence):
    dq, dk, dv of all 96 sequences and the parameter gradients dgamma,
    domega, dphi (sums over the batch and over q and k) against the oracle's
    backward run one (batch, head) at a time (the gradient of one sequence
    depends on nothing else; the parameter gradients are the sums of the
    per-sequence ones)."""
    x = W.make(W.TRAIN, device="cpu", with_grad_out=True)
    gr = _run(x, x["dO"])
    ra = ref_args(x)
    dO = f64(x["dO"])
    B, H = x["B"], x["H"]
    ref = {n: np.zeros(ra[n[1:]].shape) for n in ("dq", "dk", "dv")}
    pref = {n: np.zeros(ra[n[1:]].shape) for n in ("dgamma", "domega", "dphi")}
    for b in range(B):
        for h in range(H):
            sl = {n: ra[n][b:b + 1, h:h + 1] for n in ("q", "k", "v")}
            r = O.attn_backward(**sl, gamma=ra["gamma"][h:h + 1], omega=ra["omega"][h:h + 1],
                                phi=ra["phi"][h:h + 1], dO=dO[b:b + 1, h:h + 1])
            for n in ("dq", "dk", "dv"):
                ref[n][b, h] = r[n][0, 0]
            for n in ("dgamma", "domega", "dphi"):
                pref[n][h] += r[n][0]
    for n in ("dq", "dk", "dv"):
        g = f64(gr[n])
        assert rel_fro(g, ref[n]) <= 1e-2, n
        worst = max(rel_fro(g[b, h], ref[n][b, h]) for b in range(B) for h in range(H))
        assert worst <= 1e-2, (n, worst)
    for n in ("dgamma", "domega", "dphi"):
        assert rel_fro(f64(gr[n]), pref[n]) <= 1e-2, n


def test_backward_reuses_forward_state_sums():
    """With the forward's workspace passed in, the backward skips its own
    forward-time state pass and gives the same gradients bit for bit (the sums
    come from the same kernel on the same inputs)."""
    x = W.make(W.TRAIN, device="cuda", B=1, H=12, T=2048, with_grad_out=True)
    g = [x[n] for n in ("q", "k", "v", "gamma", "omega", "phi")]
    B, H, T = 1, 12, 2048
    assert S.chunk_fwd_plan(B, H, T)[0] > 1
    ws = torch.empty(max(S.chunk_fwd_workspace_size(B, H, T), 16), dtype=torch.uint8,
                     device="cuda")
    o, D, _, _ = S.sanatan_chunk_fwd(*g, workspace=ws)
    a = S.sanatan_chunk_bwd(*g, o, D, x["dO"], want_dphi=True)
    b = S.sanatan_chunk_bwd(*g, o, D, x["dO"], want_dphi=True, fwd_workspace=ws)
    # a workspace too small for the backward's split is ignored
    c = S.sanatan_chunk_bwd(*g, o, D, x["dO"], want_dphi=True, fwd_workspace=ws[:16])
    torch.cuda.synchronize()
    S.device_status()
    for key in ("dq", "dk", "dv"):
        assert torch.equal(a[key], b[key]) and torch.equal(a[key], c[key]), key
    for key in ("dgamma", "domega", "dphi"):
        # float atomics: the order of the per-CTA sums may differ (dphi sums
        # terms dtheta * t that cancel, so compare whole tensors)
        assert (a[key] - b[key]).norm() <= 1e-4 * a[key].norm(), key
