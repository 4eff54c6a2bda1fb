"""The harmonic feature map (Appendix B of the notes) on the GPU against the
float64 oracle: features (f32 <= 1e-5 abs), the chunked p=1 forward (f32:
<= 1e-5 on o, state relative <= 1e-5; at the full layer-forward size <= 1e-4
on o), the decode step (<= 1e-5), chunked vs decode (<= 1e-4), N = 1 against
the six-channel entry points, and the backward (f32 gradients <= 1e-4
relative; bf16 at the layer shape <= 1e-2, the gradient bar)."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import dev, f64, max_abs, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N", [1, 2, 3])
def test_features(N):
    x = W.make(W.TINY, B=1, H=2, T=50)
    x["phi"] = W.rates(2, 64, "geometric")
    g = to_dev(x)
    f = S.sanatan_featurize_harmonic(g["q"], g["gamma"], g["omega"], g["phi"], N, pos0=300)
    torch.cuda.synchronize()
    ra = ref_args(x)
    ref = O.featurize_harmonic(ra["q"], ra["gamma"], ra["omega"], ra["phi"], N, pos0=300)
    assert max_abs(f64(f), ref) <= 1e-5


@pytest.mark.parametrize("N,T", [(2, 1), (2, 7), (2, 8), (2, 9), (2, 100), (3, 1), (3, 13),
                                 (3, 100)])
def test_chunked_forward_harmonics(N, T):
    x = W.make(W.TINY, B=2, H=2, T=T)
    x["phi"] = W.rates(2, 64, "geometric")
    g = to_dev(x)
    o, D, Sx, zx = S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"],
                                                g["phi"], N, pos0=40, eps=0.2, want_state=True)
    torch.cuda.synchronize()
    ra = ref_args(x)
    o_ref, D_ref = O.attn_harmonic(**ra, N=N, pos0=40, eps=0.2)
    S_ref, z_ref = O.final_state_harmonic(ra["k"], ra["v"], ra["gamma"], ra["omega"], ra["phi"], N,
                                          pos0=40)
    assert max_abs(f64(o), o_ref) <= 1e-5
    assert rel_fro(f64(D), D_ref) <= 1e-5
    assert rel_fro(f64(Sx), S_ref) <= 1e-5 and rel_fro(f64(zx), z_ref) <= 1e-5


def test_chunked_forward_bf16_inputs_and_initial_state():
    x = W.make(W.LAYER, B=1, H=3, T=77)
    g = to_dev(x)
    ra = ref_args(x)
    rng = np.random.default_rng(4)
    S0, z0 = O.final_state_harmonic(rng.standard_normal((1, 3, 30, 64)),
                                    rng.standard_normal((1, 3, 30, 64)), ra["gamma"], ra["omega"],
                                    ra["phi"], 2, pos0=500)
    S0t, z0t = torch.tensor(S0, dtype=torch.float32), torch.tensor(z0, dtype=torch.float32)
    o, _, _, _ = S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"],
                                              g["phi"], 2, pos0=530, S0=S0t.to(dev()),
                                              z0=z0t.to(dev()))
    torch.cuda.synchronize()
    o_ref, _ = O.attn_harmonic(**ra, N=2, pos0=530, S0=f64(S0t), z0=f64(z0t))
    assert max_abs(f64(o), o_ref) <= 1e-5


@pytest.mark.parametrize("N", [2, 3])
def test_chunked_forward_full_size_sampled_sequences(N):
    """B=4, H=12, T=2048 bf16 (the layer-forward workload, all 48 sequences in
    one launch): the outputs and final state of three sampled sequences, each
    against the oracle's quadratic form (1e-4 on o, 1e-5 relative on D, S, z)."""
    x = W.make(W.LAYER, device="cpu")
    g = to_dev(x)
    o, D, Sx, zx = S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"],
                                                g["phi"], N, want_state=True)
    torch.cuda.synchronize()
    ra = ref_args(x)
    og, Dg, Sg, zg = f64(o), f64(D), f64(Sx), f64(zx)
    for b, h in ((0, 0), (1, 5), (3, 11)):
        one = {n: ra[n][b:b + 1, h:h + 1] for n in ("q", "k", "v")}
        one.update({n: ra[n][h:h + 1] for n in ("gamma", "omega", "phi")})
        o_ref, D_ref = O.attn_harmonic(**one, N=N)
        S_ref, z_ref = O.final_state_harmonic(one["k"], one["v"], one["gamma"], one["omega"],
                                              one["phi"], N)
        assert max_abs(og[b, h], o_ref[0, 0]) <= 1e-4, (b, h)
        assert rel_fro(Dg[b, h], D_ref[0, 0]) <= 1e-5, (b, h)
        assert rel_fro(Sg[b, h], S_ref[0, 0]) <= 1e-5, (b, h)
        assert rel_fro(zg[b, h], z_ref[0, 0]) <= 1e-5, (b, h)


@pytest.mark.parametrize("N", [1, 2, 3])
def test_decode_steps_match_oracle_and_chunked(N):
    """T single-token steps from the zero state reproduce the oracle (1e-5) and
    the chunked forward (1e-4)."""
    x = W.make(W.TINY, B=1, H=3, T=40)
    x["phi"] = W.rates(3, 64, "geometric")
    g = to_dev(x)
    F = S.harmonic_features(N)
    Sd = torch.zeros(3, F, 64, device=dev())
    zd = torch.zeros(3, F, device=dev())
    outs = []
    for t in range(40):
        pos = torch.full((3,), 900 + t, dtype=torch.int64, device=dev())
        outs.append(S.sanatan_decode_step_harmonic(Sd, zd, g["q"][0, :, t].contiguous(),
                                                   g["k"][0, :, t].contiguous(),
                                                   g["v"][0, :, t].contiguous(), g["gamma"],
                                                   g["omega"], g["phi"], pos, N, eps=0.1))
    od = torch.stack(outs, 1).unsqueeze(0)
    torch.cuda.synchronize()
    o_ref, _ = O.attn_harmonic(**ref_args(x), N=N, pos0=900, eps=0.1)
    assert max_abs(f64(od), o_ref) <= 1e-5
    oc, _, Sc, zc = S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"],
                                                 g["phi"], N, pos0=900, eps=0.1, want_state=True)
    torch.cuda.synchronize()
    assert max_abs(f64(od), f64(oc)) <= 1e-4
    assert rel_fro(f64(Sd), f64(Sc)[0]) <= 1e-5


def test_one_harmonic_is_the_six_channel_path():
    x = W.make(W.TINY, B=1, H=2, T=64)
    g = to_dev(x)
    a, _, _, _ = S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"],
                                              g["phi"], 1)
    b, _, _, _ = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"])
    fa = S.sanatan_featurize_harmonic(g["q"], g["gamma"], g["omega"], g["phi"], 1)
    fb = S.sanatan_featurize(g["q"], g["gamma"], g["omega"], g["phi"])
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert (fa - fb).abs().max().item() <= 1e-6


def test_argument_errors():
    x = W.make(W.TINY, B=1, H=1, T=4)
    g = to_dev(x)
    with pytest.raises(S.SanatanError) as e:
        S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 4)
    assert e.value.status == 2
    with pytest.raises(S.SanatanError) as e:
        S.sanatan_featurize_harmonic(g["q"], g["gamma"], g["omega"], g["phi"], 4)
    assert e.value.status == 2


def _rel(a, b):
    return rel_fro(f64(a), b)


def _harmonic_grads(g, N, pos0, eps, S0=None, z0=None, dO=None, want_dphi=True):
    o, D, _, _ = S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"],
                                              g["phi"], N, pos0=pos0, eps=eps, S0=S0, z0=z0)
    return S.sanatan_chunk_bwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                        N, o, D, dO, pos0=pos0, eps=eps, S0=S0, z0=z0,
                                        want_dphi=want_dphi)


@pytest.mark.parametrize("N,T,hist", [(2, 1, False), (2, 17, True), (2, 100, False),
                                      (3, 16, False), (3, 77, True)])
def test_backward_matches_oracle(N, T, hist):
    """f32 inputs: every gradient (dq, dk, dv, dgamma, domega, dphi) within 1e-4
    relative (Frobenius) of the float64 oracle, with a history (S0, z0), eps and
    a position offset."""
    x = W.make(W.TINY, B=2, H=2, T=T)
    x["phi"] = W.rates(2, 64, "geometric")
    g = to_dev(x)
    ra = ref_args(x)
    rng = np.random.default_rng(5 + T)
    dO = rng.standard_normal((2, 2, T, 64)).astype(np.float32)
    S0 = z0 = S0t = z0t = None
    if hist:
        S0, z0 = O.final_state_harmonic(rng.standard_normal((2, 2, 12, 64)),
                                        rng.standard_normal((2, 2, 12, 64)), ra["gamma"],
                                        ra["omega"], ra["phi"], N, pos0=20)
        S0t = torch.tensor(S0, dtype=torch.float32, device=dev())
        z0t = torch.tensor(z0, dtype=torch.float32, device=dev())
        S0, z0 = f64(S0t), f64(z0t)
    gr = _harmonic_grads(g, N, 32, 0.3, S0t, z0t, torch.tensor(dO, device=dev()))
    torch.cuda.synchronize()
    ref = O.attn_harmonic_backward(**ra, dO=dO.astype(np.float64), N=N, pos0=32, eps=0.3, S0=S0,
                                   z0=z0)
    for key in ("dq", "dk", "dv", "dgamma", "domega"):
        err = _rel(gr[key], ref[key])
        assert err <= 1e-4, (key, err)
    # dphi: the q and k shares (position x angle gradient) cancel up to the
    # relative positions (exactly, at T = 1), so its error is measured against
    # the larger of its own norm and the shares' size, position x |dq|, scaled
    # to the 1e-6 relative accuracy of a float32 angle gradient (1e-2 x 1e-4)
    scale = max(np.linalg.norm(ref["dphi"]), 1e-2 * (32 + T) * np.linalg.norm(ref["dq"]))
    err = np.linalg.norm(f64(gr["dphi"]) - ref["dphi"]) / scale
    assert err <= 1e-4, ("dphi", err)


@pytest.mark.parametrize("N", [2, 3])
def test_backward_full_size_sampled_heads(N):
    """B=4, H=12, T=2048 bf16 (the layer-forward workload, one launch over all 48
    sequences): for heads 0 and 11, dq, dk, dv of every sequence and the head's
    dgamma, domega, dphi (sums over the batch) within 1e-2 relative of the
    oracle (gradients are bf16 like the inputs)."""
    x = W.make(W.LAYER, device="cpu")
    g = to_dev(x)
    dOt = torch.randn(x["q"].shape[:3] + (64,), generator=torch.Generator().manual_seed(77))
    gr = _harmonic_grads(g, N, 0, 0.0, dO=dOt.to(torch.bfloat16).to(dev()))
    torch.cuda.synchronize()
    ra = ref_args(x)
    dO = f64(dOt.to(torch.bfloat16))
    for h in (0, 11):
        one = {n: ra[n][:, h:h + 1] for n in ("q", "k", "v")}
        one.update({n: ra[n][h:h + 1] for n in ("gamma", "omega", "phi")})
        ref = O.attn_harmonic_backward(**one, dO=dO[:, h:h + 1], N=N)
        for key in ("dq", "dk", "dv"):
            err = rel_fro(f64(gr[key])[:, h:h + 1], ref[key])
            assert err <= 1e-2, (h, key, err)
        for key in ("dgamma", "domega", "dphi"):
            err = rel_fro(f64(gr[key])[h:h + 1], ref[key])
            assert err <= 1e-2, (h, key, err)


def test_backward_one_harmonic_is_the_six_channel_path():
    x = W.make(W.TINY, B=1, H=2, T=40)
    g = to_dev(x)
    dO = torch.randn(1, 2, 40, 64, generator=torch.Generator().manual_seed(3)).to(dev())
    o, D, _, _ = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"])
    a = S.sanatan_chunk_bwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 1,
                                     o, D, dO, want_dphi=True)
    b = S.sanatan_chunk_bwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], o, D, dO,
                            want_dphi=True)
    torch.cuda.synchronize()
    for key in ("dq", "dk", "dv"):
        assert torch.equal(a[key], b[key]), key
    for key in ("dgamma", "domega", "dphi"):
        assert (a[key] - b[key]).abs().max().item() <= 1e-5 * (1 + b[key].abs().max().item()), key


def test_backward_empty_and_errors():
    x = W.make(W.TINY, B=1, H=2, T=0)
    g = to_dev(x)
    o = torch.empty(1, 2, 0, 64, device=dev())
    D = torch.empty(1, 2, 0, device=dev())
    gr = S.sanatan_chunk_bwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 2,
                                      o, D, o, want_dphi=True)
    torch.cuda.synchronize()
    for key in ("dgamma", "domega", "dphi"):
        assert torch.count_nonzero(gr[key]).item() == 0, key
    x = W.make(W.TINY, B=1, H=1, T=4)
    g = to_dev(x)
    o = torch.zeros(1, 1, 4, 64, device=dev())
    D = torch.ones(1, 1, 4, device=dev())
    with pytest.raises(S.SanatanError) as e:
        S.sanatan_chunk_bwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 4,
                                     o, D, o)
    assert e.value.status == 2
    with pytest.raises(S.SanatanError) as e:
        S.sanatan_chunk_bwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 2,
                                     o, D, o, workspace=torch.empty(16, dtype=torch.uint8,
                                                                    device=dev()))
    assert e.value.status == 1
