"""sanatan_decode_step against the oracle and against the chunked forward."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import dev, f64, max_abs, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu


def test_decode_over_tiny_sequence_matches_chunked_and_oracle():
    """T single-token steps from the zero state reproduce the chunked forward
    (<= 1e-4) and the oracle (<= 1e-5)."""
    x = W.make(W.TINY)
    g = to_dev(x)
    T = x["T"]
    Sd = torch.zeros(1, 384, 64, device=dev())
    zd = torch.zeros(1, 384, device=dev())
    outs = []
    for t in range(T):
        pos = torch.full((1,), t, dtype=torch.int64, device=dev())
        outs.append(S.sanatan_decode_step(Sd, zd, g["q"][0, :, t].contiguous(),
                                          g["k"][0, :, t].contiguous(), g["v"][0, :, t].contiguous(),
                                          g["gamma"], g["omega"], g["phi"], pos))
    od = torch.stack(outs, 1).unsqueeze(1)  # [1, 1, T, dv]
    oc, _, Sc, zc = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                        want_state=True)
    torch.cuda.synchronize()
    assert max_abs(f64(od), f64(oc)) <= 1e-4
    o_ref, _ = O.attn_quadratic(**ref_args(x))
    assert max_abs(f64(od), o_ref) <= 1e-5
    assert rel_fro(f64(Sd), f64(Sc)[0]) <= 1e-5 and rel_fro(f64(zd), f64(zc)[0]) <= 1e-5


# (7, 3), (19, 12): 8-CTA clusters; (20, 12), (144, 144), (300, 144): one
# 1024-thread CTA per slot; (400, 144): 4-CTA clusters; (700, 144): 256 threads
@pytest.mark.parametrize("N,G", [(144, 144), (300, 144), (7, 3), (19, 12), (20, 12), (400, 144),
                                 (700, 144)])
def test_decode_many_slots_from_random_state(N, G):
    rng = np.random.default_rng(N)
    gen = W.generator(4000 + N)
    gamma, omega, phi = W.params(G, 64, "geometric", gen)
    Ssl, zsl = [], []
    for n in range(N):
        kp = rng.standard_normal((1, 1, 20, 64))
        vp = rng.standard_normal((1, 1, 20, 64))
        g = n % G
        s_, z_ = O.final_state(kp, vp, f64(gamma)[g:g + 1], f64(omega)[g:g + 1], f64(phi)[g:g + 1])
        Ssl.append(s_[0, 0])
        zsl.append(z_[0, 0])
    S0 = torch.tensor(np.stack(Ssl), dtype=torch.float32)
    z0 = torch.tensor(np.stack(zsl), dtype=torch.float32)
    q, k, v = (t[0] for t in W.decode_tokens(N, 64, 64, 1, gen))
    pos = torch.tensor(rng.integers(20, 40000, N), dtype=torch.int64)
    Sd, zd = S0.to(dev()), z0.to(dev())
    o = S.sanatan_decode_step(Sd, zd, q.to(dev()), k.to(dev()), v.to(dev()), gamma.to(dev()),
                              omega.to(dev()), phi.to(dev()), pos.to(dev()), eps=0.25)
    torch.cuda.synchronize()
    idx = np.arange(N) % G
    S_ref, z_ref, o_ref = O.decode_step(f64(S0), f64(z0), f64(q), f64(k), f64(v),
                                        f64(gamma)[idx], f64(omega)[idx], f64(phi)[idx],
                                        pos.numpy(), eps=0.25)
    assert max_abs(f64(o), o_ref) <= 1e-5
    assert max_abs(f64(Sd), S_ref) <= 1e-5 * max(1.0, np.abs(S_ref).max())
    assert max_abs(f64(zd), z_ref) <= 1e-5 * max(1.0, np.abs(z_ref).max())


def test_decode_zero_slots_is_noop():
    e = torch.empty(0, 64, device=dev())
    o = S.sanatan_decode_step(torch.empty(0, 384, 64, device=dev()), torch.empty(0, 384, device=dev()),
                              e, e, e, torch.ones(1, device=dev()), torch.zeros(1, 64, device=dev()),
                              torch.zeros(1, 64, device=dev()), torch.empty(0, dtype=torch.int64,
                                                                            device=dev()))
    assert o.shape == (0, 64)


def _stack_tokens(q):
    """[steps, N, d] -> [1, N, steps, d] (one sequence per slot)."""
    return q.permute(1, 0, 2).unsqueeze(0).contiguous()


def test_decode_workload_B1_prefill_then_1024_steps():
    """The batched-decode workload at B = 1, at its own shape: 12 layers x 12
    heads = 144 state slots, the state built by a bf16 chunked prefill of 4096
    N(0,1) tokens (positions 0..4095), then 1024 single-token f32 steps with
    fresh N(0,1) q, k, v at positions 4096..5119.

    (1) The prefill's S and z of every slot against the oracle's final state
        (relative Frobenius <= 5e-3, the bf16-operand bar).
    (2) o after every one of the 1024 steps against the oracle's own decode
        steps, started from the oracle's state: max abs <= 5e-3, the bf16 bar,
        since the prefill state's bf16 error is inherited; every step after it
        is f32.
    (3) The same 1024 tokens through the f32 chunked forward from the GPU
        prefill state at pos0 = 4096: its outputs and final state against the
        stepped ones (<= 1e-4, the chunked-vs-decode bar)."""
    w = W.DECODE
    G = 144
    steps = w.extra["steps"]
    x = W.make(w, device="cpu", B=1)
    g = to_dev(x)
    _, _, Sx, zx = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                       want_D=False, want_state=True)
    S.device_status()
    ra = ref_args(x)
    S_ref, z_ref = O.final_state(ra["k"], ra["v"], ra["gamma"], ra["omega"], ra["phi"])
    assert rel_fro(f64(Sx), S_ref) <= 5e-3
    assert rel_fro(f64(zx), z_ref) <= 5e-3

    gen = W.generator(w.seed + 100)
    q, k, v = W.decode_tokens(G, 64, 64, steps, gen)            # [steps, 144, 64] f32
    qd, kd, vd = q.to(dev()), k.to(dev()), v.to(dev())
    S0 = Sx.reshape(G, 384, 64).clone()
    z0 = zx.reshape(G, 384).clone()
    Sd, zd = S0.clone(), z0.clone()
    od = torch.empty(steps, G, 64, device=dev())
    for i in range(steps):
        pos = torch.full((G,), 4096 + i, dtype=torch.int64, device=dev())
        S.sanatan_decode_step(Sd, zd, qd[i], kd[i], vd[i], g["gamma"], g["omega"], g["phi"], pos,
                              out=od[i])
    torch.cuda.synchronize()

    Sr, zr = S_ref[0], z_ref[0]
    gam, om, ph = ra["gamma"], ra["omega"], ra["phi"]
    q64, k64, v64 = f64(q), f64(k), f64(v)
    od64 = f64(od)
    worst = 0.0
    for i in range(steps):
        Sr, zr, o_ref = O.decode_step(Sr, zr, q64[i], k64[i], v64[i], gam, om, ph,
                                      np.full(G, 4096 + i))
        worst = max(worst, max_abs(od64[i], o_ref))
    assert worst <= 5e-3, worst
    assert rel_fro(f64(Sd), Sr) <= 5e-3 and rel_fro(f64(zd), zr) <= 5e-3

    oc, _, Sc, zc = S.sanatan_chunk_fwd(_stack_tokens(qd), _stack_tokens(kd), _stack_tokens(vd),
                                        g["gamma"], g["omega"], g["phi"], pos0=4096,
                                        S0=S0.unsqueeze(0), z0=z0.unsqueeze(0), want_state=True)
    torch.cuda.synchronize()
    assert max_abs(f64(oc)[0], np.transpose(od64, (1, 0, 2))) <= 1e-4
    assert rel_fro(f64(Sc)[0], f64(Sd)) <= 1e-5 and rel_fro(f64(zc)[0], f64(zd)) <= 1e-5


def test_decode_workload_B64_sampled_slots():
    """The batched-decode workload at B = 64 (9216 slots, a 1.85 GB state
    built by the bf16 prefill of 64 x 144 sequences of 4096 tokens), then 8
    f32 steps at positions 4096..4103 for every slot.  Sampled slots are
    checked against the oracle (prefill state, every step's o), and every
    slot's stepped outputs against the f32 chunked forward over the same
    tokens from the same state (<= 1e-4)."""
    w = W.DECODE
    G, B, steps = 144, 64, 8
    N = B * G
    x = W.make(w, device=dev(), B=B)
    _, _, Sx, zx = S.sanatan_chunk_fwd(x["q"], x["k"], x["v"], x["gamma"], x["omega"], x["phi"],
                                       want_D=False, want_state=True)
    S.device_status()
    slots = [0, 1, 143, 144, 4000, 5183, 9071, 9215]
    gen = W.generator(w.seed + 100 * B, dev())
    q, k, v = W.decode_tokens(N, 64, 64, steps, gen)
    S0 = Sx.reshape(N, 384, 64)
    z0 = zx.reshape(N, 384)
    Sd, zd = S0.clone(), z0.clone()
    od = torch.empty(steps, N, 64, device=dev())
    for i in range(steps):
        pos = torch.full((N,), 4096 + i, dtype=torch.int64, device=dev())
        S.sanatan_decode_step(Sd, zd, q[i], k[i], v[i], x["gamma"], x["omega"], x["phi"], pos,
                              out=od[i])
    # the same tokens as 64 sequences x 144 heads (slot n = 144 b + h uses head h's parameters)
    seqs = lambda t: _stack_tokens(t).reshape(B, G, steps, 64)  # noqa: E731
    oc, _, _, _ = S.sanatan_chunk_fwd(seqs(q), seqs(k), seqs(v), x["gamma"], x["omega"], x["phi"],
                                      pos0=4096, S0=Sx, z0=zx, want_D=False)
    torch.cuda.synchronize()
    assert (oc.reshape(N, steps, 64) - od.permute(1, 0, 2)).abs().max().item() <= 1e-4

    sl = torch.tensor(slots, device=dev())
    b_idx, h_idx = [n // G for n in slots], [n % G for n in slots]
    kk = torch.stack([x["k"][b, h] for b, h in zip(b_idx, h_idx)])[None]
    vv = torch.stack([x["v"][b, h] for b, h in zip(b_idx, h_idx)])[None]
    gam = f64(x["gamma"])[h_idx]
    om = f64(x["omega"])[h_idx]
    ph = f64(x["phi"])[h_idx]
    S_ref, z_ref = O.final_state(f64(kk), f64(vv), gam, om, ph)
    assert rel_fro(f64(S0[sl]), S_ref[0]) <= 5e-3
    assert rel_fro(f64(z0[sl]), z_ref[0]) <= 5e-3
    Sr, zr = S_ref[0], z_ref[0]
    for i in range(steps):
        Sr, zr, o_ref = O.decode_step(Sr, zr, f64(q[i][sl]), f64(k[i][sl]), f64(v[i][sl]), gam,
                                      om, ph, np.full(len(slots), 4096 + i))
        assert max_abs(f64(od[i][sl]), o_ref) <= 5e-3, i
