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


@pytest.mark.parametrize("N,G", [(144, 144), (300, 144), (7, 3), (400, 144), (700, 144)])
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
