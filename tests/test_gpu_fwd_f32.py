"""The all-float32 chunked forward against the float64 oracle (tolerance 1e-5
on outputs, the f32-operand bar)."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import dev, f64, max_abs, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-5


def test_tiny_workload_full_size():
    x = W.make(W.TINY)
    g = to_dev(x)
    o, D, Sx, zx = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                       want_state=True)
    torch.cuda.synchronize()
    o_ref, D_ref = O.attn_quadratic(**ref_args(x))
    assert max_abs(f64(o), o_ref) <= TOL_F32
    assert rel_fro(f64(D), D_ref) <= 1e-6
    S_ref, z_ref = O.final_state(f64(x["k"]), f64(x["v"]), f64(x["gamma"]), f64(x["omega"]),
                                 f64(x["phi"]))
    assert rel_fro(f64(Sx), S_ref) <= TOL_F32 and rel_fro(f64(zx), z_ref) <= TOL_F32


@pytest.mark.parametrize("T", [1, 31, 33, 65, 100])
def test_ragged_lengths_with_state_eps_and_offset(T):
    x = W.make(W.TINY, B=2, H=3, T=T)
    x["phi"] = W.rates(3, 64, "geometric")
    rng = np.random.default_rng(T)
    kp = rng.standard_normal((2, 3, 40, 64))
    vp = rng.standard_normal((2, 3, 40, 64))
    S0, z0 = O.final_state(kp, vp, f64(x["gamma"]), f64(x["omega"]), f64(x["phi"]), pos0=60)
    S0 = torch.tensor(S0, dtype=torch.float32)
    z0 = torch.tensor(z0, dtype=torch.float32)
    g = to_dev(x)
    o, D, Sx, zx = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                       pos0=100, eps=0.5, S0=S0.to(dev()), z0=z0.to(dev()),
                                       want_state=True)
    torch.cuda.synchronize()
    ra = ref_args(x)
    o_ref, D_ref = O.attn_quadratic(**ra, pos0=100, eps=0.5, S0=f64(S0), z0=f64(z0))
    assert max_abs(f64(o), o_ref) <= TOL_F32
    assert rel_fro(f64(D), D_ref) <= 1e-6
    S_ref, z_ref = O.final_state(ra["k"], ra["v"], ra["gamma"], ra["omega"], ra["phi"], pos0=100,
                                 S0=f64(S0), z0=f64(z0))
    assert rel_fro(f64(Sx), S_ref) <= TOL_F32 and rel_fro(f64(zx), z_ref) <= TOL_F32


def test_empty_sequence_copies_state():
    x = W.make(W.TINY, B=1, H=2, T=0)
    S0 = torch.randn(1, 2, 384, 64)
    z0 = torch.randn(1, 2, 384)
    g = to_dev(x)
    o, D, Sx, zx = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                       S0=S0.to(dev()), z0=z0.to(dev()), want_state=True)
    torch.cuda.synchronize()
    assert torch.equal(Sx.cpu(), S0) and torch.equal(zx.cpu(), z0)
