"""The rate parameterisation lambda = 0.01 tanh(lambda_raw) (reading notes
§2.2, eq. (4)) on the GPU, and its gradient chained with the backward's dphi,
against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import dev, f64, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu


def test_rate_from_raw_and_gradient():
    g = torch.Generator().manual_seed(5)
    raw = torch.randn(12, 64, generator=g) * 3
    dphi = torch.randn(12, 64, generator=g)
    phi = S.rate_from_raw(raw.to(dev()))
    dl = S.rate_from_raw_bwd(raw.to(dev()), dphi.to(dev()))
    torch.cuda.synchronize()
    assert np.abs(f64(phi) - O.rate_from_raw(f64(raw))).max() <= 1e-8
    assert np.abs(f64(dl) - O.rate_from_raw_grad(f64(raw), f64(dphi))).max() <= 1e-7


def test_attention_trained_through_raw_rates():
    """The rates of a head come from lambda_raw; the gradient of sum(o dO) in
    lambda_raw is the backward's dphi pulled back through the tanh."""
    x = W.make(W.TRAIN, B=1, H=2, T=300, with_grad_out=True)
    raw = torch.randn(2, 64, generator=torch.Generator().manual_seed(8))
    g = to_dev(x)
    phi = S.rate_from_raw(raw.to(dev()))
    o, D, _, _ = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], phi)
    gr = S.sanatan_chunk_bwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], phi, o, D, g["dO"],
                             want_dphi=True)
    dl = S.rate_from_raw_bwd(raw.to(dev()), gr["dphi"])
    S.device_status()
    ra = ref_args(x)
    ra["phi"] = O.rate_from_raw(f64(raw))
    ref = O.attn_backward(**ra, dO=f64(x["dO"]))
    want = O.rate_from_raw_grad(f64(raw), ref["dphi"])
    assert rel_fro(f64(dl), want) <= 1e-2
