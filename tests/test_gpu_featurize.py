"""sanatan_featurize against the float64 oracle's feature map."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import dev, f64, max_abs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("in_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pos0", [0, 4093, 1 << 25])
def test_featurize_f32_out(in_dtype, pos0):
    w = W.LAYER if in_dtype == "bf16" else W.TINY
    x = W.make(w, B=2, H=3, T=77)
    if w.phi_kind == "zero":
        x["phi"] = W.rates(3, 64, "geometric")
    u = x["q"].to(dev())
    out = S.sanatan_featurize(u, x["gamma"].to(dev()), x["omega"].to(dev()), x["phi"].to(dev()),
                              pos0=pos0)
    torch.cuda.synchronize()
    ref = O.featurize(f64(x["q"]), f64(x["gamma"]), f64(x["omega"]), f64(x["phi"]), pos0)
    assert max_abs(f64(out), ref) <= 5e-6


def test_featurize_bf16_out_is_rounded_f32():
    x = W.make(W.LAYER, B=1, H=2, T=130)
    args = [x[n].to(dev()) for n in ("gamma", "omega", "phi")]
    u = x["k"].to(dev())
    out = S.sanatan_featurize(u, *args, pos0=11, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ref = O.featurize(f64(x["k"]), f64(x["gamma"]), f64(x["omega"]), f64(x["phi"]), 11)
    # one bf16 rounding of a value in [-1, 1]: at most half an ulp of 1 (2^-8)
    assert max_abs(f64(out), ref) <= 2.0 ** -8 + 1e-6
    assert np.all(f64(out)[..., 0::6] == 1.0)


def test_featurize_empty():
    x = W.make(W.LAYER, B=1, H=2, T=0)
    out = S.sanatan_featurize(x["q"].to(dev()), *(x[n].to(dev()) for n in ("gamma", "omega", "phi")))
    assert out.shape == (1, 2, 0, 384)
