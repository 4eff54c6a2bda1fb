"""The bf16 tensor-core chunked forward against the float64 oracle
(max abs error <= 5e-3 on outputs: bf16 operands, f32 accumulation).

The oracle consumes the same bf16-rounded inputs promoted to float64."""
import numpy as np
import pytest
import torch

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import dev, f64, max_abs, ref_args, rel_fro, to_dev

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3      # outputs, max abs
TOL_STATE = 5e-3     # emitted S, z: relative Frobenius
TOL_DEN = 2e-3       # denominator, relative Frobenius


def run(x, **kw):
    g = to_dev(x)
    out = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                              want_state=True, **kw)
    S.device_status()
    return out


def check_full(x, pos0=0, eps=0.0, S0=None, z0=None):
    o, D, Sx, zx = run(x, pos0=pos0, eps=eps,
                       S0=None if S0 is None else S0.to(dev()),
                       z0=None if z0 is None else z0.to(dev()))
    ra = ref_args(x)
    S0r = None if S0 is None else f64(S0)
    z0r = None if z0 is None else f64(z0)
    o_ref, D_ref = O.attn_quadratic(**ra, pos0=pos0, eps=eps, S0=S0r, z0=z0r)
    S_ref, z_ref = O.final_state(ra["k"], ra["v"], ra["gamma"], ra["omega"], ra["phi"], pos0=pos0,
                                 S0=S0r, z0=z0r)
    err = max_abs(f64(o), o_ref)
    assert err <= TOL_BF16, err
    assert rel_fro(f64(D), D_ref) <= TOL_DEN
    assert rel_fro(f64(Sx), S_ref) <= TOL_STATE
    assert rel_fro(f64(zx), z_ref) <= TOL_STATE
    return err


@pytest.mark.parametrize("T", [1, 64, 127, 128, 129, 300])
def test_short_sequences(T):
    x = W.make(W.LAYER, B=1, H=2, T=T)
    check_full(x)


def test_many_segments_one_sequence():
    # 16 chunks spread over 16 segments (delta pass + scan + main pass)
    x = W.make(W.LAYER, B=1, H=1, T=2000)
    check_full(x)


def test_single_segment_many_sequences():
    # more sequences than SMs: one segment per sequence, no workspace traffic
    x = W.make(W.LAYER, B=2, H=80, T=200)
    o, D, Sx, zx = run(x)
    ra = ref_args(x)
    for b, h in ((0, 0), (1, 79), (0, 41)):
        sl = {n: ra[n][b:b + 1, h:h + 1] for n in ("q", "k", "v")}
        o_ref, _ = O.attn_quadratic(**sl, gamma=ra["gamma"][h:h + 1], omega=ra["omega"][h:h + 1],
                                    phi=ra["phi"][h:h + 1])
        assert max_abs(f64(o)[b, h], o_ref[0, 0]) <= TOL_BF16


def test_initial_state_eps_and_offset():
    x = W.make(W.LAYER, B=2, H=3, T=257)
    rng = np.random.default_rng(3)
    kp = rng.standard_normal((2, 3, 100, 64))
    vp = rng.standard_normal((2, 3, 100, 64))
    S0, z0 = O.final_state(kp, vp, f64(x["gamma"]), f64(x["omega"]), f64(x["phi"]), pos0=900)
    check_full(x, pos0=1000, eps=0.75, S0=torch.tensor(S0, dtype=torch.float32),
               z0=torch.tensor(z0, dtype=torch.float32))


def test_outputs_do_not_depend_on_position_offset():
    x = W.make(W.LAYER, B=1, H=2, T=400)
    o1, _, _, _ = run(x, pos0=0)
    o2, _, _, _ = run(x, pos0=50000)
    assert max_abs(f64(o1), f64(o2)) <= 2 * TOL_BF16


def _whole_tensor_check(x):
    """Every output of every (batch, head) against the oracle's recurrent form
    (eq. (9)) on the same bf16-rounded inputs: o element-wise (max abs), D and
    the final S, z per sequence by relative Frobenius norm."""
    o, D, Sx, zx = run(x)
    ra = ref_args(x)
    o_ref, D_ref, S_ref, z_ref = O.attn_recurrent(ra["q"], ra["k"], ra["v"], ra["gamma"],
                                                  ra["omega"], ra["phi"])
    err = max_abs(f64(o), o_ref)
    assert err <= TOL_BF16, err
    B, H = x["B"], x["H"]
    Dg, Sg, zg = f64(D), f64(Sx), f64(zx)
    for b in range(B):
        for h in range(H):
            assert rel_fro(Dg[b, h], D_ref[b, h]) <= TOL_DEN, (b, h)
            assert rel_fro(Sg[b, h], S_ref[b, h]) <= TOL_STATE, (b, h)
            assert rel_fro(zg[b, h], z_ref[b, h]) <= TOL_STATE, (b, h)
    return err


def test_layer_forward_full_size_whole_tensor():
    """B=4, H=12, T=2048 in the benchmarked launch configuration (three
    segments per sequence): every output against the oracle."""
    x = W.make(W.LAYER, device="cpu")
    _whole_tensor_check(x)


def test_long_prefill_full_size_whole_tensor():
    """B=1, H=12, T=32768 (twelve segments per sequence): every output and the
    final S, z of every head against the oracle."""
    x = W.make(W.LONG, device="cpu")
    _whole_tensor_check(x)


def test_training_shape_forward_full_size_whole_tensor():
    """B=8, H=12, T=4096 (96 sequences: the multi-wave segment split, three
    segments per sequence, 288 CTAs): every output against the oracle."""
    assert S.chunk_fwd_plan(8, 12, 4096)[0] >= 2
    x = W.make(W.TRAIN, device="cpu")
    _whole_tensor_check(x)


@pytest.mark.parametrize("H,slices", [(2, 1), (2, 2), (2, 4), (2, 8), (6, 8), (6, 12)])
def test_host_forward_pipeline(H, slices):
    """HostForward: pinned host q, k, v in, host o out, pipelined over slices
    of the sequences (whole batch rows, or head ranges of one row with their
    own gamma, omega, phi) on three streams; the outputs are those of the
    definition."""
    x = W.make(W.LAYER, device="cpu", B=4, H=H, T=300)
    hq, hk, hv = (x[n].pin_memory() for n in ("q", "k", "v"))
    ho = torch.full((4, H, 300, 64), float("nan")).pin_memory()
    g = to_dev(x, ("gamma", "omega", "phi"))
    hf = S.HostForward(4, H, 300, slices=slices)
    o_ref, _ = O.attn_quadratic(**ref_args(x))
    for _ in range(2):
        hf(hq, hk, hv, g["gamma"], g["omega"], g["phi"], ho)
        torch.cuda.current_stream().synchronize()
        S.device_status()
        assert max_abs(f64(ho), o_ref) <= TOL_BF16
    # the same pipeline captured as one CUDA graph and replayed
    hf.capture(hq, hk, hv, g["gamma"], g["omega"], g["phi"], ho)
    for _ in range(2):
        ho.fill_(float("nan"))
        hf.replay()
        torch.cuda.current_stream().synchronize()
        S.device_status()
        assert max_abs(f64(ho), o_ref) <= TOL_BF16


def test_empty_sequences_copy_the_initial_state():
    """T = 0 on the bf16 path: no output rows; the exported state is (S0, z0),
    or zeros without one."""
    x = W.make(W.LAYER, device="cpu", B=2, H=3, T=0)
    g = to_dev(x)
    S0 = torch.randn(2, 3, 384, 64, device=dev())
    z0 = torch.rand(2, 3, 384, device=dev())
    o, D, Sx, zx = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                       S0=S0, z0=z0, want_state=True)
    torch.cuda.synchronize()
    S.device_status()
    assert o.shape == (2, 3, 0, 64) and D.shape == (2, 3, 0)
    assert torch.equal(Sx, S0) and torch.equal(zx, z0)
    _, _, Sz, zz = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                       want_state=True)
    torch.cuda.synchronize()
    assert not Sz.any() and not zz.any()
