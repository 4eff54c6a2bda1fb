"""sanatan_chunk_fwd_noalloc: the tensor-core forward for callers that cannot
allocate device scratch (e.g. a plugin that only receives its input and output
buffers, or code where cudaMalloc's implicit device synchronisation is not
allowed).  It must give the results of sanatan_chunk_fwd, which uses a
caller-allocated workspace, on two calls in a row (the fixed scratch array
keeps the previous call's contents).

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test."""
import ctypes

import pytest
import torch

from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL_BF16 = 5e-3


def _ref(g):
    return S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                               want_state=True)


def _noalloc_raw(g, o, D, Sx, zx):
    """Call the entry point through the C ABI directly."""
    B, H, T, d = g["q"].shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return S.lib().sanatan_chunk_fwd_noalloc(
        p(g["q"]), p(g["k"]), p(g["v"]), p(g["gamma"]), p(g["omega"]), p(g["phi"]), B, H, T, d,
        64, 0, 0.0, None, None, p(o), p(D), p(Sx), p(zx),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


# (8, 12, 4096): the preferred split (three segments for 96 sequences) needs
# more scratch than the array holds, so the entry point uses fewer segments.
@pytest.mark.parametrize("shape", [(4, 12, 2048), (1, 3, 700), (8, 12, 4096)])
def test_noalloc_matches_workspace_entry_twice(shape):
    dev = torch.device("cuda:0")
    B, H, T = shape
    for call in range(2):
        x = W.make(W.LAYER, device="cpu", B=B, H=H, T=T - 37 * call)
        g = {n: x[n].to(dev) for n in ("q", "k", "v", "gamma", "omega", "phi")}
        o_ref, D_ref, S_ref, z_ref = _ref(g)
        Tn = x["T"]
        o = torch.full((B, H, Tn, 64), float("nan"), device=dev)
        D = torch.full((B, H, Tn), float("nan"), device=dev)
        Sx = torch.full((B, H, 384, 64), float("nan"), device=dev)
        zx = torch.full((B, H, 384), float("nan"), device=dev)
        assert _noalloc_raw(g, o, D, Sx, zx) == 0
        S.device_status()
        assert (o - o_ref).abs().max().item() <= TOL_BF16
        assert (D - D_ref).abs().max().item() <= TOL_BF16 * D_ref.abs().max().item()
        assert ((Sx - S_ref).norm() / S_ref.norm()).item() <= TOL_BF16
        assert ((zx - z_ref).norm() / z_ref.norm()).item() <= TOL_BF16


@pytest.mark.parametrize("shape", [(200, 1, 8), (64, 12, 4096)])
def test_noalloc_runs_problems_whose_split_needs_no_scratch(shape):
    """Problems with more sequences than the array has per-segment slots (more
    than 163 here) run with one segment per sequence, which needs no scratch:
    200 single-chunk sequences, and the batched-decode prefill (64 x 12
    sequences of 4096 tokens)."""
    cap = S.lib().sanatan_chunk_fwd_noalloc_max_scratch_bytes()
    assert cap == 16 << 20
    dev = torch.device("cuda:0")
    B, H, T = shape
    assert S.chunk_fwd_plan(B, H, T)[0] == 1
    assert S.chunk_fwd_workspace_size(B, H, T) == 0
    x = W.make(W.LAYER, device=dev, B=B, H=H, T=T)
    g = {n: x[n] for n in ("q", "k", "v", "gamma", "omega", "phi")}
    for _ in range(2):
        o_ref, D_ref, S_ref, z_ref = _ref(g)
        o, D, Sx, zx = S.sanatan_chunk_fwd_noalloc(g["q"], g["k"], g["v"], g["gamma"], g["omega"],
                                                   g["phi"], want_state=True)
        S.device_status()
        assert (o - o_ref).abs().max().item() <= TOL_BF16
        assert ((Sx - S_ref).norm() / S_ref.norm()).item() <= TOL_BF16
        assert ((zx - z_ref).norm() / z_ref.norm()).item() <= TOL_BF16
        del o, D, Sx, zx, o_ref, D_ref, S_ref, z_ref
