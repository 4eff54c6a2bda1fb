"""Failure detection on the GPU without a fault: a bounded device-side wait
that runs out.  The library's probe kernel waits, with the same bounded
mbarrier wait as the tensor-core kernels, on a barrier that nothing arrives
at; after its limit (1 ms here) it gives up and records a timeout, which the
host then reads through sanatan_device_status.  The context must stay usable:
the next attention call is correct and reports no error."""
import numpy as np
import pytest

import oracle.sanatan_oracle as O
from constant_state_recurrence_gb300 import sanatan as S
from constant_state_recurrence_gb300 import workloads as W
from gpu_util import f64, max_abs, ref_args, to_dev

pytestmark = pytest.mark.gpu


def _small_forward_is_correct():
    x = W.make(W.LAYER, B=1, H=2, T=300)
    g = to_dev(x)
    o, _, _, _ = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"])
    S.device_status()
    o_ref, _ = O.attn_quadratic(**ref_args(x))
    assert max_abs(f64(o), o_ref) <= 5e-3


def test_wait_that_nothing_completes_reports_timeout_and_context_survives():
    S.device_status()                       # start clean
    S.selftest_wait_timeout(1_000_000)      # 1 ms limit, nobody arrives
    with pytest.raises(S.SanatanError) as err:
        S.device_status()
    assert err.value.status == 5            # SANATAN_ERR_TIMEOUT
    S.device_status()                       # the flag was cleared by the read
    _small_forward_is_correct()


def test_wait_that_completes_reports_nothing():
    S.device_status()
    S.selftest_wait_timeout(1_000_000, arrive=True)
    S.device_status()
    _small_forward_is_correct()


def test_timeout_then_every_path_still_clean():
    S.selftest_wait_timeout(1_000_000)
    with pytest.raises(S.SanatanError):
        S.device_status()
    x = W.make(W.TRAIN, B=1, H=2, T=200, with_grad_out=True)
    g = to_dev(x)
    o, D, _, _ = S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"])
    gr = S.sanatan_chunk_bwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], o, D,
                             g["dO"])
    op, _ = S.sanatan_power_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 2)
    S.device_status()
    ref = O.attn_backward(**ref_args(x), dO=f64(x["dO"]))
    rel = np.linalg.norm(f64(gr["dq"]) - ref["dq"]) / np.linalg.norm(ref["dq"])
    assert rel <= 1e-2
    op_ref, _ = O.attn_power(**ref_args(x), p=2)
    assert max_abs(f64(op), op_ref) <= 5e-3
