"""SANATAN p=1 root-parity gated angular attention on GB300 (sm_103a).

The compute path is the C-ABI library ``libsanatan.so`` (hand-written CUDA
kernels); :mod:`constant_state_recurrence_gb300.sanatan` is its thin ctypes
binding.  :mod:`constant_state_recurrence_gb300.workloads` holds the seeded
synthetic inputs.  Importing this package loads nothing; the binding loads the
library on first use and raises if it is missing.
"""
__all__ = ["sanatan", "workloads"]
