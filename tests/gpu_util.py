"""Shared helpers of the GPU parity tests (input plumbing only)."""
import numpy as np
import torch

from constant_state_recurrence_gb300 import workloads as W

f64 = W.to_f64


def dev():
    return torch.device("cuda:0")


def to_dev(x, names=("q", "k", "v", "gamma", "omega", "phi", "dO")):
    return {n: x[n].to(dev()) for n in names if n in x}


def ref_args(x):
    return dict(q=f64(x["q"]), k=f64(x["k"]), v=f64(x["v"]), gamma=f64(x["gamma"]),
                omega=f64(x["omega"]), phi=f64(x["phi"]))


def max_abs(a, b):
    return float(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)).max())


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
