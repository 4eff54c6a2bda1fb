"""Thin ctypes binding of libsanatan.so (C ABI declared in include/sanatan.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and the current CUDA
stream.  The library is loaded on first use; if it has not been built, every
call raises RuntimeError (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libsanatan.so")

SANATAN_F32 = 0
SANATAN_BF16 = 1
_DT = {torch.float32: SANATAN_F32, torch.bfloat16: SANATAN_BF16}

_c_int, _c_i64, _c_f, _c_sz, _c_p = (ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                     ctypes.c_size_t, ctypes.c_void_p)

_SIGS = {
    "sanatan_status_string": (ctypes.c_char_p, [_c_int]),
    "sanatan_abi_version": (_c_int, []),
    "sanatan_state_bytes": (_c_sz, [_c_int] * 4),
    "sanatan_featurize": (_c_int, [_c_p, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int, _c_int,
                                   _c_i64, _c_p, _c_int, _c_p]),
    "sanatan_rate_from_raw": (_c_int, [_c_p, _c_int, _c_f, _c_p, _c_p]),
    "sanatan_rate_from_raw_bwd": (_c_int, [_c_p, _c_p, _c_int, _c_f, _c_p, _c_p]),
    "sanatan_eps_raw": (_c_f, [_c_f, _c_int, _c_int]),
    "sanatan_chunk_fwd_workspace_size": (_c_sz, [_c_int] * 6),
    "sanatan_chunk_fwd_plan": (_c_int, [_c_int] * 5 + [_c_p, _c_p]),
    "sanatan_chunk_fwd": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _c_i64, _c_f, _c_p, _c_p, _c_p, _c_p,
                                   _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "sanatan_chunk_fwd_noalloc_max_scratch_bytes": (_c_sz, []),
    "sanatan_chunk_fwd_noalloc": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int,
                                           _c_int, _c_int, _c_int, _c_i64, _c_f, _c_p, _c_p, _c_p,
                                           _c_p, _c_p, _c_p, _c_p]),
    "sanatan_chunk_bwd_workspace_size": (_c_sz, [_c_int] * 6),
    "sanatan_chunk_bwd": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int,
                                   _c_int, _c_int, _c_int, _c_i64, _c_f, _c_p, _c_p, _c_p, _c_p,
                                   _c_p, _c_int, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_sz,
                                   _c_p]),
    "sanatan_power_fwd_workspace_size": (_c_sz, [_c_int] * 5),
    "sanatan_power_fwd": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int,
                                   _c_int, _c_int, _c_i64, _c_int, _c_f, _c_p, _c_p, _c_p, _c_sz,
                                   _c_p]),
    "sanatan_ablation_fwd": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int,
                                      _c_int, _c_int, _c_i64, _c_int, _c_int, _c_f, _c_f, _c_p,
                                      _c_p, _c_p, _c_sz, _c_p]),
    "sanatan_power_bwd_workspace_size": (_c_sz, [_c_int] * 5),
    "sanatan_power_bwd": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int,
                                   _c_int, _c_int, _c_i64, _c_int, _c_f, _c_p, _c_p, _c_p, _c_int,
                                   _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "sanatan_device_status": (_c_int, [_c_p]),
    "sanatan_set_profile_events": (_c_int, [_c_p, _c_p]),
    "sanatan_selftest_wait_timeout": (_c_int, [ctypes.c_uint64, _c_int, _c_p]),
    "sanatan_stack_decode_workspace_size": (_c_sz, [_c_int] * 3),
    "sanatan_stack_decode_step": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                                           _c_int, _c_int, _c_int, _c_int, _c_f, _c_p, _c_sz,
                                           _c_p]),
    "sanatan_state_bytes_harmonic": (_c_sz, [_c_int] * 5),
    "sanatan_featurize_harmonic": (_c_int, [_c_p, _c_int, _c_p, _c_p, _c_p, _c_int, _c_int, _c_int,
                                            _c_int, _c_i64, _c_int, _c_p, _c_int, _c_p]),
    "sanatan_chunk_fwd_harmonic": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p, _c_int,
                                            _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_f,
                                            _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p]),
    "sanatan_chunk_bwd_harmonic_workspace_size": (_c_sz, [_c_int] * 6),
    "sanatan_chunk_bwd_harmonic": (_c_int, [_c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p, _c_int,
                                            _c_int, _c_int, _c_int, _c_int, _c_i64, _c_int, _c_f,
                                            _c_p, _c_p, _c_p, _c_p, _c_p, _c_int, _c_p, _c_p, _c_p,
                                            _c_p, _c_p, _c_p, _c_p, _c_sz, _c_p]),
    "sanatan_decode_step_harmonic": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p,
                                              _c_p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f,
                                              _c_p, _c_p]),
    "sanatan_decode_step": (_c_int, [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_p, _c_int,
                                     _c_int, _c_int, _c_int, _c_f, _c_p, _c_p]),
}

_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded library with argument types set (raises if not built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -m constant_state_recurrence_gb300.build` (there is no fallback)")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in _SIGS.items():
                    fn = getattr(handle, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = handle
    return _lib


def exported_symbols():
    return list(_SIGS)


class SanatanError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = lib().sanatan_status_string(status).decode()
        super().__init__(f"{fn} failed with status {status}: {msg}")


def _check(fn, status):
    if status != 0:
        raise SanatanError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _need(t, name, dtypes=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _need_params(gamma, omega, phi, H, d):
    """gamma [H], omega [H, d], phi [H, d] float32 on the device (the kernels
    read H rows of each)."""
    _need(gamma, "gamma", (torch.float32,), (H,))
    _need(omega, "omega", (torch.float32,), (H, d))
    _need(phi, "phi", (torch.float32,), (H, d))


def device_status(device=None):
    """Synchronise the current stream and raise if a kernel of the library gave
    up a bounded device-side wait since the last check."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check("sanatan_device_status", lib().sanatan_device_status(_stream(dev)))


def selftest_wait_timeout(timeout_ns=1_000_000, arrive=False, device=None):
    """Enqueue the library's failure-detection probe: a bounded wait on an
    mbarrier nobody arrives at (or, with arrive=True, one that completes)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check("sanatan_selftest_wait_timeout",
           lib().sanatan_selftest_wait_timeout(int(timeout_ns), int(bool(arrive)), _stream(dev)))


def set_profile_events(start=None, stop=None):
    """Record torch.cuda.Event `start`/`stop` around the dominant kernel of the
    following chunk_fwd / chunk_bwd calls of this thread (None, None: off)."""
    for ev in (start, stop):
        if ev is not None and ev.cuda_event == 0:
            ev.record()  # torch creates the CUDA event lazily, on first record
    a = None if start is None else ctypes.c_void_p(start.cuda_event)
    b = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    _check("sanatan_set_profile_events", lib().sanatan_set_profile_events(a, b))


def state_bytes(layers, heads, d=64, dv=64):
    return int(lib().sanatan_state_bytes(layers, heads, d, dv))


def sanatan_featurize(u, gamma, omega, phi, pos0=0, out_dtype=None, out=None):
    """Phi(u) [B, H, T, 6d] (index 6a + c) for u [B, H, T, d]."""
    _need(u, "u", (torch.float32, torch.bfloat16))
    B, H, T, d = u.shape
    odt = out_dtype or torch.float32
    if out is None:
        out = torch.empty(B, H, T, 6 * d, dtype=odt, device=u.device)
    _need(out, "out", (torch.float32, torch.bfloat16), (B, H, T, 6 * d))
    _need_params(gamma, omega, phi, H, d)
    st = lib().sanatan_featurize(_ptr(u), _DT[u.dtype], _ptr(gamma), _ptr(omega), _ptr(phi),
                                 B, H, T, d, int(pos0), _ptr(out), _DT[out.dtype],
                                 _stream(u.device))
    _check("sanatan_featurize", st)
    return out


RATE_SCALE = 0.01   # the pages' lambda = 0.01 tanh(lambda_raw)


def rate_from_raw(lambda_raw, scale=RATE_SCALE, out=None):
    """phi = scale * tanh(lambda_raw) (float32, on the device)."""
    _need(lambda_raw, "lambda_raw", (torch.float32,))
    out = torch.empty_like(lambda_raw) if out is None else out
    _need(out, "phi", (torch.float32,), tuple(lambda_raw.shape))
    _check("sanatan_rate_from_raw",
           lib().sanatan_rate_from_raw(_ptr(lambda_raw), lambda_raw.numel(), float(scale),
                                       _ptr(out), _stream(lambda_raw.device)))
    return out


def rate_from_raw_bwd(lambda_raw, dphi, scale=RATE_SCALE, out=None):
    """dlambda_raw = dphi * scale * (1 - tanh^2(lambda_raw))."""
    _need(lambda_raw, "lambda_raw", (torch.float32,))
    _need(dphi, "dphi", (torch.float32,), tuple(lambda_raw.shape))
    out = torch.empty_like(lambda_raw) if out is None else out
    _check("sanatan_rate_from_raw_bwd",
           lib().sanatan_rate_from_raw_bwd(_ptr(lambda_raw), _ptr(dphi), lambda_raw.numel(),
                                           float(scale), _ptr(out), _stream(lambda_raw.device)))
    return out


def eps_raw(eps, d=64, convention=0):
    """c * eps with c = 4d + 1e-6 (convention 0) or 4d * 1e-6 (convention 1)."""
    return float(lib().sanatan_eps_raw(float(eps), int(d), int(convention)))


def chunk_fwd_workspace_size(B, H, T, d=64, dv=64, dtype=torch.bfloat16):
    return int(lib().sanatan_chunk_fwd_workspace_size(B, H, T, d, dv, _DT[dtype]))


def chunk_fwd_plan(B, H, T, dtype=torch.bfloat16, has_initial_state=False):
    """(segments per sequence, kernel launches per call) of sanatan_chunk_fwd."""
    seg, nl = ctypes.c_int(0), ctypes.c_int(0)
    _check("sanatan_chunk_fwd_plan",
           lib().sanatan_chunk_fwd_plan(B, H, T, _DT[dtype], int(bool(has_initial_state)),
                                        ctypes.byref(seg), ctypes.byref(nl)))
    return seg.value, nl.value


def sanatan_chunk_fwd(q, k, v, gamma, omega, phi, pos0=0, eps=0.0, S0=None, z0=None,
                      want_D=True, want_state=False, out=None, D_out=None, workspace=None):
    """Causal p=1 attention over [B, H, T] sequences.

    Returns (o [B,H,T,dv] f32, D [B,H,T] f32 or None, S [B,H,6d,dv] or None,
    z [B,H,6d] or None)."""
    _need(q, "q", (torch.float32, torch.bfloat16))
    B, H, T, d = q.shape
    _need(k, "k", (q.dtype,), (B, H, T, d))
    _need(v, "v", (q.dtype,))
    dv = v.shape[-1]
    _need(v, "v", (q.dtype,), (B, H, T, dv))
    _need_params(gamma, omega, phi, H, d)
    dev = q.device
    F = 6 * d
    o = out if out is not None else torch.empty(B, H, T, dv, dtype=torch.float32, device=dev)
    _need(o, "o", (torch.float32,), (B, H, T, dv))
    D = D_out
    if D is None and want_D:
        D = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    if D is not None:
        _need(D, "D", (torch.float32,), (B, H, T))
    S = z = None
    if want_state:
        S = torch.empty(B, H, F, dv, dtype=torch.float32, device=dev)
        z = torch.empty(B, H, F, dtype=torch.float32, device=dev)
    if S0 is not None:
        _need(S0, "S0", (torch.float32,), (B, H, F, dv))
        _need(z0, "z0", (torch.float32,), (B, H, F))
    ws_size = int(lib().sanatan_chunk_fwd_workspace_size(B, H, T, d, dv, _DT[q.dtype]))
    if workspace is None and ws_size > 0:
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().sanatan_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(gamma),
                                 _ptr(omega), _ptr(phi), B, H, T, d, dv, int(pos0), float(eps),
                                 _ptr(S0), _ptr(z0), _ptr(o), _ptr(D), _ptr(S), _ptr(z),
                                 _ptr(workspace), ws_bytes, _stream(dev))
    _check("sanatan_chunk_fwd", st)
    return o, D, S, z


class HostForward:
    """sanatan_chunk_fwd over pinned HOST tensors q, k, v (bf16 [B, H, T, d])
    into a pinned host o (f32 [B, H, T, dv]), pipelined over slices of the B * H
    sequences: the host-to-device copy of slice i + 1, the attention of slice
    i and the device-to-host copy of slice i - 1 run on three CUDA streams at
    once (one cudaMemcpyAsync per tensor slice).  A slice is m = B * H / slices
    consecutive sequences: whole batch rows when H divides m, else m heads of
    one batch row (then m must divide H), with the matching rows of gamma,
    omega and phi.  Device staging (two slices of q, k, v and o, and the
    workspace) is allocated once, here, with torch; each call then allocates
    nothing.  The calling stream waits for the last copy, so `o` is complete
    once that stream is synchronised."""

    def __init__(self, B, H, T, d=64, dv=64, slices=4, device=None):
        n_seq = B * H
        if slices < 1 or n_seq % slices:
            raise ValueError("B * H must be a multiple of slices")
        m = n_seq // slices
        if not (m % H == 0 or H % m == 0):
            raise ValueError("a slice must hold whole batch rows or divide one")
        self.dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.B, self.H, self.T, self.d, self.dv, self.n, self.m = B, H, T, d, dv, slices, m
        # device shape of one slice
        self.shape = (m // H, H) if m % H == 0 else (1, m)
        sb, sh = self.shape
        mk = lambda dt, last: [torch.empty(sb, sh, T, last, dtype=dt, device=self.dev)  # noqa: E731
                               for _ in range(2)]
        self.q, self.k, self.v = mk(torch.bfloat16, d), mk(torch.bfloat16, d), mk(torch.bfloat16, dv)
        self.o = mk(torch.float32, dv)
        ws = chunk_fwd_workspace_size(sb, sh, T, d, dv)
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=self.dev)
        self.s_in = torch.cuda.Stream(self.dev)
        self.s_run = torch.cuda.Stream(self.dev)
        self.s_out = torch.cuda.Stream(self.dev)
        self.loaded = [torch.cuda.Event() for _ in range(2)]
        self.done = [torch.cuda.Event() for _ in range(2)]
        self.freed_in = [torch.cuda.Event() for _ in range(2)]
        self.freed_out = [torch.cuda.Event() for _ in range(2)]
        # per head range of a sub-row slice: its own (16-byte aligned) copies of
        # gamma, omega, phi, refreshed at every call
        self.params = {}
        if sh < H:
            for h0 in range(0, H, sh):
                self.params[h0] = (torch.empty(sh, device=self.dev),
                                   torch.empty(sh, d, device=self.dev),
                                   torch.empty(sh, d, device=self.dev))

    def _part(self, t, i):
        """Slice i of a [B, H, ...] host tensor, shaped like the device slice."""
        sb, sh = self.shape
        if sh == self.H:
            return t[i * sb:(i + 1) * sb]
        b, h0 = divmod(i * sh, self.H)
        return t[b:b + 1, h0:h0 + sh]


    def __call__(self, qh, kh, vh, gamma, omega, phi, oh, pos0=0, eps=0.0):
        for t, n in ((qh, "q"), (kh, "k"), (vh, "v"), (oh, "o")):
            if t.is_cuda or not t.is_pinned():
                raise ValueError(f"{n} must be a pinned host tensor")
        caller = torch.cuda.current_stream(self.dev)
        for st in (self.s_in, self.s_run, self.s_out):
            st.wait_stream(caller)
        sh = self.shape[1]
        if self.params:
            with torch.cuda.stream(self.s_run):
                for h0, (g, w, f) in self.params.items():
                    g.copy_(gamma[h0:h0 + sh])
                    w.copy_(omega[h0:h0 + sh])
                    f.copy_(phi[h0:h0 + sh])
        for i in range(self.n + 2):
            j = i % 2
            if i < self.n:                      # H2D of slice i into buffer j
                with torch.cuda.stream(self.s_in):
                    if i >= 2:
                        self.s_in.wait_event(self.freed_in[j])
                    self.q[j].copy_(self._part(qh, i), non_blocking=True)
                    self.k[j].copy_(self._part(kh, i), non_blocking=True)
                    self.v[j].copy_(self._part(vh, i), non_blocking=True)
                    self.loaded[j].record(self.s_in)
            if 1 <= i <= self.n:                # attention of slice i - 1
                jj = (i - 1) % 2
                g, w, f = (gamma, omega, phi) if not self.params else \
                    self.params[((i - 1) * sh) % self.H]
                with torch.cuda.stream(self.s_run):
                    self.s_run.wait_event(self.loaded[jj])
                    if i - 1 >= 2:
                        self.s_run.wait_event(self.freed_out[jj])
                    sanatan_chunk_fwd(self.q[jj], self.k[jj], self.v[jj], g, w, f, pos0=pos0,
                                      eps=eps, want_D=False, out=self.o[jj], workspace=self.ws)
                    self.freed_in[jj].record(self.s_run)
                    self.done[jj].record(self.s_run)
            if i >= 2:                          # D2H of slice i - 2
                jj = (i - 2) % 2
                with torch.cuda.stream(self.s_out):
                    self.s_out.wait_event(self.done[jj])
                    self._part(oh, i - 2).copy_(self.o[jj], non_blocking=True)
                    self.freed_out[jj].record(self.s_out)
        caller.wait_stream(self.s_out)
        return oh

    def capture(self, qh, kh, vh, gamma, omega, phi, oh, pos0=0, eps=0.0):
        """Record one call on these (fixed) host and parameter tensors as a CUDA
        graph -- every copy and kernel of the pipeline, on its three streams --
        so that replay() enqueues the whole step with one launch.  The call is
        run once first (warm-up outside the capture)."""
        self(qh, kh, vh, gamma, omega, phi, oh, pos0, eps)
        torch.cuda.current_stream(self.dev).synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self(qh, kh, vh, gamma, omega, phi, oh, pos0, eps)
        return self

    def replay(self):
        """One step of the captured pipeline on the current stream."""
        self.graph.replay()


def sanatan_chunk_fwd_noalloc(q, k, v, gamma, omega, phi, pos0=0, eps=0.0, S0=None, z0=None,
                              want_D=True, want_state=False):
    """sanatan_chunk_fwd for bf16 inputs without a workspace: the library uses
    its own fixed 16 MiB device scratch instead (for callers that cannot
    allocate).  Calls must not overlap on the GPU.  Returns (o, D, S, z)."""
    _need(q, "q", (torch.bfloat16,))
    B, H, T, d = q.shape
    _need(k, "k", (torch.bfloat16,), (B, H, T, d))
    dv = v.shape[-1]
    _need(v, "v", (torch.bfloat16,), (B, H, T, dv))
    _need_params(gamma, omega, phi, H, d)
    dev = q.device
    F = 6 * d
    o = torch.empty(B, H, T, dv, dtype=torch.float32, device=dev)
    D = torch.empty(B, H, T, dtype=torch.float32, device=dev) if want_D else None
    S = z = None
    if want_state:
        S = torch.empty(B, H, F, dv, dtype=torch.float32, device=dev)
        z = torch.empty(B, H, F, dtype=torch.float32, device=dev)
    st = lib().sanatan_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(omega),
                                         _ptr(phi), B, H, T, d, dv, int(pos0), float(eps),
                                         _ptr(S0), _ptr(z0), _ptr(o), _ptr(D), _ptr(S), _ptr(z),
                                         _stream(dev))
    _check("sanatan_chunk_fwd_noalloc", st)
    return o, D, S, z


def power_fwd_workspace_size(B, H, T, d=64, dv=64):
    return int(lib().sanatan_power_fwd_workspace_size(B, H, T, d, dv))


def sanatan_power_fwd(q, k, v, gamma, omega, phi, p, pos0=0, eps=0.0, want_D=True, out=None,
                      D_out=None, workspace=None):
    """Power-sharpened causal attention at integer power p (bf16 q, k, v).

    Returns (o [B,H,T,dv] f32, D [B,H,T] f32 or None)."""
    _need(q, "q", (torch.bfloat16,))
    B, H, T, d = q.shape
    _need(k, "k", (torch.bfloat16,), (B, H, T, d))
    dv = v.shape[-1]
    _need(v, "v", (torch.bfloat16,), (B, H, T, dv))
    _need_params(gamma, omega, phi, H, d)
    dev = q.device
    o = out if out is not None else torch.empty(B, H, T, dv, dtype=torch.float32, device=dev)
    _need(o, "o", (torch.float32,), (B, H, T, dv))
    D = D_out
    if D is None and want_D:
        D = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    if D is not None:
        _need(D, "D", (torch.float32,), (B, H, T))
    ws_size = power_fwd_workspace_size(B, H, T, d, dv)
    if workspace is None and ws_size > 0:
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().sanatan_power_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(omega), _ptr(phi),
                                 B, H, T, d, dv, int(pos0), int(p), float(eps), _ptr(o), _ptr(D),
                                 _ptr(workspace), ws_bytes, _stream(dev))
    _check("sanatan_power_fwd", st)
    return o, D


def power_bwd_workspace_size(B, H, T, d=64, dv=64):
    return int(lib().sanatan_power_bwd_workspace_size(B, H, T, d, dv))


def sanatan_power_bwd(q, k, v, gamma, omega, phi, p, o, D, dO, pos0=0, eps=0.0, want_dphi=True,
                      workspace=None):
    """Gradients of sum(o * dO) for sanatan_power_fwd (bf16 q, k, v).

    Returns a dict with dq, dk, dv (bf16), dgamma, domega and dphi (f32; dphi
    None unless want_dphi)."""
    _need(q, "q", (torch.bfloat16,))
    B, H, T, d = q.shape
    _need(k, "k", (torch.bfloat16,), (B, H, T, d))
    dv_ = v.shape[-1]
    _need(v, "v", (torch.bfloat16,), (B, H, T, dv_))
    _need(o, "o", (torch.float32,), (B, H, T, dv_))
    _need(D, "D", (torch.float32,), (B, H, T))
    _need(dO, "dO", (torch.float32, torch.bfloat16), (B, H, T, dv_))
    _need_params(gamma, omega, phi, H, d)
    dev = q.device
    dq, dk, dvo = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dgamma = torch.empty(H, dtype=torch.float32, device=dev)
    domega = torch.empty(H, d, dtype=torch.float32, device=dev)
    dphi = torch.empty(H, d, dtype=torch.float32, device=dev) if want_dphi else None
    ws_size = power_bwd_workspace_size(B, H, T, d, dv_)
    if workspace is None and ws_size > 0:
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().sanatan_power_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(omega), _ptr(phi),
                                 B, H, T, d, dv_, int(pos0), int(p), float(eps), _ptr(o), _ptr(D),
                                 _ptr(dO), _DT[dO.dtype], _ptr(dq), _ptr(dk), _ptr(dvo),
                                 _ptr(dgamma), _ptr(domega), _ptr(dphi), _ptr(workspace),
                                 ws_bytes, _stream(dev))
    _check("sanatan_power_bwd", st)
    return dict(dq=dq, dk=dk, dv=dvo, dgamma=dgamma, domega=domega, dphi=dphi)


def sanatan_ablation_fwd(q, k, v, gamma, omega, phi, p, channels, shift=0.0, pos0=0, eps=0.0,
                         want_D=True, out=None, D_out=None, workspace=None):
    """Power-sharpened causal attention with the four-channel (clipped) or the
    three-channel (optionally shifted) ablation map; bf16 q, k, v, p in {1, 2, 4}.

    Returns (o [B,H,T,dv] f32, D [B,H,T] f32 or None)."""
    _need(q, "q", (torch.bfloat16,))
    B, H, T, d = q.shape
    _need(k, "k", (torch.bfloat16,), (B, H, T, d))
    dv = v.shape[-1]
    _need(v, "v", (torch.bfloat16,), (B, H, T, dv))
    _need_params(gamma, omega, phi, H, d)
    dev = q.device
    o = out if out is not None else torch.empty(B, H, T, dv, dtype=torch.float32, device=dev)
    _need(o, "o", (torch.float32,), (B, H, T, dv))
    D = D_out
    if D is None and want_D:
        D = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    if D is not None:
        _need(D, "D", (torch.float32,), (B, H, T))
    ws_size = power_fwd_workspace_size(B, H, T, d, dv)
    if workspace is None and ws_size > 0:
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().sanatan_ablation_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(gamma), _ptr(omega),
                                    _ptr(phi), B, H, T, d, dv, int(pos0), int(p), int(channels),
                                    float(shift), float(eps), _ptr(o), _ptr(D), _ptr(workspace),
                                    ws_bytes, _stream(dev))
    _check("sanatan_ablation_fwd", st)
    return o, D


def chunk_bwd_workspace_size(B, H, T, d=64, dv=64, dtype=torch.bfloat16):
    return int(lib().sanatan_chunk_bwd_workspace_size(B, H, T, d, dv, _DT[dtype]))


def sanatan_chunk_bwd(q, k, v, gamma, omega, phi, o, D, dO, pos0=0, eps=0.0, S0=None, z0=None,
                      want_dphi=False, workspace=None, fwd_workspace=None):
    """Gradients of sum(o * dO): dict(dq, dk, dv, dgamma, domega, dphi).

    fwd_workspace: the workspace the forward that produced o and D ran with (on
    these same inputs), so that its per-segment state sums are reused."""
    _need(q, "q", (torch.float32, torch.bfloat16))
    B, H, T, d = q.shape
    dv = v.shape[-1]
    _need(k, "k", (q.dtype,), (B, H, T, d))
    _need(v, "v", (q.dtype,), (B, H, T, dv))
    _need(o, "o", (torch.float32,), (B, H, T, dv))
    _need(D, "D", (torch.float32,), (B, H, T))
    _need(dO, "dO", (torch.float32, torch.bfloat16), (B, H, T, dv))
    _need_params(gamma, omega, phi, H, d)
    dev = q.device
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    dgamma = torch.empty(H, dtype=torch.float32, device=dev)
    domega = torch.empty(H, d, dtype=torch.float32, device=dev)
    dphi = torch.empty(H, d, dtype=torch.float32, device=dev) if want_dphi else None
    ws_size = int(lib().sanatan_chunk_bwd_workspace_size(B, H, T, d, dv, _DT[q.dtype]))
    if workspace is None and ws_size > 0:
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().sanatan_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(gamma),
                                 _ptr(omega), _ptr(phi), B, H, T, d, dv, int(pos0), float(eps),
                                 _ptr(S0), _ptr(z0), _ptr(o), _ptr(D), _ptr(dO), _DT[dO.dtype],
                                 _ptr(dq), _ptr(dk), _ptr(dvv), _ptr(dgamma), _ptr(domega),
                                 _ptr(dphi), _ptr(workspace), ws_bytes, _ptr(fwd_workspace),
                                 0 if fwd_workspace is None else
                                 fwd_workspace.numel() * fwd_workspace.element_size(),
                                 _stream(dev))
    _check("sanatan_chunk_bwd", st)
    return dict(dq=dq, dk=dk, dv=dvv, dgamma=dgamma, domega=domega, dphi=dphi)


def sanatan_decode_step(S, z, q, k, v, gamma, omega, phi, pos, eps=0.0, out=None):
    """One decode token for N slots; S [N,6d,dv] and z [N,6d] are updated in
    place.  Returns o [N, dv] f32."""
    _need(q, "q", (torch.float32,))
    N, d = q.shape
    _need(k, "k", (torch.float32,), (N, d))
    _need(v, "v", (torch.float32,))
    dv = v.shape[-1]
    F = 6 * d
    _need(S, "S", (torch.float32,), (N, F, dv))
    _need(z, "z", (torch.float32,), (N, F))
    _need(pos, "pos", (torch.int64,), (N,))
    G = gamma.shape[0]
    _need(gamma, "gamma", (torch.float32,), (G,))
    _need(omega, "omega", (torch.float32,), (G, d))
    _need(phi, "phi", (torch.float32,), (G, d))
    o = out if out is not None else torch.empty(N, dv, dtype=torch.float32, device=q.device)
    _need(o, "o", (torch.float32,), (N, dv))
    st = lib().sanatan_decode_step(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v), _ptr(gamma),
                                   _ptr(omega), _ptr(phi), _ptr(pos), N, G, d, dv, float(eps),
                                   _ptr(o), _stream(q.device))
    _check("sanatan_decode_step", st)
    return o


def sanatan_stack_decode_step(x, Wqkv, Wo, S, z, gamma, omega, phi, pos, eps=0.0,
                              workspace=None):
    """One token through L attention layers; x [B, heads*64] is updated in
    place (and returned), S [L, B*heads, 384, 64] and z [L, B*heads, 384] too.
    gamma [L, heads], omega and phi [L, heads, 64], pos [B*heads] int64."""
    _need(x, "x", (torch.float32,))
    B, Dm = x.shape
    L, heads = gamma.shape
    d = Dm // heads
    _need(Wqkv, "Wqkv", (torch.float32,), (L, Dm, 3 * Dm))
    _need(Wo, "Wo", (torch.float32,), (L, Dm, Dm))
    _need(S, "S", (torch.float32,), (L, B * heads, 6 * d, d))
    _need(z, "z", (torch.float32,), (L, B * heads, 6 * d))
    _need(gamma, "gamma", (torch.float32,), (L, heads))
    _need(omega, "omega", (torch.float32,), (L, heads, d))
    _need(phi, "phi", (torch.float32,), (L, heads, d))
    _need(pos, "pos", (torch.int64,), (B * heads,))
    ws_n = int(lib().sanatan_stack_decode_workspace_size(B, heads, d))
    if workspace is None:
        workspace = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=x.device)
    _check("sanatan_stack_decode_step",
           lib().sanatan_stack_decode_step(_ptr(x), _ptr(Wqkv), _ptr(Wo), _ptr(S), _ptr(z),
                                           _ptr(gamma), _ptr(omega), _ptr(phi), _ptr(pos), B, L,
                                           heads, d, float(eps), _ptr(workspace),
                                           workspace.numel(), _stream(x.device)))
    return x


def harmonic_features(harmonics, d=64):
    """F_N = 2 (2N + 1) d features of the harmonic map."""
    return 2 * (2 * harmonics + 1) * d


def sanatan_featurize_harmonic(u, gamma, omega, phi, harmonics, pos0=0, out_dtype=None):
    """Phi_N(u) [B, H, T, F_N] of the harmonic map."""
    _need(u, "u", (torch.float32, torch.bfloat16))
    B, H, T, d = u.shape
    _need_params(gamma, omega, phi, H, d)
    out = torch.empty(B, H, T, harmonic_features(harmonics, d), dtype=out_dtype or torch.float32,
                      device=u.device)
    _check("sanatan_featurize_harmonic",
           lib().sanatan_featurize_harmonic(_ptr(u), _DT[u.dtype], _ptr(gamma), _ptr(omega),
                                            _ptr(phi), B, H, T, d, int(pos0), int(harmonics),
                                            _ptr(out), _DT[out.dtype], _stream(u.device)))
    return out


def sanatan_chunk_fwd_harmonic(q, k, v, gamma, omega, phi, harmonics, pos0=0, eps=0.0, S0=None,
                               z0=None, want_D=True, want_state=False):
    """Causal p=1 attention with the harmonic map (float32 on the CUDA cores).
    Returns (o, D or None, S [B,H,F_N,dv] or None, z [B,H,F_N] or None)."""
    _need(q, "q", (torch.float32, torch.bfloat16))
    B, H, T, d = q.shape
    _need(k, "k", (q.dtype,), (B, H, T, d))
    dv = v.shape[-1]
    _need(v, "v", (q.dtype,), (B, H, T, dv))
    _need_params(gamma, omega, phi, H, d)
    F = harmonic_features(harmonics, d)
    dev = q.device
    o = torch.empty(B, H, T, dv, dtype=torch.float32, device=dev)
    D = torch.empty(B, H, T, dtype=torch.float32, device=dev) if want_D else None
    Sx = zx = None
    if want_state:
        Sx = torch.empty(B, H, F, dv, dtype=torch.float32, device=dev)
        zx = torch.empty(B, H, F, dtype=torch.float32, device=dev)
    if S0 is not None:
        _need(S0, "S0", (torch.float32,), (B, H, F, dv))
        _need(z0, "z0", (torch.float32,), (B, H, F))
    _check("sanatan_chunk_fwd_harmonic",
           lib().sanatan_chunk_fwd_harmonic(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(gamma),
                                            _ptr(omega), _ptr(phi), B, H, T, d, dv, int(pos0),
                                            int(harmonics), float(eps), _ptr(S0), _ptr(z0),
                                            _ptr(o), _ptr(D), _ptr(Sx), _ptr(zx), _stream(dev)))
    return o, D, Sx, zx


def sanatan_chunk_bwd_harmonic(q, k, v, gamma, omega, phi, harmonics, o, D, dO, pos0=0, eps=0.0,
                               S0=None, z0=None, want_dphi=False, workspace=None):
    """Gradients of sum(o * dO) for sanatan_chunk_fwd_harmonic: dict(dq, dk, dv,
    dgamma, domega, dphi)."""
    _need(q, "q", (torch.float32, torch.bfloat16))
    B, H, T, d = q.shape
    dv = v.shape[-1]
    _need(k, "k", (q.dtype,), (B, H, T, d))
    _need(v, "v", (q.dtype,), (B, H, T, dv))
    _need(o, "o", (torch.float32,), (B, H, T, dv))
    _need(D, "D", (torch.float32,), (B, H, T))
    _need(dO, "dO", (torch.float32, torch.bfloat16), (B, H, T, dv))
    _need_params(gamma, omega, phi, H, d)
    dev = q.device
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dvv = torch.empty_like(v)
    dgamma = torch.empty(H, dtype=torch.float32, device=dev)
    domega = torch.empty(H, d, dtype=torch.float32, device=dev)
    dphi = torch.empty(H, d, dtype=torch.float32, device=dev) if want_dphi else None
    ws_size = int(lib().sanatan_chunk_bwd_harmonic_workspace_size(B, H, T, d, dv,
                                                                   int(harmonics)))
    if workspace is None and ws_size > 0:
        workspace = torch.empty(ws_size, dtype=torch.uint8, device=dev)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().sanatan_chunk_bwd_harmonic(_ptr(q), _ptr(k), _ptr(v), _DT[q.dtype], _ptr(gamma),
                                          _ptr(omega), _ptr(phi), B, H, T, d, dv, int(pos0),
                                          int(harmonics), float(eps), _ptr(S0), _ptr(z0), _ptr(o),
                                          _ptr(D), _ptr(dO), _DT[dO.dtype], _ptr(dq), _ptr(dk),
                                          _ptr(dvv), _ptr(dgamma), _ptr(domega), _ptr(dphi),
                                          _ptr(workspace), ws_bytes, _stream(dev))
    _check("sanatan_chunk_bwd_harmonic", st)
    return dict(dq=dq, dk=dk, dv=dvv, dgamma=dgamma, domega=domega, dphi=dphi)


def sanatan_decode_step_harmonic(S, z, q, k, v, gamma, omega, phi, pos, harmonics, eps=0.0):
    """One decode token with the harmonic map; S [N,F_N,dv], z [N,F_N] in place."""
    _need(q, "q", (torch.float32,))
    N, d = q.shape
    _need(k, "k", (torch.float32,), (N, d))
    dv = v.shape[-1]
    _need(v, "v", (torch.float32,), (N, dv))
    F = harmonic_features(harmonics, d)
    _need(S, "S", (torch.float32,), (N, F, dv))
    _need(z, "z", (torch.float32,), (N, F))
    _need(pos, "pos", (torch.int64,), (N,))
    G = gamma.shape[0]
    _need_params(gamma, omega, phi, G, d)
    o = torch.empty(N, dv, dtype=torch.float32, device=q.device)
    _check("sanatan_decode_step_harmonic",
           lib().sanatan_decode_step_harmonic(_ptr(S), _ptr(z), _ptr(q), _ptr(k), _ptr(v),
                                              _ptr(gamma), _ptr(omega), _ptr(phi), _ptr(pos), N,
                                              G, d, dv, int(harmonics), float(eps), _ptr(o),
                                              _stream(q.device)))
    return o


class SanatanAttention(torch.autograd.Function):
    """autograd wrapper: forward = sanatan_chunk_fwd, backward = sanatan_chunk_bwd."""

    @staticmethod
    def forward(ctx, q, k, v, gamma, omega, phi, pos0=0, eps=0.0):
        B, H, T, d = q.shape
        ws_size = chunk_fwd_workspace_size(B, H, T, d, v.shape[-1], q.dtype)
        ws = torch.empty(max(ws_size, 16), dtype=torch.uint8, device=q.device)
        o, D, _, _ = sanatan_chunk_fwd(q, k, v, gamma, omega, phi, pos0=pos0, eps=eps,
                                       workspace=ws)
        ctx.save_for_backward(q, k, v, gamma, omega, phi, o, D)
        ctx.pos0, ctx.eps = pos0, eps
        ctx.fwd_ws = ws   # its per-segment state sums serve the backward
        return o

    @staticmethod
    def backward(ctx, dO):
        q, k, v, gamma, omega, phi, o, D = ctx.saved_tensors
        g = sanatan_chunk_bwd(q, k, v, gamma, omega, phi, o, D, dO.contiguous(), pos0=ctx.pos0,
                              eps=ctx.eps, want_dphi=True, fwd_workspace=ctx.fwd_ws)
        return g["dq"], g["dk"], g["dv"], g["dgamma"], g["domega"], g["dphi"], None, None
