"""Thin ctypes binding to libdspark.so: argument marshalling only.

Every function takes torch tensors that already live on the GPU (or None where
the C ABI allows NULL), passes their data pointers and the current CUDA
stream, and raises DSparkError on a non-OK status.  No computation happens
here; there is no CPU fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_LIB = None

DSPARK_BF16 = 0
DSPARK_F32 = 1

SYMBOLS = (
    "dspark_status_string",
    "dspark_last_error",
    "dspark_version",
    "dspark_workspace_bytes",
    "dspark_device_status",
    "dspark_draft_sample",
    "dspark_confidence",
    "dspark_schedule",
    "dspark_verify",
    "dspark_launch_count",
    "dspark_trace_start",
    "dspark_trace_stop",
    "dspark_trace_collect",
    "dspark_trace_kinds",
    "dspark_trace_get",
    "dspark_schedule_noalloc",
    "dspark_draft_schedule",
    "dspark_check_wait_timeout",
    "dspark_schedule_async",
    "dspark_draft_sample_rnn",
    "dspark_verify_rnn",
)


class DSparkError(RuntimeError):
    def __init__(self, fn, code, msg):
        super().__init__(f"{fn} failed: {code} ({msg})")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load the in-tree libdspark.so (it must have been built; see build.py)."""
    global _LIB
    if _LIB is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"libdspark.so not built at {path}; run "
                               "`python -m draft_sampling_lossless_gb300.build`")
        L = ctypes.CDLL(path)
        c_int, c_float, c_size, vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p
        L.dspark_status_string.restype = ctypes.c_char_p
        L.dspark_status_string.argtypes = [c_int]
        L.dspark_last_error.restype = ctypes.c_char_p
        L.dspark_last_error.argtypes = []
        L.dspark_version.restype = ctypes.c_char_p
        L.dspark_version.argtypes = []
        L.dspark_workspace_bytes.restype = c_size
        L.dspark_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int]
        L.dspark_device_status.restype = c_int
        L.dspark_device_status.argtypes = [vp, c_int, ctypes.POINTER(ctypes.c_uint32), vp]
        L.dspark_draft_sample.restype = c_int
        L.dspark_draft_sample.argtypes = [c_int, c_int, c_int, c_int, c_float, vp, vp, vp, c_int,
                                          vp, vp, vp, vp, vp, vp, c_size, vp]
        L.dspark_confidence.restype = c_int
        L.dspark_confidence.argtypes = [c_int, c_int, c_int, c_int, c_int, vp, vp, vp, c_int, vp,
                                        vp, vp, vp, vp, vp, vp, c_size, vp]
        L.dspark_schedule.restype = c_int
        L.dspark_schedule.argtypes = [c_int, c_int, vp, vp, c_int, c_int, c_int, vp, vp, vp, vp,
                                      vp, c_size, vp]
        L.dspark_verify.restype = c_int
        L.dspark_verify.argtypes = [c_int, c_int, c_int, c_int, c_float, vp, vp, vp, c_int, vp,
                                    vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, vp, vp, vp, vp,
                                    vp, c_size, vp]
        L.dspark_schedule_noalloc.restype = c_int
        L.dspark_schedule_noalloc.argtypes = [c_int, c_int, vp, vp, c_int, c_int, c_int, vp, vp,
                                              vp, vp, vp, vp]
        L.dspark_draft_schedule.restype = c_int
        L.dspark_draft_schedule.argtypes = [c_int, c_int, c_int, c_int, c_float, vp, vp, vp, c_int,
                                            vp, vp, c_int, vp, vp, vp, vp, vp, vp, c_int, c_int,
                                            c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, c_size,
                                            vp]
        L.dspark_schedule_async.restype = c_int
        L.dspark_schedule_async.argtypes = [c_int, c_int, vp, vp, vp, vp, vp, vp, vp, c_size, vp]
        L.dspark_draft_sample_rnn.restype = c_int
        L.dspark_draft_sample_rnn.argtypes = [c_int, c_int, c_int, c_int, c_float, vp, vp, vp, vp,
                                              c_int, vp, vp, vp, vp, vp, vp, vp, c_size, vp]
        L.dspark_verify_rnn.restype = c_int
        L.dspark_verify_rnn.argtypes = [c_int, c_int, c_int, c_int, c_float, vp, vp, vp, c_int,
                                        vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, vp, vp, vp,
                                        vp, vp, c_size, vp]
        L.dspark_check_wait_timeout.restype = c_int
        L.dspark_check_wait_timeout.argtypes = [c_int, vp, c_size, vp]
        L.dspark_launch_count.restype = ctypes.c_longlong
        L.dspark_launch_count.argtypes = []
        for f in ("dspark_trace_start", "dspark_trace_stop", "dspark_trace_collect",
                  "dspark_trace_kinds"):
            getattr(L, f).restype = c_int
            getattr(L, f).argtypes = []
        L.dspark_trace_get.restype = c_int
        L.dspark_trace_get.argtypes = [c_int, ctypes.POINTER(ctypes.c_char_p),
                                       ctypes.POINTER(ctypes.c_longlong),
                                       ctypes.POINTER(ctypes.c_double)]
        _LIB = L
    return _LIB


def launch_count() -> int:
    return int(lib().dspark_launch_count())


def trace_start():
    _check("dspark_trace_start", lib().dspark_trace_start())


def trace_stop():
    lib().dspark_trace_stop()


def trace_collect() -> int:
    n = lib().dspark_trace_collect()
    if n < 0:
        raise DSparkError("dspark_trace_collect", "DSPARK_ERR_CUDA", "event read failed")
    return n


def trace_totals() -> dict:
    """{kernel name: (launches, total ms)} accumulated since trace_start()."""
    L = lib()
    out = {}
    for i in range(L.dspark_trace_kinds()):
        name, cnt, ms = ctypes.c_char_p(), ctypes.c_longlong(), ctypes.c_double()
        _check("dspark_trace_get", L.dspark_trace_get(i, ctypes.byref(name), ctypes.byref(cnt),
                                                      ctypes.byref(ms)))
        out[name.value.decode()] = (int(cnt.value), float(ms.value))
    return out


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor or None")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdspark must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dt(t) -> int:
    if t.dtype == torch.bfloat16:
        return DSPARK_BF16
    if t.dtype == torch.float32:
        return DSPARK_F32
    raise TypeError(f"unsupported element type {t.dtype}")


def _check(fn, code):
    if code != 0:
        L = lib()
        raise DSparkError(fn, L.dspark_status_string(code).decode(), L.dspark_last_error().decode())


def version() -> str:
    return lib().dspark_version().decode()


def workspace_bytes(R, gamma, V, r, n_sps=0) -> int:
    return int(lib().dspark_workspace_bytes(R, gamma, V, r, n_sps))


def alloc_workspace(R, gamma, V, r, n_sps=0, device="cuda") -> torch.Tensor:
    """A zeroed workspace (uint8) sized for every call at these sizes."""
    n = workspace_bytes(R, gamma, V, r, n_sps)
    if n == 0:
        raise ValueError("sizes out of range")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def device_status(ws, clear=False, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    _check("dspark_device_status",
           lib().dspark_device_status(_p(ws), int(clear), ctypes.byref(flags), _stream(stream)))
    return int(flags.value)


def dspark_draft_sample(z, E, Wt, anchor, u_draft, temperature, tokens, q_lse, q_tok, ws,
                        stream=None):
    R, G, V = z.shape
    r = E.shape[1]
    _check("dspark_draft_sample", lib().dspark_draft_sample(
        R, G, V, r, float(temperature), _p(z), _p(E), _p(Wt), _dt(z), _p(anchor), _p(u_draft),
        _p(tokens), _p(q_lse), _p(q_tok), _p(ws), ws.numel(), _stream(stream)))


def dspark_draft_sample_rnn(z, E, U, Wt, anchor, u_draft, temperature, tokens, q_lse, q_tok, S,
                            ws, stream=None):
    R, G, V = z.shape
    r = E.shape[1]
    _check("dspark_draft_sample_rnn", lib().dspark_draft_sample_rnn(
        R, G, V, r, float(temperature), _p(z), _p(E), _p(U), _p(Wt), _dt(z), _p(anchor),
        _p(u_draft), _p(tokens), _p(q_lse), _p(q_tok), _p(S), _p(ws), ws.numel(),
        _stream(stream)))


def dspark_confidence(R, gamma, hidden, w, E1, anchor, tokens, sts_t, c_in, c_out, a_out, ws,
                      stream=None):
    if c_in is None:
        d = hidden.shape[2]
        V, r = E1.shape
        dt = _dt(hidden)
    else:
        d, V, r, dt = 0, 2, 1, DSPARK_F32
    _check("dspark_confidence", lib().dspark_confidence(
        R, gamma, d, r, V, _p(hidden), _p(w), _p(E1), dt, _p(anchor), _p(tokens), _p(sts_t),
        _p(c_in), _p(c_out), _p(a_out), _p(ws), ws.numel(), _stream(stream)))


def dspark_schedule(a, sps, early_stop, max_B, ell, row_off, B_out, E_out, ws, stream=None):
    R, G = a.shape
    _check("dspark_schedule", lib().dspark_schedule(
        R, G, _p(a), _p(sps), sps.numel(), int(early_stop), int(max_B), _p(ell), _p(row_off),
        _p(B_out), _p(E_out), _p(ws), ws.numel(), _stream(stream)))


def dspark_schedule_async(a, capacity, ell, row_off, B_out, E_out, ws, stream=None):
    """Capacity scheduling: capacity is a one-element int32 device tensor."""
    R, G = a.shape
    _check("dspark_schedule_async", lib().dspark_schedule_async(
        R, G, _p(a), _p(capacity), _p(ell), _p(row_off), _p(B_out), _p(E_out), _p(ws), ws.numel(),
        _stream(stream)))


def dspark_draft_schedule(z, E, Wt, anchor, u_draft, temperature, hidden, w, E1, sts_t, c_in,
                          sps, early_stop, max_B, tokens, q_lse, q_tok, c_out, a_out, ell,
                          row_off, B_out, E_out, ws, stream=None):
    R, G, V = z.shape
    r = E.shape[1]
    d = hidden.shape[2] if hidden is not None else 0
    _check("dspark_draft_schedule", lib().dspark_draft_schedule(
        R, G, V, r, float(temperature), _p(z), _p(E), _p(Wt), _dt(z), _p(anchor), _p(u_draft),
        d, _p(hidden), _p(w), _p(E1), _p(sts_t), _p(c_in), _p(sps), sps.numel(),
        int(early_stop), int(max_B), _p(tokens), _p(q_lse), _p(q_tok), _p(c_out), _p(a_out),
        _p(ell), _p(row_off), _p(B_out), _p(E_out), _p(ws), ws.numel(), _stream(stream)))


def dspark_verify(z, E, Wt, anchor, tokens, q_lse, q_tok, ell, row_off, target, u_acc, u_fin,
                  temperature, n_acc, out_tokens, p_lse, ws, stream=None):
    R, G, V = z.shape
    r = E.shape[1]
    _check("dspark_verify", lib().dspark_verify(
        R, G, V, r, float(temperature), _p(z), _p(E), _p(Wt), _dt(z), _p(anchor), _p(tokens),
        _p(q_lse), _p(q_tok), _p(ell), _p(row_off), _p(target), target.shape[0], _p(u_acc),
        _p(u_fin), _p(n_acc), _p(out_tokens), _p(p_lse), _p(ws), ws.numel(), _stream(stream)))


def dspark_verify_rnn(z, S, Wt, tokens, q_lse, q_tok, ell, row_off, target, u_acc, u_fin,
                      temperature, n_acc, out_tokens, p_lse, ws, stream=None):
    R, G, V = z.shape
    r = S.shape[2]
    _check("dspark_verify_rnn", lib().dspark_verify_rnn(
        R, G, V, r, float(temperature), _p(z), _p(S), _p(Wt), _dt(z), _p(tokens), _p(q_lse),
        _p(q_tok), _p(ell), _p(row_off), _p(target), target.shape[0], _p(u_acc), _p(u_fin),
        _p(n_acc), _p(out_tokens), _p(p_lse), _p(ws), ws.numel(), _stream(stream)))


def dspark_schedule_noalloc(a, sps, early_stop, max_B, ell, row_off, B_out, E_out,
                            dev_status=None, stream=None):
    """The scheduler with library-internal static scratch (no workspace): for
    callers that cannot allocate device memory.  Calls sharing a process must
    not overlap on the GPU."""
    R, G = a.shape
    _check("dspark_schedule_noalloc", lib().dspark_schedule_noalloc(
        R, G, _p(a), _p(sps), sps.numel(), int(early_stop), int(max_B), _p(ell), _p(row_off),
        _p(B_out), _p(E_out), _p(dev_status), _stream(stream)))


def dspark_check_wait_timeout(limit_us, ws, stream=None):
    """Runs the library's bounded waits against barriers nothing completes
    (diagnostic); afterwards the workspace's status word has the timeout bit."""
    _check("dspark_check_wait_timeout",
           lib().dspark_check_wait_timeout(int(limit_us), _p(ws), ws.numel(), _stream(stream)))
