"""The C++ CPU oracle (oracle/dspark_oracle.cpp) behind the same Python API
as the numpy oracle (TEST INFRASTRUCTURE ONLY: used by the tests, the
package smoke check and the benchmark's CPU-baseline leg).

build() compiles it with g++ (OpenMP, no FMA contraction, no
machine-specific flags) into oracle/libdspark_oracle.so.  Every function
takes float64 / integer numpy arrays; OpenMP splits independent requests
over set_threads(n) threads (default: every core this process may use).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dspark_oracle.cpp")
LIB = os.path.join(HERE, "libdspark_oracle.so")
CXXFLAGS = ["-O3", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]

_L = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + ".tmp"
        cxx = os.environ.get("CXX", "g++")
        r = subprocess.run([cxx, *CXXFLAGS, SRC, "-o", tmp], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"oracle build failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


def _lib():
    global _L
    if _L is None:
        build()
        L = ctypes.CDLL(LIB)
        i, i64, d, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        sig = {
            "oc_set_threads": (None, [i]),
            "oc_get_threads": (i, []),
            "oc_markov_bias": (None, [i, i, i, vp, vp, vp, vp]),
            "oc_softmax_rows": (None, [i, i, vp, vp, vp]),
            "oc_inverse_cdf": (None, [i, i, vp, vp, vp]),
            "oc_first_argmax": (None, [i, i, vp, vp]),
            "oc_to_fixed": (None, [i64, vp, vp]),
            "oc_draft_distribution": (None, [i, i, i, d, vp, vp, vp, vp, vp]),
            "oc_draft_sample": (None, [i, i, i, i, d, vp, vp, vp, vp, vp, vp, vp, vp]),
            "oc_confidence": (None, [i, i, i, i, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "oc_schedule": (i, [i, i, vp, vp, i64, i, i64, vp, vp, vp, vp, vp, vp, vp]),
            "oc_schedule_capacity": (None, [i, i, vp, i64, vp, vp, vp, vp, vp]),
            "oc_verify": (None, [i, i, i, i, d, vp, vp, vp, vp, vp, vp, vp, vp, i64, vp, vp,
                                 vp, vp, vp, vp, vp, vp]),
            "oc_final_weights": (None, [i, i, d, vp, vp, vp, i64, vp, i, vp, vp]),
            "oc_draft_sample_rnn": (None, [i, i, i, i, i, d, vp, vp, vp, vp, vp, vp, vp, vp,
                                           vp, vp]),
            "oc_rnn_states": (None, [i, i, i, i, vp, vp, vp, vp, vp]),
            "oc_round_state": (None, [i64, i, vp, vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _L = L
        set_threads(len(os.sched_getaffinity(0)))
    return _L


def set_threads(n: int) -> None:
    _lib().oc_set_threads(int(n))


def threads() -> int:
    return int(_lib().oc_get_threads())


def _f(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _i(x):
    return np.ascontiguousarray(x, dtype=np.int64)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------- helpers

def markov_bias(E, W, prev):
    E, W, prev = _f(E), _f(W), _i(np.atleast_1d(prev))
    V, r = E.shape
    out = np.empty((prev.shape[0], W.shape[1]))
    _lib().oc_markov_bias(prev.shape[0], W.shape[1], r, _p(E), _p(W), _p(prev), _p(out))
    return out


def inverse_cdf(weights, u):
    w, u = _f(weights), _f(np.atleast_1d(u))
    out = np.empty(w.shape[0], dtype=np.int64)
    _lib().oc_inverse_cdf(w.shape[0], w.shape[1], _p(w), _p(u), _p(out))
    return out


def first_argmax(y):
    y = _f(y)
    out = np.empty(y.shape[0], dtype=np.int64)
    _lib().oc_first_argmax(y.shape[0], y.shape[1], _p(y), _p(out))
    return out


def softmax_rows(y):
    y = _f(y)
    e = np.empty_like(y)
    lse = np.empty(y.shape[0])
    _lib().oc_softmax_rows(y.shape[0], y.shape[1], _p(y), _p(e), _p(lse))
    return e, lse


def to_fixed(a):
    a = _f(a)
    out = np.empty(a.shape, dtype=np.int64)
    _lib().oc_to_fixed(a.size, _p(a), _p(out))
    return out


def draft_distribution(z_k, E, W, prev, T):
    z_k, E, W, prev = _f(z_k), _f(E), _f(W), _i(np.atleast_1d(prev))
    q = np.empty_like(z_k)
    _lib().oc_draft_distribution(z_k.shape[0], z_k.shape[1], E.shape[1], float(T), _p(z_k),
                                 _p(E), _p(W), _p(prev), _p(q))
    return q


def draft_distribution_rows(z_k, rows, W, T):
    """softmax((z_k + rows W) / T): the rows serve as the table, row n for
    request n."""
    rows = _f(rows)
    return draft_distribution(z_k, rows, W, np.arange(rows.shape[0]), T)


def _dt(dtype):
    if dtype not in ("bf16", "f32"):
        raise ValueError(f"state type {dtype!r}: bf16 or f32")
    return 0 if dtype == "bf16" else 1


def round_to(x, dtype):
    x = _f(x)
    out = np.empty_like(x)
    _lib().oc_round_state(x.size, _dt(dtype), _p(x), _p(out))
    return out


def rnn_states(E, U, anchor, tokens, dtype):
    E, U, anchor, tokens = _f(E), _f(U), _i(anchor), _i(tokens)
    R, G = tokens.shape
    r = E.shape[1]
    S = np.empty((R, G, r))
    _lib().oc_rnn_states(R, G, r, _dt(dtype), _p(E), _p(U), _p(anchor), _p(tokens), _p(S))
    return S


# --------------------------------------------------------------- stages

def draft_sample(z, E, W, anchor, u_draft, T):
    z, E, W, anchor = _f(z), _f(E), _f(W), _i(anchor)
    R, G, V = z.shape
    u = _f(u_draft) if u_draft is not None else np.zeros((R, G))
    tokens = np.empty((R, G), dtype=np.int64)
    q_lse = np.empty((R, G))
    q_tok = np.empty((R, G))
    _lib().oc_draft_sample(R, G, V, E.shape[1], float(T), _p(z), _p(E), _p(W), _p(anchor), _p(u),
                           _p(tokens), _p(q_lse), _p(q_tok))
    return tokens, q_lse, q_tok


def draft_sample_rnn(z, E, U, W, anchor, u_draft, T, dtype):
    z, E, U, W, anchor = _f(z), _f(E), _f(U), _f(W), _i(anchor)
    R, G, V = z.shape
    r = E.shape[1]
    u = _f(u_draft) if u_draft is not None else np.zeros((R, G))
    tokens = np.empty((R, G), dtype=np.int64)
    q_lse = np.empty((R, G))
    q_tok = np.empty((R, G))
    S = np.empty((R, G, r))
    _lib().oc_draft_sample_rnn(R, G, V, r, _dt(dtype), float(T), _p(z), _p(E), _p(U), _p(W),
                               _p(anchor), _p(u), _p(tokens), _p(q_lse), _p(q_tok), _p(S))
    return tokens, q_lse, q_tok, S


def confidence(h, w, E1, anchor, tokens, sts_t, c_in=None):
    if c_in is not None:
        c_in = _f(c_in)
        R, G = c_in.shape
        c, a = np.empty((R, G)), np.empty((R, G))
        _lib().oc_confidence(R, G, 0, 0, None, None, None, None, None, None, _p(c_in), _p(c),
                             _p(a))
        return c, a
    h, w, E1, anchor, tokens, sts = _f(h), _f(w), _f(E1), _i(anchor), _i(tokens), _f(sts_t)
    R, G, d = h.shape
    c, a = np.empty((R, G)), np.empty((R, G))
    _lib().oc_confidence(R, G, d, E1.shape[1], _p(h), _p(w), _p(E1), _p(anchor), _p(tokens),
                         _p(sts), None, _p(c), _p(a))
    return c, a


def schedule(a, sps, early_stop=True, max_B=0):
    a, sps = _f(a), _f(sps)
    R, G = a.shape
    N = R * G
    imax = N if max_B <= 0 else max(0, min(N, max_B - R))
    ell = np.empty(R, dtype=np.int64)
    row_off = np.empty(R + 1, dtype=np.int64)
    B = np.empty(1, dtype=np.int64)
    E = np.empty(1)
    ist = np.empty(1, dtype=np.int64)
    theta = np.empty(imax + 1)
    order = np.empty(N, dtype=np.int64)
    rc = _lib().oc_schedule(R, G, _p(a), _p(sps), sps.shape[0], int(bool(early_stop)),
                            int(max_B), _p(ell), _p(row_off), _p(B), _p(E), _p(ist), _p(theta),
                            _p(order))
    if rc != 0:
        raise ValueError("SPS table shorter than the largest batch considered")
    return dict(ell=ell, row_off=row_off, B=int(B[0]), E=float(E[0]), i_star=int(ist[0]),
                theta=theta, order=order)


def schedule_capacity(a, K):
    a = _f(a)
    R, G = a.shape
    ell = np.empty(R, dtype=np.int64)
    row_off = np.empty(R + 1, dtype=np.int64)
    B = np.empty(1, dtype=np.int64)
    E = np.empty(1)
    ist = np.empty(1, dtype=np.int64)
    _lib().oc_schedule_capacity(R, G, _p(a), int(K), _p(ell), _p(row_off), _p(B), _p(E), _p(ist))
    return dict(ell=ell, row_off=row_off, B=int(B[0]), E=float(E[0]), i_star=int(ist[0]))


def verify(z, E, W, anchor, tokens, T, ell, row_off, target, u_acc, u_fin, states=None):
    z, E, W = _f(z), _f(E), _f(W)
    S = None if states is None else _f(states)
    anchor, tokens, ell, row_off = _i(anchor), _i(tokens), _i(ell), _i(row_off)
    target = _f(target)
    R, G, V = z.shape
    u_acc = _f(u_acc) if u_acc is not None else np.zeros((R, G))
    u_fin = _f(u_fin) if u_fin is not None else np.zeros(R)
    n_rows = target.shape[0]
    n_acc = np.empty(R, dtype=np.int64)
    out = np.empty((R, G + 1), dtype=np.int64)
    p_lse = np.empty(n_rows)
    kind = np.empty(R, dtype=np.int64)
    frow = np.empty(R, dtype=np.int64)
    _lib().oc_verify(R, G, V, E.shape[1], float(T), _p(z), _p(E), _p(W), _p(anchor), _p(tokens),
                     _p(ell), _p(row_off), _p(target), n_rows, _p(u_acc), _p(u_fin), _p(n_acc),
                     _p(out), _p(p_lse), _p(kind), _p(frow), _p(S))
    rows = np.concatenate([row_off[r] + np.arange(ell[r] + 1) for r in range(R)])
    return dict(n_acc=n_acc, out_tokens=out, p_lse={int(x): float(p_lse[x]) for x in rows},
                final_kind=kind, final_row=frow)


def final_weights(z, E, W, anchor, tokens, T, target_row, j, r, rejected, states=None):
    E, W, trow = _f(E), _f(W), _f(target_row)
    srow = None if states is None else _f(states[r, j, :])
    V = trow.shape[0]
    prev = int(anchor[r]) if j == 0 else int(tokens[r, j - 1])
    zrow = _f(z[r, j, :]) if rejected else np.zeros(V)
    w = np.empty(V)
    _lib().oc_final_weights(V, E.shape[1], float(T), _p(zrow), _p(E), _p(W), prev, _p(trow),
                            int(bool(rejected)), _p(w), _p(srow))
    return w
