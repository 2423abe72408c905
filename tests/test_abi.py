"""The C-ABI library builds for sm_103a, loads, exports every symbol that
include/dspark.h declares, and rejects bad host-visible arguments before
touching the GPU (no compute calls here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_\w+)\s*\(", src)))


def test_header_declares_the_four_stage_calls():
    fns = declared_functions()
    for f in ("dspark_draft_sample", "dspark_confidence", "dspark_schedule", "dspark_verify"):
        assert f in fns


def test_library_exports_every_declared_symbol(lib):
    L = lib.lib()
    for f in declared_functions():
        assert hasattr(L, f), f"{f} not exported"
    assert set(lib.SYMBOLS) == set(declared_functions())


def test_version_and_status_strings(lib):
    assert "sm_103a" in lib.version()
    L = lib.lib()
    assert L.dspark_status_string(0) == b"DSPARK_OK"
    assert L.dspark_status_string(1) == b"DSPARK_ERR_INVALID_ARG"
    assert L.dspark_status_string(99) == b"DSPARK_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    assert lib.workspace_bytes(64, 7, 151936, 256) > 64 * 151936 * 4
    assert lib.workspace_bytes(0, 7, 1024, 16) == 0
    assert lib.workspace_bytes(4, 33, 1024, 16) == 0  # gamma > 32
    assert lib.workspace_bytes(4, 4, 1, 16) == 0
    assert lib.workspace_bytes(4, 4, 1024, 0) == 0


def test_workspace_grows_with_the_batch_and_caps_the_fused_scratch(lib):
    """The fused head and scheduler keep 32 lane partials, a Theta key and a
    prefix per candidate for at most 8192 candidates (larger batches take the
    separate launches): doubling gamma below the cap adds that scratch, above
    it only the per-candidate arrays every path needs."""
    R, V, r = 512, 4096, 64
    w8, w16, w32 = (lib.workspace_bytes(R, g, V, r) for g in (8, 16, 32))
    fused_scratch = 4096 * (32 * 4 + 16)  # the 4096 candidates gamma 8 -> 16 adds
    assert w16 - w8 > fused_scratch
    assert w32 - w16 < fused_scratch  # 8192 -> 16384 candidates: capped


def _null():
    return ctypes.c_void_p(None)


def _fake():
    # a non-null pointer that is never dereferenced: validation fails first
    return ctypes.c_void_p(0x1000)


def _err(L):
    return L.dspark_last_error().decode()


def test_draft_rejects_bad_arguments_without_launching(lib):
    L = lib.lib()
    f, n = _fake(), _null()
    ws_n = 1 << 30
    args = lambda R=4, G=4, V=1024, r=16, T=1.0, z=f, u=f, dt=1, ws=f: (
        R, G, V, r, T, z, f, f, dt, f, u, f, f, f, ws, ws_n, n)
    assert L.dspark_draft_sample(*args(R=0)) == 1
    assert L.dspark_draft_sample(*args(G=33)) == 1
    assert L.dspark_draft_sample(*args(V=1022)) == 1  # f32 needs V % 4 == 0
    assert L.dspark_draft_sample(*args(V=1020, dt=0)) == 1  # bf16 needs V % 8 == 0
    assert L.dspark_draft_sample(*args(dt=7)) == 1
    assert L.dspark_draft_sample(*args(T=-1.0)) == 1
    assert L.dspark_draft_sample(*args(T=float("nan"))) == 1
    assert L.dspark_draft_sample(*args(z=n)) == 1
    assert "z is NULL" in _err(L)
    assert L.dspark_draft_sample(*args(u=n)) == 1  # uniforms needed when T > 0
    assert L.dspark_draft_sample(*args(ws=n)) == 1
    small = list(args())
    small[15] = 1024
    assert L.dspark_draft_sample(*small) == 4  # DSPARK_ERR_WORKSPACE
    unaligned = list(args())
    unaligned[14] = ctypes.c_void_p(0x1010)
    assert L.dspark_draft_sample(*unaligned) == 1


def test_schedule_rejects_short_sps_and_bad_caps(lib):
    L = lib.lib()
    f, n = _fake(), _null()
    R, G = 4, 4
    # imax = R*G = 16: needs n_sps > 20
    assert L.dspark_schedule(R, G, f, f, 20, 1, 0, f, f, f, f, f, 1 << 20, n) == 1
    assert "SPS table" in _err(L)
    assert L.dspark_schedule(R, G, f, f, 100, 1, 3, f, f, f, f, f, 1 << 20, n) == 1  # max_B < R
    assert L.dspark_schedule(R, G, f, f, 100, 1, -1, f, f, f, f, f, 1 << 20, n) == 1
    assert L.dspark_schedule(R, G, n, f, 100, 1, 0, f, f, f, f, f, 1 << 20, n) == 1
    assert L.dspark_schedule(R, G, f, f, 100, 1, 0, f, f, f, f, f, 16, n) == 4


def test_confidence_and_verify_reject_bad_arguments(lib):
    L = lib.lib()
    f, n = _fake(), _null()
    # head path needs hidden states
    assert L.dspark_confidence(4, 4, 64, 16, 1024, n, f, f, 1, f, f, f, n, f, f, f, 1 << 20, n) == 1
    # d = 0 allowed only with c_in; here c_in NULL -> invalid
    assert L.dspark_confidence(4, 4, 0, 16, 1024, f, f, f, 1, f, f, f, n, f, f, f, 1 << 20, n) == 1
    assert L.dspark_verify(4, 4, 1024, 16, 1.0, f, f, f, 1, f, f, f, f, f, f, f, 0, f, f, f, f,
                           n, f, 1 << 30, n) == 1  # n_target_rows = 0
    assert L.dspark_verify(4, 4, 1024, 16, 1.0, f, f, f, 1, f, f, f, f, f, f, f, 20, n, f, f, f,
                           n, f, 1 << 30, n) == 1  # u_acc NULL with T > 0


def test_draft_schedule_rejects_bad_arguments_without_launching(lib):
    """The fused call validates the draft's, the head's and the scheduler's
    arguments before it launches anything (every case below fails one)."""
    L = lib.lib()
    f, n = _fake(), _null()
    ws_n = 1 << 30

    def call(R=4, G=4, V=1024, r=16, T=1.0, dt=0, d=64, hidden=f, c_in=n, n_sps=100,
             max_B=0, sps=f, ws_bytes=ws_n):
        return L.dspark_draft_schedule(R, G, V, r, T, f, f, f, dt, f, f, d, hidden, f, f, f, c_in,
                                       sps, n_sps, 1, max_B, f, f, f, f, f, f, f, f, f, f,
                                       ws_bytes, n)

    assert call(R=0) == 1
    assert call(T=-1.0) == 1
    assert call(hidden=n) == 1  # the head needs hidden states when c_in is NULL
    assert call(d=0) == 1
    assert call(n_sps=20) == 1  # imax = R*G = 16: needs n_sps > 20
    assert "SPS table" in _err(L)
    assert call(max_B=3) == 1  # a cap below R
    assert call(sps=n) == 1
    assert call(ws_bytes=1024) == 4  # DSPARK_ERR_WORKSPACE


def test_wait_check_rejects_bad_arguments_without_launching(lib):
    L = lib.lib()
    f, n = _fake(), _null()
    assert L.dspark_check_wait_timeout(0, f, 1024, n) == 1
    assert L.dspark_check_wait_timeout(1000001, f, 1024, n) == 1
    assert L.dspark_check_wait_timeout(1000, n, 1024, n) == 1
    assert L.dspark_check_wait_timeout(1000, ctypes.c_void_p(0x1010), 1024, n) == 1
    assert L.dspark_check_wait_timeout(1000, f, 128, n) == 4


def test_schedule_async_rejects_bad_arguments_without_launching(lib):
    L = lib.lib()
    f, n = _fake(), _null()
    args = lambda R=4, G=4, a=f, cap=f, ws=f, nb=1 << 20: (R, G, a, cap, f, f, f, f, ws, nb, n)
    assert L.dspark_schedule_async(*args(R=0)) == 1
    assert L.dspark_schedule_async(*args(G=33)) == 1
    assert L.dspark_schedule_async(*args(a=n)) == 1
    assert L.dspark_schedule_async(*args(cap=n)) == 1
    assert "capacity is NULL" in _err(L)
    assert L.dspark_schedule_async(*args(ws=n)) == 1
    assert L.dspark_schedule_async(*args(nb=256)) == 4


def test_rnn_calls_reject_bad_arguments_without_launching(lib):
    L = lib.lib()
    f, n = _fake(), _null()
    ws_n = 1 << 30
    # R, G, V, r, T, z, E, U, Wt, dt, anchor, u, tokens, q_lse, q_tok, S, ws, ws_bytes, stream
    args = lambda U=f, S=f, r=16, T=1.0: (4, 4, 1024, r, T, f, f, U, f, 1, f, f, f, f, f, S, f,
                                           ws_n, n)
    assert L.dspark_draft_sample_rnn(*args(U=n)) == 1
    assert "U is NULL" in _err(L)
    assert L.dspark_draft_sample_rnn(*args(S=n)) == 1
    assert L.dspark_draft_sample_rnn(*args(S=ctypes.c_void_p(0x1008))) == 1  # not 16-byte aligned
    assert L.dspark_draft_sample_rnn(*args(r=2000)) == 1  # rank above 1024
    # verify: R, G, V, r, T, z, S, Wt, dt, tokens, q_lse, q_tok, ell, row_off, target,
    # n_rows, u_acc, u_fin, n_acc, out_tokens, p_lse, ws, ws_bytes, stream
    v = lambda S=f, rows=20, ua=f: (4, 4, 1024, 16, 1.0, f, S, f, 1, f, f, f, f, f, f, rows, ua,
                                    f, f, f, n, f, ws_n, n)
    assert L.dspark_verify_rnn(*v(S=n)) == 1  # the states are needed when T > 0
    assert L.dspark_verify_rnn(*v(S=ctypes.c_void_p(0x1008))) == 1
    assert L.dspark_verify_rnn(*v(rows=0)) == 1
    assert L.dspark_verify_rnn(*v(ua=n)) == 1
