"""The two CPU oracles -- the numpy restatement and the plain C++ one -- agree
on every stage on seeded mid-size workloads: token ids, lengths, batch sizes
and acceptance counts exactly, real values to 1e-12 relative (they sum in
different orders only inside the bias matmul and the confidence dot
products)."""

import numpy as np
import pytest
import torch

import oracle.dspark_oracle as npo
from draft_sampling_lossless_gb300 import synth, target_model
from oracle import native as cpo

W = synth.WORKLOADS

CASES = {
    "tiny": W["tiny"],
    "mid_bf16": W["qwen3_4b"].scaled(name="mid_bf16", R=6, gamma=5, V=3000, r=32, d=48, n_sps=0),
    "mid_t07": W["deepseek"].scaled(name="mid_t07", R=5, gamma=6, V=2504, r=16, d=40),
    "mid_greedy": W["greedy"].scaled(name="mid_greedy", R=6, gamma=4, V=2000, r=16, d=24),
    "stress_small": W["stress"].scaled(name="stress_small", R=48, gamma=16, V=512, r=16, n_sps=0),
}


def close(a, b, tol=1e-12):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    assert np.all(np.abs(a - b) <= tol * np.maximum(np.abs(b), 1e-300)), np.max(np.abs(a - b))


@pytest.mark.parametrize("name", sorted(CASES))
def test_numpy_and_cpp_oracles_agree(name):
    cpo.build()
    wl = CASES[name]
    inp = synth.make_inputs(wl)
    f = synth.to_f64
    z, E, Wm = f(inp.z), f(inp.E), f(inp.W)
    anchor = inp.anchor.numpy().astype(np.int64)
    out = {}
    for tag, o in (("np", npo), ("cpp", cpo)):
        tok, ql, qt = o.draft_sample(z, E, Wm, anchor, f(inp.u_draft), wl.T)
        c, a = o.confidence(f(inp.h), f(inp.w_conf), E, anchor, tok, f(inp.sts_t),
                            c_in=f(inp.c_in))
        a32 = a.astype(np.float32).astype(np.float64)
        sch = o.schedule(a32, f(inp.sps), early_stop=True)
        glob = o.schedule(a32, f(inp.sps), early_stop=False)
        cap = o.schedule_capacity(a32, glob["B"] - 1)
        dense = target_model.target_logits(inp, torch.from_numpy(tok))
        G = wl.gamma
        ell = np.arange(wl.R) % (G + 1)  # every length, ragged
        row_off = np.concatenate([[0], np.cumsum(1 + ell)])
        rows = np.concatenate([r * (G + 1) + np.arange(ell[r] + 1) for r in range(wl.R)])
        tgt = f(dense.reshape(-1, wl.V)[torch.from_numpy(rows)])
        ver = o.verify(z, E, Wm, anchor, tok, wl.T, ell, row_off, tgt, f(inp.u_acc), f(inp.u_fin))
        out[tag] = (tok, ql, qt, c, a, sch, glob, cap, ver)
    (t1, ql1, qt1, c1, a1, s1, g1, k1, v1), (t2, ql2, qt2, c2, a2, s2, g2, k2, v2) = \
        out["np"], out["cpp"]
    assert np.array_equal(t1, t2)
    close(ql1, ql2)
    close(qt1, qt2)
    close(c1, c2, 1e-13)
    close(a1, a2, 1e-13)
    for x, y in ((s1, s2), (g1, g2), (k1, k2)):
        assert np.array_equal(x["ell"], y["ell"]) and np.array_equal(x["row_off"], y["row_off"])
        assert x["B"] == y["B"] and x["E"] == y["E"] and x["i_star"] == y["i_star"]
    assert np.array_equal(s1["theta"], s2["theta"])
    assert np.array_equal(v1["n_acc"], v2["n_acc"])
    assert np.array_equal(v1["out_tokens"], v2["out_tokens"])
    assert np.array_equal(v1["final_kind"], v2["final_kind"])
    assert v1["p_lse"].keys() == v2["p_lse"].keys()
    close([v1["p_lse"][k] for k in v1["p_lse"]], [v2["p_lse"][k] for k in v1["p_lse"]])


def test_cpp_oracle_threads_give_identical_results():
    """OpenMP splits independent requests only: 1 thread and all threads give
    the same bits."""
    cpo.build()
    wl = CASES["mid_t07"]
    inp = synth.make_inputs(wl, seed=77)
    f = synth.to_f64
    args = (f(inp.z), f(inp.E), f(inp.W), inp.anchor.numpy().astype(np.int64), f(inp.u_draft),
            wl.T)
    n0 = cpo.threads()
    try:
        cpo.set_threads(1)
        one = cpo.draft_sample(*args)
        cpo.set_threads(max(2, n0))
        many = cpo.draft_sample(*args)
    finally:
        cpo.set_threads(n0)
    for x, y in zip(one, many):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("name", ["tiny", "mid_bf16", "mid_t07", "mid_greedy"])
def test_numpy_and_cpp_oracles_agree_on_the_rnn_head(name):
    """RNN head: tokens and states exactly (the state is quantised in the same
    fp32 / float64 steps on both sides), q to 1e-12, and verification with the
    states as the draft's bias rows."""
    cpo.build()
    wl = CASES[name]
    inp = synth.make_inputs(wl)
    f = synth.to_f64
    z, E, Wm = f(inp.z), f(inp.E), f(inp.W)
    U = f(synth.rnn_recurrence(wl))
    anchor = inp.anchor.numpy().astype(np.int64)
    out = {}
    for tag, o in (("np", npo), ("cpp", cpo)):
        tok, ql, qt, S = o.draft_sample_rnn(z, E, U, Wm, anchor, f(inp.u_draft), wl.T, wl.dtype)
        S2 = o.rnn_states(E, U, anchor, tok, wl.dtype)
        dense = target_logits_for(inp, tok, S)
        G = wl.gamma
        ell = np.arange(wl.R) % (G + 1)
        row_off = np.concatenate([[0], np.cumsum(1 + ell)])
        rows = np.concatenate([dense[n, : ell[n] + 1] for n in range(wl.R)])
        ver = o.verify(z, E, Wm, anchor, tok, wl.T, ell, row_off, rows, f(inp.u_acc),
                       f(inp.u_fin), states=S)
        out[tag] = (tok, ql, qt, S, S2, ver)
    a, b = out["np"], out["cpp"]
    assert np.array_equal(a[0], b[0])
    close(a[1], b[1])
    close(a[2], b[2])
    assert np.array_equal(a[3], b[3]) and np.array_equal(a[3], a[4]) and np.array_equal(b[3], b[4])
    for k in ("n_acc", "out_tokens", "final_kind", "final_row"):
        assert np.array_equal(a[5][k], b[5][k]), k


def target_logits_for(inp, tok, S):
    return target_model.target_logits(inp, torch.from_numpy(tok),
                                      states=torch.from_numpy(S)).double().numpy()
