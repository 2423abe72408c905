"""GPU parity of every stage against the CPU oracle on small and mid-size
seeded workloads (several vocabulary tiles, a ragged last tile, ragged verify
batches), through the C ABI.  See parity.py for the comparison rules."""

import numpy as np
import pytest
import torch

from oracle import native as oracle  # the plain C++ CPU oracle
from draft_sampling_lossless_gb300 import synth, target_model
from parity import Case, Stats

W = synth.WORKLOADS

SMALL = {
    "tiny": W["tiny"],
    "tiny_ragged_f32": W["tiny"].scaled(name="tiny_ragged_f32", R=3, gamma=3, V=1500, r=8, d=16),
    "mid_bf16": W["qwen3_4b"].scaled(name="mid_bf16", R=8, gamma=5, V=3000, r=64, d=128,
                                     n_sps=0),
    "mid_t07": W["deepseek"].scaled(name="mid_t07", R=6, gamma=6, V=2504, r=32, d=96),
    "mid_greedy": W["greedy"].scaled(name="mid_greedy", R=8, gamma=5, V=3000, r=64, d=128),
    "stress_small": W["stress"].scaled(name="stress_small", R=64, gamma=16, V=1000, r=32,
                                       n_sps=0),
    "one_request": W["qwen3_4b"].scaled(name="one_request", R=1, gamma=1, V=264, r=16, d=8,
                                        n_sps=0),
    # an odd number of 256-token tiles: with R <= 64 the last tile pair of the
    # tensor-core draft has no second tile
    "odd_tiles": W["qwen3_4b"].scaled(name="odd_tiles", R=40, gamma=3, V=2800, r=64, d=32,
                                      n_sps=0),
    # more than 2048 partials per request: the finish re-reads its segments
    "big_vocab": W["qwen3_4b"].scaled(name="big_vocab", R=3, gamma=2, V=300000, r=64, d=16,
                                      n_sps=0),
    # more than 64 requests on one 128-row tile (the unpaired tensor-core layout)
    "rows_100": W["qwen3_4b"].scaled(name="rows_100", R=100, gamma=3, V=4000, r=128, d=32,
                                     n_sps=0),
    # bf16 with a rank above the tensor-core path's 256: the CUDA-core draft
    # and final draw
    "big_rank_bf16": W["qwen3_4b"].scaled(name="big_rank_bf16", R=5, gamma=3, V=2000, r=320,
                                          d=24, n_sps=0),
    # more requests than the row pass lists in shared memory (plain-load row
    # pass over every (request, position)), several 128-row tiles in the draft
    "many_requests": W["qwen3_4b"].scaled(name="many_requests", R=1100, gamma=2, V=512, r=16,
                                          d=8, n_sps=0),
}

pytestmark = pytest.mark.gpu


def _full(case_name, seed=None):
    st = Stats()
    c = Case(SMALL[case_name], seed=seed)
    c.draft(st)
    c.confidence(st)
    a32 = c.a_o.astype(np.float32)
    o = c.schedule(st, a32, early_stop=True)
    c.schedule(st, a32, early_stop=False)
    c.verify(st, o["ell"])
    return st


@pytest.mark.parametrize("name", list(SMALL))
def test_all_stages_match_oracle(name):
    st = _full(name)
    assert st.unexplained == [], st.unexplained
    assert st.near_ties <= max(1, int(1e-4 * st.decisions)), (st.near_ties, st.decisions)


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_mid_bf16_more_seeds(seed):
    st = _full("mid_bf16", seed=seed)
    assert st.unexplained == [], st.unexplained


def test_extreme_uniforms():
    """u = 0 and u = 1 - 2^-24 for the draft draws and the final draws: the
    ends of the inverse-CDF searches (first partial, tile, group and token
    with mass; the last ones).  Mismatches there can only be near-ties, since
    both ends sit where the tiniest probabilities decide; each must be one."""
    c = Case(SMALL["mid_bf16"], seed=7)
    R, G = c.wl.R, c.wl.gamma
    top = np.float32(1.0 - 2.0 ** -24)
    ud = np.zeros((R, G), dtype=np.float32)
    ud[::2] = top
    ud[:, 1::2] = top - ud[:, 1::2]  # alternate the ends along each row too
    uf = np.where(np.arange(R) % 2 == 0, top, np.float32(0.0)).astype(np.float32)
    c.u_draft = ud.astype(np.float64)
    c.g["u_draft"] = torch.from_numpy(ud).cuda()
    c.u_fin = uf.astype(np.float64)
    c.g["u_fin"] = torch.from_numpy(uf).cuda()
    st = Stats()
    c.draft(st)
    c.confidence(st)
    o = c.schedule(st, c.a_o.astype(np.float32), early_stop=True)
    c.verify(st, o["ell"])
    assert st.unexplained == [], st.unexplained


def test_verify_full_block_and_empty_prefix():
    """l = gamma (bonus row draws) and l = 0 (only the correction / bonus
    draw at position 1) for every request."""
    st = Stats()
    c = Case(SMALL["mid_bf16"])
    c.draft(st)
    G = c.wl.gamma
    for ell in (np.full(c.wl.R, G), np.zeros(c.wl.R, dtype=np.int64),
                np.arange(c.wl.R) % (G + 1)):
        c.verify(st, ell)
    assert st.unexplained == [], st.unexplained


@pytest.mark.parametrize("R,G", [(1, 1), (3, 4), (64, 7), (256, 16), (2048, 16), (37, 32)])
@pytest.mark.parametrize("mode", ["early", "global"])
def test_schedule_random_survival(R, G, mode):
    rng = np.random.default_rng(R * 100 + G)
    wl = W["stress"].scaled(R=R, gamma=G, V=64, r=16, n_sps=0)
    c_in = rng.beta(8, 2, size=(R, G)).astype(np.float32)
    a32 = np.cumprod(c_in.astype(np.float64), axis=1).astype(np.float32)
    # ties across requests: copy some rows
    if R > 2:
        a32[1] = a32[0]
    case = Case.__new__(Case)
    case.wl = wl
    case.sps64 = synth.to_f64(synth.sps_table(wl))
    case.g = dict(sps=synth.sps_table(wl).cuda())
    from draft_sampling_lossless_gb300.pipeline import DSparkStep

    case.step = DSparkStep(R, G, 64, 16)
    st = Stats()
    case.schedule(st, a32, early_stop=(mode == "early"))
    for cap in (R, R + 1, R + (R * G) // 3):
        case.schedule(st, a32, early_stop=(mode == "early"), max_B=cap)


def test_schedule_sawtooth_modes_differ_like_the_oracle():
    wl = W["stress"].scaled(R=4, gamma=4, V=64, r=16, n_sps=0)
    a32 = np.array([[0.9, 0.81, 0.72, 0.6]] * 4, dtype=np.float32)
    sps = np.full(wl.n_sps_eff, 100.0, dtype=np.float32)
    sps[5] = 10.0  # a dip right after the first candidate
    case = Case.__new__(Case)
    case.wl = wl
    case.sps64 = sps.astype(np.float64)
    case.g = dict(sps=torch.from_numpy(sps).cuda())
    from draft_sampling_lossless_gb300.pipeline import DSparkStep

    case.step = DSparkStep(4, 4, 64, 16)
    st = Stats()
    es = case.schedule(st, a32, early_stop=True)
    gl = case.schedule(st, a32, early_stop=False)
    assert es["B"] == 4 and gl["B"] == 20


def test_chained_pipeline_tiny_matches_oracle_chain():
    """The four GPU stages chained on the GPU's own outputs reproduce the
    oracle's chain end to end on the tiny workload (no near-tie occurs on
    these inputs; if one did, the chains would legitimately diverge)."""
    wl = SMALL["tiny"]
    c = Case(wl)
    g = c.g
    s = c.step
    s.draft(g["z"], g["E"], g["Wt"], g["anchor"], g["u_draft"], wl.T)
    s.confidence(g["h"], g["w"], g["E"], g["anchor"], g["sts"])
    s.schedule(g["sps"], True, 0)
    torch.cuda.synchronize()
    Bn = int(s.B.item())
    tok = s.tokens.clone()
    # target built from the GPU's own tokens (a harness input, not an oracle input)
    dense = target_model.target_logits(c.inp, tok.cpu())
    ell = s.ell.cpu().numpy()
    rows = np.concatenate([r * (wl.gamma + 1) + np.arange(ell[r] + 1) for r in range(wl.R)])
    packed = dense.reshape(-1, wl.V)[torch.from_numpy(rows)].contiguous().cuda()
    assert packed.shape[0] == Bn
    s.verify(g["z"], g["E"], g["Wt"], g["anchor"], packed, g["u_acc"], g["u_fin"], wl.T)
    torch.cuda.synchronize()
    assert s.status() == 0
    # oracle chain
    t_o, ql_o, qt_o = oracle.draft_sample(c.z64, c.E64, c.W64, c.anchor, c.u_draft, wl.T)
    assert np.array_equal(t_o, tok.cpu().numpy())
    _, a_o = oracle.confidence(c.h64, c.w64, c.E64, c.anchor, t_o, c.sts64)
    assert np.allclose(s.a.cpu().numpy(), a_o, rtol=1e-5, atol=0)
    sched = oracle.schedule(a_o.astype(np.float32).astype(np.float64), c.sps64, True)
    assert np.array_equal(sched["ell"], ell)
    dense_o = target_model.target_logits(c.inp, torch.from_numpy(t_o))
    tgt = synth.to_f64(dense_o.reshape(-1, wl.V)[torch.from_numpy(rows)])
    o = oracle.verify(c.z64, c.E64, c.W64, c.anchor, t_o, wl.T, sched["ell"], sched["row_off"],
                      tgt, c.u_acc, c.u_fin)
    assert np.array_equal(o["n_acc"], s.n_acc.cpu().numpy())
    assert np.array_equal(o["out_tokens"], s.out_tokens.cpu().numpy())
