"""GPU parity of the RNN sequential head (dspark_draft_sample_rnn,
dspark_verify_rnn) against the CPU oracle through the C ABI: the states
S[n][k] bit for bit (they are quantised in the same fixed fp32 / double
steps on both sides), tokens and acceptance counts bit for bit up to counted
near-ties, q_lse / q_tok / p_lse within 1e-5 relative.

Cases: the fp32 CUDA-core path (tiny shapes, a ragged last tile), the bf16
tensor-core path at T = 1, 0.7 and 0 (greedy), a rank above the tensor-core
limit, more states than vocabulary entries (the final draw's bias rows are
rows of S, R * gamma of them, not token ids), and the full Qwen3-4B and
DeepSeek-scale shapes on sampled requests."""

import numpy as np
import pytest

import conftest
from draft_sampling_lossless_gb300 import synth
from parity import Case, Stats

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

CASES = {
    "tiny": W["tiny"],
    "tiny_ragged_f32": W["tiny"].scaled(name="tiny_ragged_f32", R=3, gamma=3, V=1500, r=8, d=16),
    "mid_bf16": W["qwen3_4b"].scaled(name="mid_bf16", R=8, gamma=5, V=3000, r=64, d=128,
                                     n_sps=0),
    "mid_t07": W["deepseek"].scaled(name="mid_t07", R=6, gamma=6, V=2504, r=32, d=96),
    "mid_greedy": W["greedy"].scaled(name="mid_greedy", R=8, gamma=5, V=3000, r=64, d=128),
    "big_rank_bf16": W["qwen3_4b"].scaled(name="big_rank_bf16", R=5, gamma=3, V=2000, r=320,
                                          d=24, n_sps=0),
    # R * gamma = 2200 states for a vocabulary of 512 tokens
    "many_states": W["qwen3_4b"].scaled(name="many_states", R=1100, gamma=2, V=512, r=16, d=8,
                                        n_sps=0),
    "rows_100": W["qwen3_4b"].scaled(name="rows_100", R=100, gamma=3, V=4000, r=128, d=32,
                                     n_sps=0),
}


def _run(wl, seed=None, sample=None):
    st = Stats()
    c = Case(wl, seed=seed, sample=sample, head="rnn", gen_device="cuda" if wl.R >= 64 else "cpu")
    c.draft(st)
    G = wl.gamma
    ell_s = np.arange(len(c.sample)) % (G + 1)  # every length, ragged
    c.verify(st, ell_s)
    c.verify(st, np.full(len(c.sample), G))  # full blocks: bonus draws
    return st


@pytest.mark.parametrize("name", list(CASES))
def test_rnn_head_matches_oracle(name):
    wl = CASES[name]
    sample = None if wl.R <= 128 else np.array([0, 1, 517, wl.R - 1])
    st = _run(wl, sample=sample)
    assert st.unexplained == [], st.unexplained
    assert st.near_ties <= max(1, int(1e-4 * st.decisions)), (st.near_ties, st.decisions)


@pytest.mark.parametrize("seed", [21, 22])
def test_rnn_head_more_seeds(seed):
    st = _run(CASES["mid_bf16"], seed=seed)
    assert st.unexplained == [], st.unexplained


@pytest.mark.parametrize("name", ["qwen3_4b", "deepseek"])
def test_rnn_head_full_size_sampled(name):
    wl = W[name]
    st = Stats()
    for seed in (None, 5):
        st.merge(_run(wl, seed=seed, sample=np.array([0, 1, wl.R // 2, wl.R - 1])))
    assert st.unexplained == [], st.unexplained
    conftest.SUMMARY.append(f"RNN head full-size parity {name}: decisions={st.decisions} "
                            f"near_ties={st.near_ties} worst_rel="
                            f"{ {k: f'{v:.2e}' for k, v in st.worst_rel.items()} }")
