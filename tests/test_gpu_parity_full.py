"""GPU parity at the full sizes of the five workloads, in the launch
configuration the benchmark times: the library runs every request, the oracle
recomputes a sample of requests one by one (requests are independent in the
draft, confidence and verify stages); the scheduler is compared on all
candidates."""

import numpy as np
import pytest
import torch

from draft_sampling_lossless_gb300 import synth
from parity import Case, Stats

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


def _sample(R):
    return np.unique(np.array([0, 1, R // 2, R - 1]))


@pytest.mark.parametrize("name", ["tiny", "qwen3_4b", "deepseek", "greedy", "stress"])
def test_full_size_sampled_parity(name):
    wl = W[name]
    st = Stats()
    c = Case(wl, gen_device="cuda", sample=_sample(wl.R))
    c.draft(st)
    c.confidence(st)
    # scheduler on all candidates: survival of the sampled requests from the
    # oracle, the rest from the same seeded Beta draw (any valid survival set)
    rng = np.random.default_rng(wl.seed)
    a_all = np.cumprod(rng.beta(8, 2, size=(wl.R, wl.gamma)), axis=1)
    a_all[c.sample] = c.a_o
    a32 = a_all.astype(np.float32)
    o = c.schedule(st, a32, early_stop=True)
    c.schedule(st, a32, early_stop=False)
    c.verify(st, o["ell"][c.sample])
    # every sampled request also with a full block (bonus draws)
    c.verify(st, np.full(len(c.sample), wl.gamma))
    assert st.unexplained == [], st.unexplained
    print(f"{name}: decisions={st.decisions} near_ties={st.near_ties} "
          f"worst_rel={ {k: f'{v:.2e}' for k, v in st.worst_rel.items()} }")
