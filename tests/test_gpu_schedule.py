"""The cluster radix-sort scheduler and the capacity (asynchronous) scheduler
against the C++ oracle, bit for bit: l_r, row_off, B and E.  Sizes span one
CTA, the cluster boundaries (4096 candidates a CTA) and the largest batch the
library takes (2^20 candidates); survival values with cross-request ties, a
single repeated value (every radix pass but the first is the identity), zeros
and invalid values (NaN, negative, +inf: flagged, counted as 0)."""

import numpy as np
import pytest
import torch

from draft_sampling_lossless_gb300 import synth
from draft_sampling_lossless_gb300.pipeline import DSparkStep
from oracle import native as oracle

pytestmark = pytest.mark.gpu


def _sps(R, G, kind="sawtooth", n=None):
    wl = synth.WORKLOADS["stress"].scaled(R=R, gamma=G, n_sps=n or 0, sps=kind)
    return synth.sps_table(wl)


def _survival(rng, R, G):
    c = rng.beta(8, 2, size=(R, G))
    return np.cumprod(c, axis=1).astype(np.float32)


def _gpu(a32, sps, early, max_B=0, step=None):
    R, G = a32.shape
    s = step or DSparkStep(R, G, 64, 16)
    s.schedule(sps.cuda(), early, max_B, a=torch.from_numpy(a32).cuda())
    torch.cuda.synchronize()
    return s


def _same(s, o):
    assert np.array_equal(s.ell.cpu().numpy(), o["ell"]), "l_r differs"
    assert np.array_equal(s.row_off.cpu().numpy(), o["row_off"]), "row_off differs"
    assert int(s.B.item()) == o["B"]
    assert float(s.E.item()) == o["E"]


@pytest.mark.parametrize("R,G", [(1, 3), (128, 32), (129, 32), (256, 16), (257, 16),
                                 (1000, 33 - 1), (4096, 8), (32768, 32)])
@pytest.mark.parametrize("mode", ["early", "global"])
def test_radix_scheduler_matches_oracle(R, G, mode):
    rng = np.random.default_rng(R * 37 + G)
    a32 = _survival(rng, R, G)
    if R > 3:
        a32[R // 2] = a32[0]  # cross-request ties
        a32[-1, G // 2:] = 0.0
    sps = _sps(R, G)
    early = mode == "early"
    s = _gpu(a32, sps, early)
    assert s.status() == 0
    _same(s, oracle.schedule(a32.astype(np.float64), sps.double().numpy(), early_stop=early))
    cap = R + (R * G) // 5
    s = _gpu(a32, sps, early, max_B=cap, step=s)
    _same(s, oracle.schedule(a32.astype(np.float64), sps.double().numpy(), early_stop=early,
                             max_B=cap))


def test_radix_scheduler_one_repeated_value():
    """Every key equal: passes 1-3 see one digit and are skipped; the order
    is the flat index order."""
    R, G = 3000, 7
    a32 = np.full((R, G), 0.375, dtype=np.float32)
    sps = _sps(R, G, "linear")
    for early in (True, False):
        s = _gpu(a32, sps, early)
        _same(s, oracle.schedule(a32.astype(np.float64), sps.double().numpy(), early_stop=early))
        for cap in (R + 1, R + 4 * G + 3):
            s = _gpu(a32, sps, early, max_B=cap)
            o = oracle.schedule(a32.astype(np.float64), sps.double().numpy(), early_stop=early,
                                max_B=cap)
            _same(s, o)


def test_radix_scheduler_flags_invalid_values_and_counts_them_as_zero():
    R, G = 700, 9
    rng = np.random.default_rng(4)
    a32 = _survival(rng, R, G)
    bad = a32.copy()
    bad[3, 4] = np.nan
    bad[10, 0] = -0.5
    bad[20, 8] = np.inf
    clean = bad.copy()
    clean[3, 4] = clean[10, 0] = clean[20, 8] = 0.0
    sps = _sps(R, G)
    s = _gpu(bad, sps, False)
    assert s.status() & 0x2
    _same(s, oracle.schedule(clean.astype(np.float64), sps.double().numpy(), early_stop=False))


@pytest.mark.parametrize("R,G", [(4, 4), (64, 7), (256, 16), (2048, 16)])
def test_async_capacity_from_two_steps_earlier(R, G):
    """The capacity is the global search's B on the survival values of two
    steps earlier, produced on the device and read there; the current
    candidates fill it in the current order."""
    rng = np.random.default_rng(R + 1000 * G)
    a_old, a_now = _survival(rng, R, G), _survival(rng, R, G)
    sps = _sps(R, G)
    old = _gpu(a_old, sps, False)
    s = DSparkStep(R, G, 64, 16)
    s.schedule_async(old.B, a=torch.from_numpy(a_now).cuda())
    torch.cuda.synchronize()
    assert s.status() == 0
    K = oracle.schedule(a_old.astype(np.float64), sps.double().numpy(), early_stop=False)["B"]
    assert int(old.B.item()) == K
    _same(s, oracle.schedule_capacity(a_now.astype(np.float64), K))


@pytest.mark.parametrize("K", [-5, 0, 3, 4, 5, 17, 20, 21, 1000])
def test_async_capacity_is_clamped(K):
    R, G = 4, 4
    rng = np.random.default_rng(9)
    a32 = _survival(rng, R, G)
    a32[1] = a32[0]
    s = DSparkStep(R, G, 64, 16)
    s.schedule_async(torch.tensor([K], dtype=torch.int32, device="cuda"),
                     a=torch.from_numpy(a32).cuda())
    torch.cuda.synchronize()
    _same(s, oracle.schedule_capacity(a32.astype(np.float64), K))
    assert int(s.B.item()) == min(max(K, R), R * (G + 1))
