"""dspark_schedule_noalloc (the scheduler whose scratch is a static array in
the library, for callers that cannot allocate device memory -- engines that
replay a fixed, pre-reserved memory map, or plugins inside a framework that
owns the device heap) against the workspace scheduler dspark_schedule,
through the C ABI, on two calls in a row.  Collected last on purpose."""

import numpy as np
import pytest
import torch

from draft_sampling_lossless_gb300 import binding as B
from draft_sampling_lossless_gb300 import build, synth

pytestmark = pytest.mark.gpu


def _run(fn, a, sps, early, max_B, **kw):
    R, G = a.shape
    dev = a.device
    ell = torch.full((R,), -7, dtype=torch.int32, device=dev)
    row_off = torch.full((R + 1,), -7, dtype=torch.int32, device=dev)
    Bo = torch.zeros((1,), dtype=torch.int32, device=dev)
    Eo = torch.zeros((1,), dtype=torch.float64, device=dev)
    fn(a, sps, early, max_B, ell, row_off, Bo, Eo, **kw)
    torch.cuda.synchronize()
    return ell.cpu(), row_off.cpu(), int(Bo.item()), float(Eo.item())


def _case(R, G, seed):
    rng = np.random.default_rng(seed)
    a = np.cumprod(rng.beta(8, 2, size=(R, G)), axis=1).astype(np.float32)
    wl = synth.WORKLOADS["stress"].scaled(R=R, gamma=G, n_sps=0)
    return torch.from_numpy(a).cuda(), synth.sps_table(wl).cuda()


def test_noalloc_matches_workspace_scheduler_twice():
    build.ensure_built()
    # the larger problem first, then a smaller one: the second call must not
    # see anything the first left in the shared static scratch
    for (R, G, seed, early, cap) in [(2048, 16, 5, True, 0), (64, 7, 6, False, 300)]:
        a, sps = _case(R, G, seed)
        ws = B.alloc_workspace(R, G, 64, 16)
        want = _run(lambda *x: B.dspark_schedule(*x, ws), a, sps, early, cap)
        status = torch.zeros((1,), dtype=torch.int32, device="cuda")
        got = _run(B.dspark_schedule_noalloc, a, sps, early, cap, dev_status=status)
        assert torch.equal(got[0], want[0]), "l_r differs"
        assert torch.equal(got[1], want[1]), "row_off differs"
        assert got[2] == want[2] and got[3] == want[3]
        assert int(status.item()) == 0


def test_noalloc_rejects_more_candidates_than_its_scratch():
    build.ensure_built()
    a = torch.zeros((2049, 16), dtype=torch.float32, device="cuda")
    sps = torch.ones((40000,), dtype=torch.float32, device="cuda")
    with pytest.raises(B.DSparkError) as ei:
        _run(B.dspark_schedule_noalloc, a, sps, True, 0)
    assert "32768" in str(ei.value)
