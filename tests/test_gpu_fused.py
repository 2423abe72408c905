"""dspark_draft_schedule (draft + confidence head + scheduler in one call)
against the three separate calls on the same inputs: every output must be
bit-identical.  The separate calls are each held to the oracle by
test_gpu_parity.py, so this carries their parity over to the fused call.
Covers the fused persistent launch (bf16 tensor-core draft with the head's
one-pass form, or given confidences) and the shapes that fall back to three
launches (fp32, a Markov rank above 256, more than 8192 candidates, a hidden
size above 4096)."""

import numpy as np
import pytest
import torch

from draft_sampling_lossless_gb300 import synth, target_model
from draft_sampling_lossless_gb300.pipeline import DSparkStep

from test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

CASES = {
    **{k: SMALL[k] for k in ("tiny", "tiny_ragged_f32", "mid_bf16", "mid_t07", "mid_greedy",
                             "stress_small", "one_request", "odd_tiles", "rows_100",
                             "big_rank_bf16", "many_requests")},
    # the bench's shape, smaller vocabulary
    "qwen_shape": W["qwen3_4b"].scaled(name="qwen_shape", V=20000, n_sps=0),
    # more candidates than the fused launch takes (R * gamma > 8192): three launches
    "many_candidates": W["stress"].scaled(name="many_candidates", R=520, gamma=16, V=512, r=16,
                                          n_sps=0),
    # a hidden size past the fused head (d > 4096): three launches, the
    # confidence kernel's one-pass form with a second batch of h loads
    "wide_hidden": W["qwen3_4b"].scaled(name="wide_hidden", R=4, gamma=3, V=1024, r=64, d=4104,
                                        n_sps=0),
    # past the one-pass form (d > 8192): three launches, the general dot products
    "wider_hidden": W["qwen3_4b"].scaled(name="wider_hidden", R=4, gamma=3, V=1024, r=64,
                                         d=8200, n_sps=0),
}

OUTPUTS = ("tokens", "q_lse", "q_tok", "c", "a", "ell", "row_off", "B", "E")


def _inputs(wl, seed=None):
    inp = synth.make_inputs(wl, device="cuda", seed=seed)
    g = dict(z=inp.z, E=inp.E, Wt=inp.Wt(), anchor=inp.anchor, ud=inp.u_draft, h=inp.h,
             w=inp.w_conf, sts=inp.sts_t, c_in=inp.c_in, sps=inp.sps)
    return g


def _separate(wl, g, early_stop, max_B):
    s = DSparkStep(wl.R, wl.gamma, wl.V, wl.r, wl.n_sps_eff)
    s.draft(g["z"], g["E"], g["Wt"], g["anchor"], g["ud"], wl.T)
    s.confidence(g["h"], g["w"], g["E"], g["anchor"], g["sts"], c_in=g["c_in"])
    s.schedule(g["sps"], early_stop, max_B)
    torch.cuda.synchronize()
    assert s.status() == 0, f"device status {s.status():#x}"
    return s


def _fused(wl, g, early_stop, max_B):
    s = DSparkStep(wl.R, wl.gamma, wl.V, wl.r, wl.n_sps_eff)
    s.draft_schedule(g["z"], g["E"], g["Wt"], g["anchor"], g["ud"], wl.T, g["h"], g["w"],
                     g["E"], g["sts"], g["sps"], c_in=g["c_in"], early_stop=early_stop,
                     max_B=max_B)
    torch.cuda.synchronize()
    assert s.status() == 0, f"device status {s.status():#x}"
    return s


def _same(a: DSparkStep, b: DSparkStep):
    for name in OUTPUTS:
        x, y = getattr(a, name).cpu(), getattr(b, name).cpu()
        assert torch.equal(x.view(torch.uint8) if x.dtype.is_floating_point else x,
                           y.view(torch.uint8) if y.dtype.is_floating_point else y), name


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("early_stop", [True, False])
def test_fused_equals_separate_calls(name, early_stop):
    wl = CASES[name]
    g = _inputs(wl)
    _same(_separate(wl, g, early_stop, 0), _fused(wl, g, early_stop, 0))


def test_fused_with_batch_cap():
    wl = CASES["mid_bf16"]
    g = _inputs(wl, seed=5)
    cap = wl.R + 7
    a, b = _separate(wl, g, True, cap), _fused(wl, g, True, cap)
    _same(a, b)
    assert int(b.B.item()) <= cap


def test_fused_full_size_workload():
    """The bench's workload (Qwen3-4B shape) at full size."""
    wl = W["qwen3_4b"]
    g = _inputs(wl)
    _same(_separate(wl, g, True, 0), _fused(wl, g, True, 0))


def test_fused_repeated_calls_reuse_workspace():
    """Two fused steps on one workspace (the grid-barrier counter and the
    scratch are re-initialised per call)."""
    wl = CASES["mid_t07"]
    g1, g2 = _inputs(wl, seed=11), _inputs(wl, seed=12)
    s = DSparkStep(wl.R, wl.gamma, wl.V, wl.r, wl.n_sps_eff)
    for g in (g1, g2):
        s.draft_schedule(g["z"], g["E"], g["Wt"], g["anchor"], g["ud"], wl.T, g["h"], g["w"],
                         g["E"], g["sts"], g["sps"], c_in=g["c_in"])
    torch.cuda.synchronize()
    assert s.status() == 0
    _same(_separate(wl, g2, True, 0), s)


def _verify_with(wl, g, step_src, ell, row_off, target, ws_step=None):
    """dspark_verify on a fresh (or the given) step with explicit lengths."""
    s = ws_step or DSparkStep(wl.R, wl.gamma, wl.V, wl.r, wl.n_sps_eff, max_rows=target.shape[0])
    s.verify(g["z"], g["E"], g["Wt"], g["anchor"], target, g["ua"], g["uf"], wl.T,
             tokens=step_src.tokens, q_lse=step_src.q_lse, q_tok=step_src.q_tok, ell=ell,
             row_off=row_off)
    torch.cuda.synchronize()
    return s


def test_row_pass_decide_flags_bad_length_and_leaves_counters_zero():
    """A request whose verify length is out of range gets no rows in the row
    pass; its decide still runs (flags the row-range bit, emits -1s, n_acc 0),
    the other requests are unaffected, and the per-request counters the row
    pass uses are back at zero for the next call on the same workspace."""
    wl = CASES["mid_bf16"]
    inp = synth.make_inputs(wl, device="cuda", seed=21)
    g = dict(z=inp.z, E=inp.E, Wt=inp.Wt(), anchor=inp.anchor, ud=inp.u_draft, h=inp.h,
             w=inp.w_conf, sts=inp.sts_t, c_in=inp.c_in, sps=inp.sps, ua=inp.u_acc, uf=inp.u_fin)
    src = _fused(wl, g, True, 0)
    R, G = wl.R, wl.gamma
    ell_ok = src.ell.clone()
    bad = 3
    ell_ok[bad] = 0
    counts = (1 + ell_ok).to(torch.int64)
    row_off = torch.zeros(R + 1, dtype=torch.int32, device="cuda")
    row_off[1:] = torch.cumsum(counts, 0).to(torch.int32)
    dense = target_model.target_logits(inp, src.tokens).reshape(R, G + 1, wl.V)
    rows = torch.cat([r * (G + 1) + torch.arange(int(counts[r]), device="cuda") for r in range(R)])
    target = dense.reshape(-1, wl.V)[rows].contiguous()
    ref = _verify_with(wl, g, src, ell_ok, row_off, target)
    assert ref.status() == 0
    ell_bad = ell_ok.clone()
    ell_bad[bad] = G + 3
    s = _verify_with(wl, g, src, ell_bad, row_off, target)
    assert s.status() & 0x4, f"row-range flag not set: {s.status():#x}"
    out, ref_out = s.out_tokens.cpu(), ref.out_tokens.cpu()
    assert torch.all(out[bad] == -1) and int(s.n_acc[bad].item()) == 0
    keep = torch.arange(R) != bad
    assert torch.equal(out[keep], ref_out[keep])
    assert torch.equal(s.n_acc.cpu()[keep], ref.n_acc.cpu()[keep])
    # the same workspace again, valid lengths: the same results as a fresh one
    s.status(clear=True)
    again = _verify_with(wl, g, src, ell_ok, row_off, target, ws_step=s)
    assert again.status() == 0
    assert torch.equal(again.out_tokens.cpu(), ref_out)
    assert torch.equal(again.n_acc.cpu(), ref.n_acc.cpu())
