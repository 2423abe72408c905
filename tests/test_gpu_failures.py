"""Failure handling on the GPU, in the forms that leave the device usable:
bad data made on the host (a NaN / +inf logit, token ids outside the
vocabulary) must set the matching bit of the workspace's status word and
leave every other request's results unchanged; the library's bounded waits,
run against barriers that nothing completes, must give up, set the timeout
bit and return; and calls from two host threads on one device, each with its
own workspace and stream, must give the single-thread results."""

import threading

import numpy as np
import pytest
import torch

from draft_sampling_lossless_gb300 import binding as B
from draft_sampling_lossless_gb300 import synth, target_model
from draft_sampling_lossless_gb300.pipeline import DSparkStep

pytestmark = pytest.mark.gpu

TOKEN_RANGE, NONFINITE, TIMEOUT = 0x1, 0x2, 0x10

MID = synth.WORKLOADS["qwen3_4b"].scaled(name="mid_bf16", R=8, gamma=5, V=3000, r=64, d=128,
                                         n_sps=0)
MID_F32 = synth.WORKLOADS["tiny"].scaled(name="tiny_f32", R=6, gamma=4, V=1500, r=8, d=16)


def _g(wl, seed=3):
    inp = synth.make_inputs(wl, device="cuda", seed=seed)
    return inp, dict(z=inp.z, E=inp.E, Wt=inp.Wt(), anchor=inp.anchor, ud=inp.u_draft, h=inp.h,
                     w=inp.w_conf, sts=inp.sts_t, c_in=inp.c_in, sps=inp.sps, ua=inp.u_acc,
                     uf=inp.u_fin)


def _draft(wl, g, fused):
    s = DSparkStep(wl.R, wl.gamma, wl.V, wl.r, wl.n_sps_eff)
    if fused:
        s.draft_schedule(g["z"], g["E"], g["Wt"], g["anchor"], g["ud"], wl.T, g["h"], g["w"],
                         g["E"], g["sts"], g["sps"], c_in=g["c_in"])
    else:
        s.draft(g["z"], g["E"], g["Wt"], g["anchor"], g["ud"], wl.T)
    torch.cuda.synchronize()
    return s


def _rows_equal(a, b, rows):
    for name in ("tokens", "q_lse", "q_tok"):
        x, y = getattr(a, name).cpu()[rows], getattr(b, name).cpu()[rows]
        assert torch.equal(x, y), name


@pytest.mark.parametrize("wl", [MID, MID_F32], ids=["bf16_tensor_core", "f32_cuda_core"])
@pytest.mark.parametrize("fused", [False, True], ids=["draft", "draft_schedule"])
def test_nonfinite_logits_are_flagged_and_other_requests_unchanged(wl, fused):
    inp, g = _g(wl)
    clean = _draft(wl, g, fused)
    assert clean.status() == 0
    bad = dict(g)
    bad["z"] = g["z"].clone()
    bad["z"][2, 1, 100] = float("nan")
    bad["z"][5, 3, wl.V - 1] = float("inf")
    s = _draft(wl, bad, fused)
    assert s.status() & NONFINITE, f"{s.status():#x}"
    keep = [n for n in range(wl.R) if n not in (2, 5)]
    _rows_equal(s, clean, keep)
    # the positions before the bad logit are unchanged too
    for n, k in ((2, 1), (5, 3)):
        assert torch.equal(s.tokens[n, :k].cpu(), clean.tokens[n, :k].cpu())
    t = s.tokens.cpu()
    assert bool(((t >= 0) & (t < wl.V)).all())


@pytest.mark.parametrize("fused", [False, True], ids=["draft", "draft_schedule"])
def test_out_of_range_anchor_is_flagged_and_drafts_without_bias(fused):
    """An anchor outside [-1, V) is flagged and treated as -1 (no bias at
    the first position): that request's draft equals a run with anchor -1."""
    wl = MID
    inp, g = _g(wl, seed=5)
    ref = dict(g)
    ref["anchor"] = g["anchor"].clone()
    ref["anchor"][3] = -1
    want = _draft(wl, ref, fused)
    assert want.status() == 0
    bad = dict(g)
    bad["anchor"] = g["anchor"].clone()
    bad["anchor"][3] = wl.V + 7
    s = _draft(wl, bad, fused)
    assert s.status() & TOKEN_RANGE, f"{s.status():#x}"
    _rows_equal(s, want, list(range(wl.R)))


def test_verify_out_of_range_token_is_rejected_and_flagged():
    """A drafted token outside the vocabulary fails its acceptance test (and
    is flagged); every other request verifies as before."""
    wl = MID
    inp, g = _g(wl, seed=8)
    src = _draft(wl, g, True)
    R, G = wl.R, wl.gamma
    ell = torch.full((R,), G, dtype=torch.int32, device="cuda")
    row_off = (torch.arange(R + 1, dtype=torch.int32, device="cuda") * (G + 1)).contiguous()
    target = target_model.target_logits(inp, src.tokens).reshape(-1, wl.V).contiguous()

    def run(tokens):
        s = DSparkStep(R, G, wl.V, wl.r, wl.n_sps_eff, max_rows=target.shape[0])
        s.verify(g["z"], g["E"], g["Wt"], g["anchor"], target, g["ua"], g["uf"], wl.T,
                 tokens=tokens, q_lse=src.q_lse, q_tok=src.q_tok, ell=ell, row_off=row_off)
        torch.cuda.synchronize()
        return s

    clean = run(src.tokens)
    assert clean.status() == 0
    bad_tok = src.tokens.clone()
    bad_tok[1, 0] = wl.V + 3
    s = run(bad_tok)
    assert s.status() & TOKEN_RANGE, f"{s.status():#x}"
    assert int(s.n_acc[1].item()) == 0
    keep = torch.arange(R) != 1
    assert torch.equal(s.n_acc.cpu()[keep], clean.n_acc.cpu()[keep])
    assert torch.equal(s.out_tokens.cpu()[keep], clean.out_tokens.cpu()[keep])
    f = int(s.out_tokens[1, 0].item())
    assert 0 <= f < wl.V and bool((s.out_tokens[1, 1:] == -1).all())


def test_bounded_waits_give_up_and_the_device_stays_usable():
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    B.dspark_check_wait_timeout(2000, ws)  # 2 ms per wait
    t1.record()
    torch.cuda.synchronize()
    assert B.device_status(ws) & TIMEOUT
    res = ws[128:136].view(torch.int32).cpu().tolist()
    assert res == [0, 1], res  # the mbarrier wait failed, the grid wait gave up
    assert int(ws[64:68].view(torch.int32).item()) == 0  # counter put back
    assert t0.elapsed_time(t1) < 1000.0  # both waits ended near their limits
    # the same device runs a normal step afterwards
    inp, g = _g(MID, seed=9)
    s = _draft(MID, g, True)
    assert s.status() == 0
    with pytest.raises(B.DSparkError):
        B.dspark_check_wait_timeout(0, ws)


def test_two_host_threads_on_one_device():
    """Two host threads, each with its own workspace and stream, issue the
    fused call on different inputs at the same time: the results equal the
    single-thread results."""
    wl = MID
    inputs = [_g(wl, seed=40 + i)[1] for i in range(2)]
    want = [_draft(wl, g, True) for g in inputs]
    got = [None, None]
    err = []

    def work(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                out = []
                for _ in range(5):
                    s = DSparkStep(wl.R, wl.gamma, wl.V, wl.r, wl.n_sps_eff)
                    g = inputs[i]
                    s.draft_schedule(g["z"], g["E"], g["Wt"], g["anchor"], g["ud"], wl.T, g["h"],
                                     g["w"], g["E"], g["sts"], g["sps"], c_in=g["c_in"])
                    out.append(s)
            st.synchronize()
            got[i] = out
        except Exception as e:  # reported below
            err.append(e)

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    assert not err, err
    for i in range(2):
        for s in got[i]:
            assert s.status() == 0
            for name in ("tokens", "q_lse", "a", "ell", "B"):
                assert torch.equal(getattr(s, name).cpu(), getattr(want[i], name).cpu()), name


@pytest.mark.skipif(not torch.cuda.is_available() or torch.cuda.device_count() < 2,
                    reason="needs two visible GPUs")
def test_every_visible_device_runs_the_step():
    """Launch set-up is per device: the same call on each visible device in
    turn gives the same results."""
    wl = MID
    ref = None
    for dev in range(torch.cuda.device_count()):
        with torch.cuda.device(dev):
            inp = synth.make_inputs(wl, device=f"cuda:{dev}", seed=3)
            s = DSparkStep(wl.R, wl.gamma, wl.V, wl.r, wl.n_sps_eff, device=f"cuda:{dev}")
            s.draft_schedule(inp.z, inp.E, inp.Wt(), inp.anchor, inp.u_draft, wl.T, inp.h,
                             inp.w_conf, inp.E, inp.sts_t, inp.sps)
            torch.cuda.synchronize(dev)
            assert s.status() == 0
            t = s.tokens.cpu()
            ref = t if ref is None else ref
            assert torch.equal(t, ref)
