"""Benchmark of one DSpark speculative step (draft -> confidence -> schedule
-> verify) on the Qwen3-4B-shaped workload (R=64, gamma=7, V=151936, r=256,
hidden 2560, bf16), through the libdspark C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload tiny|qwen3_4b|deepseek|greedy|stress] [--early-stop 0|1]
                  [--verify-only]

The other workloads are measured with --workload; --early-stop 0 runs the
scheduler's global search; --verify-only times the verification alone on
the scheduler's ragged batch (metric: verified rows/s).

Prints ONE JSON line on rank 0.  `value` is draft+verify positions/s
(R * gamma per step) over the device-timed steps (CUDA events on the launching
stream, one CUDA-graph replay of the whole step per timed iteration, L2
flushed between iterations); `e2e` is the same metric through the public
calls with pinned host buffers copied in and the result copied out inside the
timed region.  Multi-GPU runs are independent replicas (weak scaling; the
path has no data exchange at one scheduler per GPU).  `--impl reference`
times the CPU oracle on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from draft_sampling_lossless_gb300 import synth, target_model  # noqa: E402

METRIC = "draft+verify positions/s"
UNIT = "positions/s"
L2_FLUSH_BYTES = 512 << 20

# Algorithmic bytes per launch of each kernel (what the method must move), as
# functions of the workload and the scheduled batch B.
def algorithmic_bytes(kind, wl, B, n_rej):
    e = 2 if wl.dtype == "bf16" else 4
    R, V, r = wl.R, wl.V, wl.r
    if kind == "verify_rows":
        return B * V * e
    if kind == "rnn_state":  # U once, the E rows and previous states of every request
        return r * r * e + 2 * R * r * e
    if kind in ("draft_partial", "draft_fused_tc"):
        return R * V * e + (r * V * e if kind == "draft_fused_tc" else 0)
    if kind == "draft_persistent_tc":  # all gamma positions; W read once (L2-resident)
        return wl.gamma * R * V * e + r * V * e
    if kind == "markov_bias":
        return r * V * e
    if kind == "final_partial":
        return R * V * e + n_rej * V * e
    if kind == "final_tc":  # target row of every request, z row of each rejection, W once
        return R * V * e + n_rej * V * e + r * V * e
    return None


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self.gpu), "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        except Exception:
            return None
        if not rows:
            return None

        def fnum(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [fnum(r[1]) for r in rows if fnum(r[1]) is not None]
        mx = [fnum(r[2]) for r in rows if fnum(r[2]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for i, nm in enumerate(names):
                if r[5 + i].lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, world: int) -> float:
    """Max over ranks (the slowest replica defines the job time)."""
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: int, seconds_per_step_local: float, world: int):
    """Whole-job throughput: units all ranks processed / max-over-ranks time."""
    t = reduce_max(seconds_per_step_local, world)
    return units_per_rank * world / t, t


# --------------------------------------------------------------------- ours

def run_ours(args, wl, world, rank, local):
    from draft_sampling_lossless_gb300 import binding as Bd
    from draft_sampling_lossless_gb300 import build
    from draft_sampling_lossless_gb300.pipeline import DSparkStep

    build.ensure_built()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    inp = synth.make_inputs(wl, device=dev)
    Wt = inp.Wt()
    g = dict(z=inp.z, E=inp.E, Wt=Wt, anchor=inp.anchor, ud=inp.u_draft, ua=inp.u_acc,
             uf=inp.u_fin, h=inp.h, w=inp.w_conf, sts=inp.sts_t, c_in=inp.c_in, sps=inp.sps)
    step = DSparkStep(wl.R, wl.gamma, wl.V, wl.r, wl.n_sps_eff, device=dev)
    rnn = args.head == "rnn"
    if rnn:
        g["U"] = synth.rnn_recurrence(wl, device=dev)

    def front():
        if rnn:  # RNN head: the draft, then the head and the scheduler
            step.draft_rnn(g["z"], g["E"], g["U"], g["Wt"], g["anchor"], g["ud"], wl.T)
            step.confidence(g["h"], g["w"], g["E"], g["anchor"], g["sts"], c_in=g["c_in"])
            step.schedule(g["sps"], early_stop=bool(args.early_stop))
            return
        # draft + confidence head + scheduler: one call (one launch here)
        step.draft_schedule(g["z"], g["E"], g["Wt"], g["anchor"], g["ud"], wl.T, g["h"], g["w"],
                            g["E"], g["sts"], g["sps"], c_in=g["c_in"],
                            early_stop=bool(args.early_stop))

    # pass 0: the scheduled batch and the target logits the target model would
    # produce for it (a harness input, packed in the scheduler's row order)
    front()
    torch.cuda.synchronize()
    Bn = int(step.B.item())
    ell = step.ell.cpu().numpy()
    dense = target_model.target_logits(inp, step.tokens, states=step.S if rnn else None)
    rows = np.concatenate([r * (wl.gamma + 1) + np.arange(ell[r] + 1) for r in range(wl.R)])
    target = dense.reshape(-1, wl.V)[torch.from_numpy(rows).to(dev)].contiguous()
    del dense
    step.p_lse = torch.zeros((Bn,), dtype=torch.float64, device=dev)

    def verify():
        if rnn:
            step.verify_rnn(g["z"], g["Wt"], target, g["ua"], g["uf"], wl.T)
            return
        step.verify(g["z"], g["E"], g["Wt"], g["anchor"], target, g["ua"], g["uf"], wl.T)

    def full_step():
        front()
        verify()

    # --verify-only times the verification alone on the scheduler's batch
    one_step = verify if args.verify_only else full_step
    full_step()
    torch.cuda.synchronize()
    assert step.status() == 0, f"device status {step.status():#x}"
    assert int(step.B.item()) == Bn
    n_rej = int((step.n_acc < step.ell).sum().item())
    mean_acc = float(step.n_acc.float().mean().item())

    # CUDA graph of the whole step
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            one_step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    c0 = Bd.launch_count()
    with torch.cuda.graph(graph):
        one_step()
    launches_per_step = Bd.launch_count() - c0
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    for _ in range(args.warmup):
        flush.zero_()
        graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.1)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = [a.elapsed_time(b) for a, b in ev]
    ms_local = sum(ms) / len(ms)
    units = Bn if args.verify_only else wl.R * wl.gamma
    value, t_max = aggregate(units, ms_local / 1e3, world)
    assert step.status() == 0, f"device status {step.status():#x}"

    # per-kernel device times: the same step captured with tracing on
    Bd.trace_start()
    tgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(tgraph):
        one_step()
    Bd.trace_stop()
    for i in range(args.steps):
        flush.zero_()
        tgraph.replay()
        torch.cuda.synchronize()
        Bd.trace_collect()
    totals = {k: v for k, v in Bd.trace_totals().items() if v[0] > 0}
    del tgraph

    # end to end through the public calls with pinned host buffers
    e2e = None if args.verify_only or rnn else run_e2e(args, wl, inp, g, step, target, dev, Bd)

    peaks, psrc = read_peaks()
    kernels = {k: {"launches_per_step": v[0] / args.steps, "avg_us": 1e3 * v[1] / v[0],
                   "share": v[1] / sum(x[1] for x in totals.values())}
               for k, v in totals.items()}
    dom = max(totals, key=lambda k: totals[k][1])
    roof = roofline_entry(dom, totals[dom], wl, Bn, n_rej, peaks, psrc)

    out = {
        "metric": "verify rows/s" if args.verify_only else METRIC, "value": value,
        "unit": "rows/s" if args.verify_only else UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": f"{wl.name}: R={wl.R} gamma={wl.gamma} V={wl.V} r={wl.r} "
                               f"d={wl.d} T={wl.T}", "B": Bn, "mean_n_acc": mean_acc,
                   "early_stop": bool(args.early_stop), "head": args.head,
                   "timed": "verification only" if args.verify_only else "the whole step",
                   "l2": "flushed between timed steps (512 MiB write)", "cuda_graph": True,
                   "parallelism": f"replicas x{world}"},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "roofline": roof,
        "kernels": kernels,
    }
    if rank == 0 and world == 1 and not (args.no_cpu_baseline or args.verify_only or rnn):
        out["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_budget)
    return out


def roofline_entry(kind, tot, wl, Bn, n_rej, peaks, psrc):
    launches, ms = tot
    avg_s = ms / launches / 1e3
    nbytes = algorithmic_bytes(kind, wl, Bn, n_rej)
    traffic = recorded_traffic(kind, wl)
    if nbytes is None:
        return {"kernel": kind, "bound": "latency", "achieved": None, "peak": None,
                "unit": "GB/s", "frac": None, "traffic": traffic, "avg_us": avg_s * 1e6}
    ach = nbytes / avg_s / 1e9
    peak = float(peaks["hbm_gbs"])
    return {"kernel": kind, "bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
            "frac": ach / peak, "traffic": traffic, "algorithmic_bytes": nbytes,
            "avg_us": avg_s * 1e6, "peak_source": f"{psrc} hbm_gbs"}


def recorded_traffic(kind, wl):
    """DRAM bytes per launch from the committed ncu summary, valid only while
    the kernel source is unchanged (checked by content hash)."""
    import hashlib

    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    want = {}
    with open(p) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = dict(kv.split("=", 1) for kv in line.split())
            want[(parts.get("kernel"), parts.get("workload"))] = parts
    e = want.get((kind, wl.name))
    if e is None:
        return None
    # the kernel's sources ('+'-separated), hashed in order
    hs = hashlib.sha256()
    for name in e["file"].split("+"):
        src = os.path.join(ROOT, "draft_sampling_lossless_gb300", "csrc", name)
        if not os.path.exists(src):
            return None
        hs.update(open(src, "rb").read())
    if hs.hexdigest()[:16] != e.get("sha"):
        return None
    return float(e["bytes_per_launch"])


def run_e2e(args, wl, inp, g, step, target, dev, Bd):
    """Per step: pinned host -> device copies of the step's inputs (base
    logits, hidden states, anchors, uniforms, target logits), the library
    calls (draft + confidence + schedule in one, then verify), and device ->
    host copies of the result (emitted tokens, n_acc, B)."""
    pin = lambda t: (t.cpu().pin_memory() if t is not None else None)
    host = dict(z=pin(inp.z), h=pin(inp.h), anchor=pin(inp.anchor), ud=pin(inp.u_draft),
                ua=pin(inp.u_acc), uf=pin(inp.u_fin), c_in=pin(inp.c_in), target=pin(target))
    dbuf = {k: (torch.empty_like(v, device=dev) if v is not None else None) for k, v in host.items()}
    out_h = dict(out=torch.empty(step.out_tokens.shape, dtype=torch.int32).pin_memory(),
                 nacc=torch.empty(step.n_acc.shape, dtype=torch.int32).pin_memory(),
                 B=torch.empty((1,), dtype=torch.int32).pin_memory())
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = sum(v.numel() * v.element_size() for v in out_h.values())

    # Two device copies of the inputs: while step j computes from one, step
    # j + 1's inputs stream into the other on a copy stream (the draft's
    # first, then the verification's), so the host link never idles; each
    # step's copy is still inside the timed region, and the host reads each
    # step's result before it enqueues the next step.
    bufs = [dbuf, {k: (torch.empty_like(v) if v is not None else None) for k, v in dbuf.items()}]
    copy_stream = torch.cuda.Stream(device=dev)
    draft_in = ("z", "h", "anchor", "ud", "c_in")
    verify_in = ("target", "ua", "uf")
    ev = lambda: torch.cuda.Event()
    drafted_in, verified_in, computed = [ev(), ev()], [ev(), ev()], [None, None]

    def copies(j):
        b, s = bufs[j % 2], j % 2
        if computed[s] is not None:
            copy_stream.wait_event(computed[s])  # the step that last read this set
        with torch.cuda.stream(copy_stream):
            for k in draft_in:
                if host[k] is not None:
                    b[k].copy_(host[k], non_blocking=True)
            drafted_in[s].record(copy_stream)
            for k in verify_in:
                if host[k] is not None:
                    b[k].copy_(host[k], non_blocking=True)
            verified_in[s].record(copy_stream)

    def compute(j):
        b, s = bufs[j % 2], j % 2
        cur = torch.cuda.current_stream()
        cur.wait_event(drafted_in[s])
        step.draft_schedule(b["z"], g["E"], g["Wt"], b["anchor"], b["ud"], wl.T, b["h"], g["w"],
                            g["E"], g["sts"], g["sps"], c_in=b["c_in"],
                            early_stop=bool(args.early_stop))
        cur.wait_event(verified_in[s])
        step.verify(b["z"], g["E"], g["Wt"], b["anchor"], b["target"], b["ua"], b["uf"], wl.T)
        computed[s] = ev()
        computed[s].record(cur)
        out_h["out"].copy_(step.out_tokens, non_blocking=True)
        out_h["nacc"].copy_(step.n_acc, non_blocking=True)
        out_h["B"].copy_(step.B, non_blocking=True)
        done = ev()
        done.record(cur)
        return done

    def run(n_steps):
        copies(0)
        for j in range(n_steps):
            done = compute(j)
            if j + 1 < n_steps:
                copies(j + 1)
            done.synchronize()  # the host reads step j's result

    run(max(3, args.warmup))
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 50))
    t0 = time.perf_counter()
    run(n)
    t = (time.perf_counter() - t0) / n
    return {"value": wl.R * wl.gamma / t, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": t * 1e3, "steps": n,
            "timing": "host wall clock around copies + calls + result read; each step's inputs "
                      "copied on a copy stream into one of two device buffers while the previous "
                      "step computes; the host reads every step's result"}


# --------------------------------------------------------------------- CPU

def oracle_step(wl, inp, reqs, cache):
    """The plain C++ CPU oracle over a sub-batch of requests (scheduled as its
    own batch): draft, confidence, schedule and verify are timed; the target
    model's stand-in (building the target rows from the oracle's draft) is not.
    Returns the seconds spent in the four stages."""
    from oracle import native as oracle

    f = synth.to_f64
    idx = torch.as_tensor(reqs, dtype=torch.long)
    if "E" not in cache:
        cache["E"], cache["W"] = f(inp.E), f(inp.W)
    E, W = cache["E"], cache["W"]
    z = f(inp.z[idx])
    anchor = inp.anchor[idx].numpy().astype(np.int64)
    t0 = time.perf_counter()
    tok, _, _ = oracle.draft_sample(z, E, W, anchor, f(inp.u_draft[idx]), wl.T)
    c_in = f(inp.c_in[idx]) if inp.c_in is not None else None
    h = f(inp.h[idx]) if inp.h is not None else None
    _, a = oracle.confidence(h, f(inp.w_conf) if inp.w_conf is not None else None, E, anchor,
                             tok, f(inp.sts_t), c_in=c_in)
    sch = oracle.schedule(a.astype(np.float32).astype(np.float64), f(inp.sps), True)
    t1 = time.perf_counter()
    # the target model's forward pass is outside the path: its stand-in builds
    # the sub-batch's target rows for the drafted tokens (not timed)
    sub = synth.Inputs(wl.scaled(R=len(reqs)), inp.z[idx], inp.E, inp.W, inp.anchor[idx],
                       inp.u_draft[idx], inp.u_acc[idx], inp.u_fin[idx], None, None,
                       inp.sts_t, None, inp.sps)
    dense = target_model.target_logits(sub, torch.from_numpy(tok))
    G = wl.gamma
    rows = np.concatenate([r * (G + 1) + np.arange(sch["ell"][r] + 1) for r in range(len(reqs))])
    tgt = f(dense.reshape(-1, wl.V)[torch.from_numpy(rows)])
    t2 = time.perf_counter()
    oracle.verify(z, E, W, anchor, tok, wl.T, sch["ell"], sch["row_off"], tgt,
                  f(inp.u_acc[idx]), f(inp.u_fin[idx]))
    return (t1 - t0) + (time.perf_counter() - t2)


def cpu_inputs(wl):
    return synth.make_inputs(wl, device="cpu")


def _timed_oracle(wl, inp, n_req, threads, budget_s, cache):
    """Sub-batches of n_req consecutive requests through the oracle on
    `threads` OpenMP threads until about budget_s seconds of stage time."""
    from oracle import native as oracle

    n0 = oracle.threads()
    oracle.set_threads(threads)
    try:
        done, spent, k = 0, 0.0, 0
        while spent < budget_s or done == 0:
            reqs = [(k + i) % wl.R for i in range(n_req)]
            spent += oracle_step(wl, inp, reqs, cache)
            done += n_req
            k += n_req
    finally:
        oracle.set_threads(n0)
    return done, spent


def cpu_baseline(wl, budget_s=15.0, inp=None):
    """The plain C++ oracle, as it stands, on the host cores: one thread on
    single requests, and every core (OpenMP over requests) on sub-batches of
    one request per core; bounded to about budget_s seconds in all."""
    inp = inp or cpu_inputs(wl)
    cores = len(os.sched_getaffinity(0))
    n_req = min(cores, wl.R)  # distinct requests, one a core
    cache = {}
    d1, t1 = _timed_oracle(wl, inp, 1, 1, budget_s / 3, cache)
    dn, tn = _timed_oracle(wl, inp, n_req, cores, 2 * budget_s / 3, cache)
    return {"value": dn * wl.gamma / tn, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{dn} requests of {wl.name} in sub-batches of {n_req} (one a core), all "
                      f"four stages of the plain C++ oracle (double), {tn:.1f} s of stage time; "
                      f"the target stand-in untimed",
            "single_thread": {"value": d1 * wl.gamma / t1, "unit": UNIT, "cores": 1,
                              "sample": f"{d1} single requests, {t1:.1f} s"}}


def run_reference(args, wl):
    """The reference arm: the plain C++ CPU oracle (there is no reference
    implementation to install), every host core, each step one sub-batch of
    one request per core."""
    inp = cpu_inputs(wl)
    cores = len(os.sched_getaffinity(0))
    cache = {}
    from oracle import native as oracle

    oracle.set_threads(cores)
    n_req = min(cores, wl.R)  # distinct requests, one a core
    for i in range(args.warmup):
        oracle_step(wl, inp, [(i * n_req + j) % wl.R for j in range(n_req)], cache)
    times = []
    budget = 150.0
    t_all = time.perf_counter()
    for i in range(args.steps):
        times.append(oracle_step(wl, inp, [(i * n_req + j) % wl.R for j in range(n_req)], cache))
        if time.perf_counter() - t_all > budget and len(times) >= 3:
            break
    t = sum(times) / len(times)
    value = n_req * wl.gamma / t
    sample = (f"{len(times)} timed steps, each a sub-batch of {n_req} requests of {wl.name} "
              f"(one a core) through all four stages of the plain C++ oracle")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{wl.name}: R={wl.R} gamma={wl.gamma} V={wl.V} r={wl.r} "
                                   f"d={wl.d} T={wl.T}", "sample_requests_per_step": n_req},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_4b", choices=list(synth.WORKLOADS))
    ap.add_argument("--early-stop", type=int, default=1, choices=[0, 1],
                    help="scheduler stop rule: 1 early stop, 0 global search")
    ap.add_argument("--verify-only", action="store_true",
                    help="time the verification alone on the scheduled batch")
    ap.add_argument("--head", default="markov", choices=["markov", "rnn"],
                    help="sequential head of the draft: the Markov head, or the RNN head "
                         "(state launch + draw per position; no e2e or CPU legs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    wl = synth.WORKLOADS[args.workload]
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, wl)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    out = run_ours(args, wl, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
