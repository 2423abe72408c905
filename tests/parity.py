"""Parity harness: runs the CUDA library (through the C ABI) and the CPU oracle
on the same seeded inputs, stage by stage, and compares them under the
comparison rules of the method's target:

* token ids, l_r, B, n_acc: bit-exact, except near-ties -- a sampled token
  whose separating oracle CDF boundary lies within 1e-6 (normalised) of
  u * total, an acceptance test with |u - p/q| < 1e-6, or a greedy choice whose
  top-2 gap is below 1e-6 * max|y|.  Near-ties are counted; any other
  mismatch is "unexplained".
* q_lse, q_tok, p_lse, c, a: within 1e-5 relative.

The GPU stages downstream of a stage are fed the ORACLE's outputs of that
stage, so no oracle input ever comes from the CUDA path.  After a near-tie in
a request's draft the rest of that request's draft positions are conditioned
on different prefixes and are not compared.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

from oracle import native as oracle  # the plain C++ CPU oracle
from draft_sampling_lossless_gb300 import synth, target_model
from draft_sampling_lossless_gb300.pipeline import DSparkStep

REL = 1e-5
TIE = 1e-6


@dataclass
class Stats:
    decisions: int = 0
    near_ties: int = 0
    unexplained: list = field(default_factory=list)
    value_checks: int = 0
    worst_rel: dict = field(default_factory=dict)
    tie_kinds: dict = field(default_factory=dict)  # near-ties by decision kind
    tie_details: list = field(default_factory=list)  # (kind, details) of each near-tie

    def tie(self, kind, detail=None):
        self.near_ties += 1
        self.tie_kinds[kind] = self.tie_kinds.get(kind, 0) + 1
        if detail is not None:
            self.tie_details.append((kind, detail))

    def rel(self, name, got, want, tol=REL):
        got = np.asarray(got, dtype=np.float64)
        want = np.asarray(want, dtype=np.float64)
        err = np.abs(got - want) / np.maximum(np.abs(want), 1e-300)
        err = np.where((got == want), 0.0, err)
        w = float(np.max(err)) if err.size else 0.0
        self.worst_rel[name] = max(self.worst_rel.get(name, 0.0), w)
        self.value_checks += err.size
        assert w <= tol, f"{name}: worst relative error {w:.3e} > {tol:.0e}"

    def merge(self, o: "Stats"):
        self.decisions += o.decisions
        self.near_ties += o.near_ties
        self.unexplained += o.unexplained
        self.tie_details += o.tie_details
        self.value_checks += o.value_checks
        for k, v in o.tie_kinds.items():
            self.tie_kinds[k] = self.tie_kinds.get(k, 0) + v
        for k, v in o.worst_rel.items():
            self.worst_rel[k] = max(self.worst_rel.get(k, 0.0), v)


def cdf_near_tie(w: np.ndarray, u: float, g: int, o: int) -> bool:
    C = np.cumsum(w)
    S = C[-1]
    thr = u * S
    lo, hi = min(g, o), max(g, o)
    return abs(C[lo] - thr) <= TIE * S and abs(C[hi - 1] - thr) <= TIE * S


def cdf_tie_detail(w: np.ndarray, u: float, g: int, o: int) -> dict:
    """Where a differing draw sits: the normalised distance of u from the
    oracle's boundaries between the two tokens, their probabilities."""
    C = np.cumsum(w)
    S = C[-1]
    lo, hi = min(g, o), max(g, o)
    return dict(gpu=g, oracle=o, d_lo=float((C[lo] - u * S) / S),
                d_hi=float((C[hi - 1] - u * S) / S), p_gpu=float(w[g] / S),
                p_oracle=float(w[o] / S), u=float(u))


def argmax_near_tie(y: np.ndarray, g: int, o: int) -> bool:
    return abs(y[g] - y[o]) <= TIE * max(float(np.max(np.abs(y))), 1e-30)


class Case:
    """Inputs of one workload on both sides (float64 numpy for the oracle,
    torch on the GPU for the library)."""

    def __init__(self, wl: synth.Workload, seed=None, gen_device="cpu", sample=None,
                 head="markov"):
        self.wl = wl
        self.head = head
        self.inp = synth.make_inputs(wl, device=gen_device, seed=seed)
        self.seed = seed
        R = wl.R
        self.sample = np.arange(R) if sample is None else np.asarray(sample)
        s = torch.as_tensor(self.sample, dtype=torch.long, device=self.inp.z.device)
        f = synth.to_f64
        self.z64 = f(self.inp.z[s])
        self.E64 = f(self.inp.E)
        self.W64 = f(self.inp.W)
        self.anchor = self.inp.anchor[s].cpu().numpy().astype(np.int64)
        self.u_draft = f(self.inp.u_draft[s])
        self.u_acc = f(self.inp.u_acc[s])
        self.u_fin = f(self.inp.u_fin[s])
        self.h64 = f(self.inp.h[s]) if self.inp.h is not None else None
        self.w64 = f(self.inp.w_conf)
        self.sts64 = f(self.inp.sts_t)
        self.c_in64 = f(self.inp.c_in[s]) if self.inp.c_in is not None else None
        self.sps64 = f(self.inp.sps)
        d = "cuda"
        self.g = dict(z=self.inp.z.to(d), E=self.inp.E.to(d), Wt=self.inp.Wt().to(d),
                      anchor=self.inp.anchor.to(d), u_draft=self.inp.u_draft.to(d),
                      u_acc=self.inp.u_acc.to(d), u_fin=self.inp.u_fin.to(d),
                      h=None if self.inp.h is None else self.inp.h.to(d),
                      w=None if self.inp.w_conf is None else self.inp.w_conf.to(d),
                      sts=self.inp.sts_t.to(d),
                      c_in=None if self.inp.c_in is None else self.inp.c_in.to(d),
                      sps=self.inp.sps.to(d))
        self.S_o = None
        if head == "rnn":
            U = synth.rnn_recurrence(wl, device=gen_device, seed=seed)
            self.U64 = f(U)
            self.g["U"] = U.to(d)
        wlr = wl
        self.step = DSparkStep(wlr.R, wlr.gamma, wlr.V, wlr.r, wlr.n_sps_eff)

    # ------------------------------------------------------------ draft
    def draft(self, st: Stats):
        wl, g = self.wl, self.g
        rnn = self.head == "rnn"
        if rnn:
            self.step.draft_rnn(g["z"], g["E"], g["U"], g["Wt"], g["anchor"], g["u_draft"], wl.T)
        else:
            self.step.draft(g["z"], g["E"], g["Wt"], g["anchor"], g["u_draft"], wl.T)
        torch.cuda.synchronize()
        assert self.step.status() == 0, f"device status {self.step.status():#x}"
        tok_g = self.step.tokens.cpu().numpy()[self.sample]
        qlse_g = self.step.q_lse.cpu().numpy()[self.sample]
        qtok_g = self.step.q_tok.cpu().numpy()[self.sample]
        if rnn:
            S_g = synth.to_f64(self.step.S)[self.sample]
            tok_o, qlse_o, qtok_o, S_o = oracle.draft_sample_rnn(
                self.z64, self.E64, self.U64, self.W64, self.anchor, self.u_draft, wl.T, wl.dtype)
            self.S_o = S_o
        else:
            tok_o, qlse_o, qtok_o = oracle.draft_sample(self.z64, self.E64, self.W64,
                                                        self.anchor, self.u_draft, wl.T)
        self.tok_o, self.qlse_o, self.qtok_o = tok_o, qlse_o, qtok_o
        n_s, G = tok_o.shape
        for i in range(n_s):
            prev = self.anchor[i]
            for k in range(G):
                st.decisions += 1
                if rnn:  # the state that drafts position k: bit for bit (by value)
                    assert np.array_equal(S_g[i, k], S_o[i, k]), (
                        f"state of request {self.sample[i]} position {k} differs in "
                        f"{int(np.sum(S_g[i, k] != S_o[i, k]))} entries")
                st.rel("q_lse", qlse_g[i, k], qlse_o[i, k])
                if tok_g[i, k] == tok_o[i, k]:
                    st.rel("q_tok", qtok_g[i, k], qtok_o[i, k])
                    prev = tok_o[i, k]
                    continue
                if rnn:
                    y = self.z64[i, k] + S_o[i, k] @ self.W64
                else:
                    y = self.z64[i, k] + oracle.markov_bias(self.E64, self.W64,
                                                            np.array([prev]))[0]
                if wl.T == 0.0:
                    tie = argmax_near_tie(y, int(tok_g[i, k]), int(tok_o[i, k]))
                else:
                    yy = y / wl.T
                    tie = cdf_near_tie(np.exp(yy - yy.max()), self.u_draft[i, k],
                                       int(tok_g[i, k]), int(tok_o[i, k]))
                if tie:
                    st.tie("draft", None if wl.T == 0.0 else dict(
                        k=k, **cdf_tie_detail(np.exp(yy - yy.max()), self.u_draft[i, k],
                                              int(tok_g[i, k]), int(tok_o[i, k]))))
                else:
                    st.unexplained.append(("draft", int(self.sample[i]), k, int(tok_g[i, k]),
                                           int(tok_o[i, k])))
                break  # later positions condition on different prefixes

    def oracle_tokens_full(self):
        """Oracle tokens scattered into a full [R, gamma] array (other
        requests: deterministic placeholders, never compared)."""
        R, G = self.wl.R, self.wl.gamma
        full = np.zeros((R, G), dtype=np.int64)
        full[:] = (np.arange(R)[:, None] * 7919 + np.arange(G)[None, :] * 104729) % self.wl.V
        full[self.sample] = self.tok_o
        return full

    # ------------------------------------------------------------ confidence
    def confidence(self, st: Stats):
        wl, g = self.wl, self.g
        tok_full = torch.from_numpy(self.oracle_tokens_full()).to(torch.int32).cuda()
        self.step.confidence(g["h"], g["w"], g["E"], g["anchor"], g["sts"], c_in=g["c_in"],
                             tokens=tok_full)
        torch.cuda.synchronize()
        assert self.step.status() == 0
        c_g = self.step.c.cpu().numpy()[self.sample]
        a_g = self.step.a.cpu().numpy()[self.sample]
        c_o, a_o = oracle.confidence(self.h64, self.w64, self.E64, self.anchor, self.tok_o,
                                     self.sts64, c_in=self.c_in64)
        st.rel("c", c_g, c_o)
        st.rel("a", a_g, a_o)
        assert np.all(np.diff(a_g, axis=1) <= 0), "survival increased"
        self.a_o = a_o

    # ------------------------------------------------------------ schedule
    def schedule(self, st: Stats, a32: np.ndarray, early_stop=True, max_B=0):
        """Both sides on the same fp32 survival values."""
        a_t = torch.from_numpy(a32.astype(np.float32)).cuda()
        self.step.schedule(self.g["sps"], early_stop, max_B, a=a_t)
        torch.cuda.synchronize()
        assert self.step.status() == 0
        o = oracle.schedule(a32.astype(np.float32).astype(np.float64), self.sps64,
                            early_stop=early_stop, max_B=max_B)
        ell_g = self.step.ell.cpu().numpy()
        ro_g = self.step.row_off.cpu().numpy()
        st.decisions += 1
        assert np.array_equal(ell_g, o["ell"]), "l_r differs"
        assert np.array_equal(ro_g, o["row_off"]), "row_off differs"
        assert int(self.step.B.item()) == o["B"]
        assert float(self.step.E.item()) == o["E"], (float(self.step.E.item()), o["E"])
        return o

    # ------------------------------------------------------------ verify
    def verify(self, st: Stats, ell_s: np.ndarray):
        """Verification of the sampled requests with l = ell_s (sampled
        requests), the oracle's draft outputs, and a packed target."""
        wl, g = self.wl, self.g
        R, G, V = wl.R, wl.gamma, wl.V
        tok_full = self.oracle_tokens_full()
        S_full = None
        if self.head == "rnn":  # oracle states of the sampled requests, zeros elsewhere
            S_full = np.zeros((R, G, wl.r))
            S_full[self.sample] = self.S_o
            S_full = torch.from_numpy(S_full).to(wl.torch_dtype)
        dense = target_model.target_logits(self.inp, torch.from_numpy(tok_full), seed=self.seed,
                                           states=S_full)
        ell = np.zeros(R, dtype=np.int64)
        ell[self.sample] = ell_s
        row_off = np.concatenate([[0], np.cumsum(1 + ell)])
        rows = np.concatenate([r * (G + 1) + np.arange(ell[r] + 1) for r in range(R)])
        rows_t = torch.from_numpy(rows).to(dense.device)
        packed = dense.reshape(R * (G + 1), V)[rows_t].contiguous()
        qlse = np.zeros((R, G))
        qtok = np.full((R, G), 0.5)
        qlse[self.sample] = self.qlse_o
        qtok[self.sample] = self.qtok_o
        c = lambda x, dt: torch.from_numpy(np.ascontiguousarray(x)).to(dt).cuda()
        self.step.p_lse = torch.zeros((packed.shape[0],), dtype=torch.float64, device="cuda")
        if S_full is not None:
            self.step.verify_rnn(g["z"], g["Wt"], packed.cuda(), g["u_acc"], g["u_fin"], wl.T,
                                 S=S_full.cuda(), tokens=c(tok_full, torch.int32),
                                 q_lse=c(qlse, torch.float64), q_tok=c(qtok, torch.float32),
                                 ell=c(ell, torch.int32), row_off=c(row_off, torch.int32))
        else:
            self.step.verify(g["z"], g["E"], g["Wt"], g["anchor"], packed.cuda(), g["u_acc"],
                             g["u_fin"], wl.T, tokens=c(tok_full, torch.int32),
                             q_lse=c(qlse, torch.float64), q_tok=c(qtok, torch.float32),
                             ell=c(ell, torch.int32), row_off=c(row_off, torch.int32))
        torch.cuda.synchronize()
        assert self.step.status() == 0, f"device status {self.step.status():#x}"
        nacc_g = self.step.n_acc.cpu().numpy()[self.sample]
        out_g = self.step.out_tokens.cpu().numpy()[self.sample]
        plse_g = self.step.p_lse.cpu().numpy()
        # oracle on the sampled requests only
        s_rows = np.concatenate([row_off[r] + np.arange(ell[r] + 1) for r in self.sample])
        tgt64 = synth.to_f64(packed[torch.from_numpy(s_rows).to(packed.device)])
        ro_s = np.concatenate([[0], np.cumsum(1 + ell_s)])
        o = oracle.verify(self.z64, self.E64, self.W64, self.anchor, self.tok_o, wl.T, ell_s,
                          ro_s, tgt64, self.u_acc, self.u_fin, states=self.S_o)
        # p_lse of every verified row
        want = np.array([o["p_lse"][i] for i in range(len(s_rows))])
        st.rel("p_lse", plse_g[s_rows], want)
        for i in range(len(self.sample)):
            na_o, na_g = int(o["n_acc"][i]), int(nacc_g[i])
            st.decisions += min(ell_s[i], na_o + 1) + 1
            if na_o != na_g:
                j = min(na_o, na_g)  # the first differing acceptance test
                tie = self._accept_tie(i, j, ro_s, tgt64)
                if tie:
                    st.tie("accept")
                else:
                    st.unexplained.append(("accept", int(self.sample[i]), j, na_g, na_o))
                continue
            assert np.array_equal(out_g[i, :na_o], o["out_tokens"][i, :na_o])
            assert np.all(out_g[i, na_o + 1:] == -1)
            fg, fo = int(out_g[i, na_o]), int(o["out_tokens"][i, na_o])
            if fg == fo:
                continue
            trow = tgt64[ro_s[i] + na_o]
            if wl.T == 0.0:
                tie = argmax_near_tie(trow, fg, fo)
            else:
                w = oracle.final_weights(self.z64, self.E64, self.W64, self.anchor, self.tok_o,
                                         wl.T, trow, na_o, i, na_o < ell_s[i], states=self.S_o)
                tie = cdf_near_tie(w, self.u_fin[i], fg, fo)
            if tie:
                st.tie("final", None if wl.T == 0.0 else cdf_tie_detail(w, self.u_fin[i], fg, fo))
            else:
                st.unexplained.append(("final", int(self.sample[i]), na_o, fg, fo))
        return o

    def _accept_tie(self, i, j, ro_s, tgt64):
        wl = self.wl
        x = int(self.tok_o[i, j])
        trow = tgt64[ro_s[i] + j]
        if wl.T == 0.0:
            return argmax_near_tie(trow, int(np.argmax(trow)), x)
        y = trow / wl.T
        e, lse = oracle.softmax_rows(y[None, :])
        p_x = float(np.exp(y[x] - lse[0]))
        if self.S_o is not None:
            q = oracle.draft_distribution_rows(self.z64[i:i + 1, j, :], self.S_o[i:i + 1, j, :],
                                               self.W64, wl.T)[0]
        else:
            prev = np.array([self.anchor[i] if j == 0 else self.tok_o[i, j - 1]])
            q = oracle.draft_distribution(self.z64[i:i + 1, j, :], self.E64, self.W64, prev,
                                          wl.T)[0]
        return abs(self.u_acc[i, j] - p_x / q[x]) <= TIE
