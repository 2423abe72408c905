"""One DSpark speculative step on the GPU: output buffers plus the
libdspark calls (the four stages, or draft + confidence + schedule fused
and verify), enqueued on one stream.  Marshalling only -- every stage
runs in the CUDA library."""

from __future__ import annotations

import torch

from . import binding as B


class DSparkStep:
    """Device buffers for a step with R requests, draft length gamma,
    vocabulary V and Markov rank r.  Calls are asynchronous on `stream`."""

    def __init__(self, R, gamma, V, r, n_sps=0, device="cuda", max_rows=None):
        self.R, self.gamma, self.V, self.r = R, gamma, V, r
        dev = torch.device(device)
        i32, f32, f64 = torch.int32, torch.float32, torch.float64
        self.tokens = torch.zeros((R, gamma), dtype=i32, device=dev)
        self.q_lse = torch.zeros((R, gamma), dtype=f64, device=dev)
        self.q_tok = torch.zeros((R, gamma), dtype=f32, device=dev)
        self.c = torch.zeros((R, gamma), dtype=f32, device=dev)
        self.a = torch.zeros((R, gamma), dtype=f32, device=dev)
        self.ell = torch.zeros((R,), dtype=i32, device=dev)
        self.row_off = torch.zeros((R + 1,), dtype=i32, device=dev)
        self.B = torch.zeros((1,), dtype=i32, device=dev)
        self.E = torch.zeros((1,), dtype=f64, device=dev)
        self.n_acc = torch.zeros((R,), dtype=i32, device=dev)
        self.out_tokens = torch.zeros((R, gamma + 1), dtype=i32, device=dev)
        rows = max_rows if max_rows is not None else R * (gamma + 1)
        self.p_lse = torch.zeros((rows,), dtype=f64, device=dev)
        self.ws = B.alloc_workspace(R, gamma, V, r, n_sps, device=dev)
        self.S = None  # RNN head states, allocated by draft_rnn

    def draft(self, z, E, Wt, anchor, u_draft, T, stream=None):
        B.dspark_draft_sample(z, E, Wt, anchor, u_draft, T, self.tokens, self.q_lse, self.q_tok,
                              self.ws, stream)

    def draft_rnn(self, z, E, U, Wt, anchor, u_draft, T, stream=None):
        """The draft with the RNN head; the states land in self.S [R, gamma, r]
        (allocated on first use, in E's dtype)."""
        if self.S is None or self.S.dtype != E.dtype:
            self.S = torch.zeros((self.R, self.gamma, self.r), dtype=E.dtype, device=E.device)
        B.dspark_draft_sample_rnn(z, E, U, Wt, anchor, u_draft, T, self.tokens, self.q_lse,
                                  self.q_tok, self.S, self.ws, stream)

    def verify_rnn(self, z, Wt, target, u_acc, u_fin, T, S=None, tokens=None, q_lse=None,
                   q_tok=None, ell=None, row_off=None, stream=None):
        B.dspark_verify_rnn(z, self.S if S is None else S, Wt,
                            self.tokens if tokens is None else tokens,
                            self.q_lse if q_lse is None else q_lse,
                            self.q_tok if q_tok is None else q_tok,
                            self.ell if ell is None else ell,
                            self.row_off if row_off is None else row_off, target, u_acc, u_fin,
                            T, self.n_acc, self.out_tokens,
                            self.p_lse if self.p_lse.numel() >= target.shape[0] else None,
                            self.ws, stream)

    def confidence(self, hidden, w, E1, anchor, sts_t, c_in=None, tokens=None, stream=None):
        B.dspark_confidence(self.R, self.gamma, hidden, w, E1, anchor,
                            self.tokens if tokens is None else tokens, sts_t, c_in, self.c,
                            self.a, self.ws, stream)

    def schedule(self, sps, early_stop=True, max_B=0, a=None, stream=None):
        B.dspark_schedule(self.a if a is None else a, sps, early_stop, max_B, self.ell,
                          self.row_off, self.B, self.E, self.ws, stream)

    def schedule_async(self, capacity, a=None, stream=None):
        """Capacity (asynchronous) scheduling: the batch holds exactly the
        first capacity - R candidates (clamped); capacity is a one-element
        int32 device tensor, e.g. the B of a global-search schedule of the
        survival values two steps earlier."""
        B.dspark_schedule_async(self.a if a is None else a, capacity, self.ell, self.row_off,
                                self.B, self.E, self.ws, stream)

    def draft_schedule(self, z, E, Wt, anchor, u_draft, T, hidden, w, E1, sts_t, sps,
                       c_in=None, early_stop=True, max_B=0, stream=None):
        """draft + confidence + schedule in one call (one launch when the
        shapes allow it); the same results as the three calls."""
        B.dspark_draft_schedule(z, E, Wt, anchor, u_draft, T, hidden, w, E1, sts_t, c_in, sps,
                                early_stop, max_B, self.tokens, self.q_lse, self.q_tok, self.c,
                                self.a, self.ell, self.row_off, self.B, self.E, self.ws, stream)

    def verify(self, z, E, Wt, anchor, target, u_acc, u_fin, T, tokens=None, q_lse=None,
               q_tok=None, ell=None, row_off=None, stream=None):
        B.dspark_verify(z, E, Wt, anchor, self.tokens if tokens is None else tokens,
                        self.q_lse if q_lse is None else q_lse,
                        self.q_tok if q_tok is None else q_tok,
                        self.ell if ell is None else ell,
                        self.row_off if row_off is None else row_off, target, u_acc, u_fin, T,
                        self.n_acc, self.out_tokens,
                        self.p_lse if self.p_lse.numel() >= target.shape[0] else None, self.ws,
                        stream)

    def status(self, clear=False) -> int:
        return B.device_status(self.ws, clear)
