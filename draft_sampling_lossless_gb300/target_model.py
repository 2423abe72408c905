"""Stand-in for the target model's forward pass (harness only).

The target model is outside the library's path: verification consumes its
logits as an input.  The workload descriptions fix how those logits relate
to the draft: for draft position j+1 the target is correlated with the
draft's own logits at that position -- the backbone's base logits plus the
Markov bias of the previous token -- so for request n

    t[n, j] = alpha_n * (z[n, j] + E[x_j] W) + sigma_n * noise[n, j],
    x_0 = anchor[n], x_j = tokens[n, j-1],

and the bonus row (after the last draft position) is alpha_n * z' + noise
with fresh logits z'.  The greedy workload's target row is z + E[x_j] W with
one token raised to the row maximum + 1: the drafted token with probability
0.8, else another token.  With the RNN head the draft's bias row at position
j+1 is its state s_j instead of E[x_j] (``states``, [R, gamma, r]).

The Markov bias here is a plain fp32 torch matmul over the gathered E rows;
the random draws (alpha, noise, z', the greedy picks) come from
``synth.target_draws``.  The same tensor is handed to both the CUDA library
and the CPU oracle, so this module's own rounding decides nothing in a
parity comparison.  An anchor of -1 means no bias at the first position.
"""

from __future__ import annotations

import torch

from . import synth


def _bias(inp: synth.Inputs, prev: torch.Tensor) -> torch.Tensor:
    """[n, V] fp32: E[prev] @ W, rows with prev < 0 zero."""
    ok = prev >= 0
    rows = torch.zeros((prev.shape[0], inp.E.shape[1]), dtype=torch.float32, device=inp.E.device)
    rows[ok] = inp.E[prev[ok]].float()
    return rows @ inp.W.float()


def target_logits(inp: synth.Inputs, tokens: torch.Tensor, seed: int | None = None,
                  states: torch.Tensor | None = None) -> torch.Tensor:
    """Dense target logits [R, gamma+1, V] in the workload's dtype: row j is
    the target distribution for draft position j+1, row gamma the bonus row.
    tokens: [R, gamma] drafted token ids (any integer dtype, any device);
    states: the RNN head's states [R, gamma, r], or None (Markov head)."""
    wl = inp.wl
    dev = inp.z.device
    R, G, V = wl.R, wl.gamma, wl.V
    dt = wl.torch_dtype
    dr = synth.target_draws(inp, seed)
    tok = tokens.to(dev).long()
    prev = torch.cat([inp.anchor.to(dev).long().view(R, 1), tok[:, : G - 1]], dim=1)  # x_j

    def bias(r0, r1):
        n = r1 - r0
        if states is not None:
            rows = states[r0:r1].to(dev).float().reshape(n * G, -1)
            return (rows @ inp.W.float()).view(n, G, V)
        return _bias(inp, prev[r0:r1].reshape(-1)).view(n, G, V)

    out = torch.empty((R, G + 1, V), dtype=dt, device=dev)
    if wl.target == "mix":
        for r0, r1, noise in dr.noise_chunks(wl, dev):
            y = inp.z[r0:r1].float() + bias(r0, r1)
            base = torch.cat([y, dr.z_bonus[r0:r1].float()], dim=1)
            a = dr.alpha[r0:r1].view(-1, 1, 1)
            s = dr.noise_std[r0:r1].view(-1, 1, 1)
            out[r0:r1] = (a * base + s * noise).to(dt)
        return out
    if wl.target == "greedy":
        for r0 in range(0, R, dr.chunk):
            r1 = min(R, r0 + dr.chunk)
            y = inp.z[r0:r1].float() + bias(r0, r1)
            out[r0:r1, :G] = y.to(dt)
        out[:, G:] = dr.z_bonus
        pick = torch.where(dr.keep, tok, (tok + 1 + dr.other) % V)
        rowmax = out[:, :G, :].float().amax(dim=-1)
        ridx = torch.arange(R, device=dev).view(-1, 1).expand(R, G)
        jidx = torch.arange(G, device=dev).view(1, -1).expand(R, G)
        out[ridx, jidx, pick] = (rowmax + 1.0).to(dt)
        return out
    raise ValueError(wl.target)
