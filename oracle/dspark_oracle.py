"""CPU oracle for the DSpark per-step hot path (TEST INFRASTRUCTURE ONLY).

Plain, slow, float64 numpy restatement of the four stages of one DSpark
speculative step.  It exists to check the CUDA library: only the test suite,
the package smoke check and the benchmark's CPU-baseline leg may import it.
The product path never calls it and shares no code with it.

Sources (page title, then section):

* "DeepSeek DSpark: Confidence-Scheduled Speculative Decoding 技术解析"
  (CSDN tutorial), section 四 "DSpark 的解法：半自回归 Draft" -- the draft
  head samples left to right, feeding the previous token into the next
  position.
* "DSpark.让每一轮计算，多走几步" (interactive explainer), "Markov head" panel
  -- a low-rank transition table adds a bias to the vocabulary scores before
  each draw; the two-token experiment (scores 0/0, +ln 9 gives 90%/10%);
  the survival panel (a_j = c_1 ... c_j; E = R + sum a; rate = E / T(B));
  the lossless panel (accept with min(1, p/q), resample from max(p - q, 0)
  normalised, bonus token from the next target distribution).
* "DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
  Generation" (news article), sections 2.1 (confidence head
  c_k = sigma(w . [h_k ; W1[x_{k-1}]]), sequential temperature scaling),
  2.2 (hardware-aware prefix scheduler: maximise tau * SPS(B) with
  B = sum_r (1 + l_r), greedy sort with early stop) and challenge 2 (global
  search without early stop).
* "为什么DSpark 可以加速推理？以及DSpark会不会导致降智？" (forum post),
  section "投机解码在数学上会不会影响最终生成结果？" -- acceptance
  probability sum_x min(p, q), failure mass sum_x max(0, p - q), and the
  emitted marginal equal to p.

Readings where the pages are silent:

* x_0 is the anchor token, so the Markov bias is applied from the first
  draft position on; an anchor of -1 switches the first-position bias off.
* The temperature divides the sum of base logit and bias; the same
  temperature is applied to the target logits.  Temperature 0 is greedy.
* Inverse CDF: with u in [0, 1), the token is the smallest v whose running
  sum C_v (accumulated in index order) exceeds u * C_{V-1}; if rounding
  leaves none, the last token with non-zero weight.
* Confidence head: no bias term; W1 is the Markov embedding E; STS divides
  the confidence logit by t_k.
* Scheduler: Theta_i = (R + S_i) * SPS[R + i], with S_i the sum of the i
  largest survival values taken in the order (a descending, request
  ascending, position ascending); every a is rounded to the nearest multiple
  of 2^-40 and summed as an integer so that the sum does not depend on the
  order of additions.  Early stop adds candidate i+1 only while
  Theta_{i+1} > Theta_i; global mode takes the first argmax.
* Capacity scheduling: a capacity K fixed before the step (the batch the
  global search chose on the survival values two steps earlier) is filled
  with the first min(max(K - R, 0), R * gamma) candidates of the current
  order.
* RNN sequential head (the pages name it and give no formula): an Elman
  recurrence over the block's prefix, s_k = tanh(E[x_{k-1}] + s_{k-1} U) with
  s_{-1} = 0 and U an r x r matrix; s_k takes the place of the Markov row
  E[x_{k-1}] in the bias (bias_k = s_k W), so U = 0 leaves a one-token
  memory.  The confidence head keeps W1[x_{k-1}] as written.  The state is
  stored in the table's type (bf16 or fp32) and its pre-activation is
  accumulated in fp32 -- the embedding first, then the fused multiply-adds
  s_{k-1}[i] * U[i][j] for i ascending -- and tanh is taken in float64: the
  stored state is a quantised value, so both implementations take its
  rounding in the same precision.
* Verification: accept draft position j iff u_acc < p_j(x_j) / q_j(x_j)
  (strict); on the first rejection sample max(0, p - q) normalised with the
  request's final uniform, or p itself if that mass is zero; if every
  verified position is accepted, sample the bonus row with the final uniform.
  Greedy: accept iff the draft token is the target argmax (lowest index on
  ties); the correction / bonus token is the target argmax.

All functions take float64 numpy arrays (bf16 / fp32 inputs converted
exactly) and integer arrays; they are vectorised over requests only.
"""

from __future__ import annotations

import numpy as np

FIX_SHIFT = 40  # survival values are summed as integers in units of 2^-40


# --------------------------------------------------------------------------
# Markov bias and draft distribution (explainer "Markov head" panel;
# news article section 创新一, second stage: low-rank matrix implementation)
# --------------------------------------------------------------------------

def markov_bias(E: np.ndarray, W: np.ndarray, prev: np.ndarray) -> np.ndarray:
    """bias[n, v] = sum_i E[prev[n], i] * W[i, v]; rows with prev < 0 are zero.

    E: [V, r], W: [r, V] (float64), prev: [n] token ids.  Returns [n, V].
    """
    prev = np.asarray(prev, dtype=np.int64)
    rows = np.zeros((prev.shape[0], E.shape[1]), dtype=np.float64)
    ok = prev >= 0
    rows[ok] = E[prev[ok]]
    return rows @ W


def inverse_cdf(weights: np.ndarray, u: np.ndarray) -> np.ndarray:
    """Smallest v with C_v > u * C_{V-1}, C the index-order running sum.

    weights: [n, V] non-negative float64; u: [n].  Rows whose threshold is not
    exceeded (rounding) take their last token with non-zero weight.
    """
    C = np.cumsum(weights, axis=1)
    thr = u * C[:, -1]
    idx = np.sum(C <= thr[:, None], axis=1)
    V = weights.shape[1]
    bad = idx >= V
    if np.any(bad):
        for n in np.nonzero(bad)[0]:
            nz = np.nonzero(weights[n] > 0)[0]
            idx[n] = nz[-1] if nz.size else V - 1
    return idx.astype(np.int64)


def first_argmax(y: np.ndarray) -> np.ndarray:
    """Lowest index attaining the row maximum (np.argmax returns the first)."""
    return np.argmax(y, axis=1).astype(np.int64)


def softmax_rows(y: np.ndarray):
    """(weights exp(y - max), lse) per row, float64."""
    m = np.max(y, axis=1)
    e = np.exp(y - m[:, None])
    S = np.cumsum(e, axis=1)[:, -1]
    return e, m + np.log(S)


def draft_sample(z, E, W, anchor, u_draft, T):
    """Semi-autoregressive draft with the Markov head.

    For k = 1..gamma (left to right): y = (z_k + E[x_{k-1}] W) / T,
    q_k = softmax(y), x_k = inverse_cdf(q_k, u_k).  Greedy when T == 0.

    z: [R, gamma, V]; returns tokens [R, gamma] int64, q_lse [R, gamma]
    (natural-log normaliser of y; the maximum of z + bias when greedy) and
    q_tok [R, gamma] = q_k(x_k) (1 when greedy).
    """
    R, G, V = z.shape
    tokens = np.zeros((R, G), dtype=np.int64)
    q_lse = np.zeros((R, G))
    q_tok = np.zeros((R, G))
    prev = np.asarray(anchor, dtype=np.int64).copy()
    for k in range(G):
        y = z[:, k, :] + markov_bias(E, W, prev)
        if T == 0.0:
            x = first_argmax(y)
            q_lse[:, k] = y[np.arange(R), x]
            q_tok[:, k] = 1.0
        else:
            y = y / T
            e, lse = softmax_rows(y)
            x = inverse_cdf(e, u_draft[:, k])
            q_lse[:, k] = lse
            q_tok[:, k] = np.exp(y[np.arange(R), x] - lse)
        tokens[:, k] = x
        prev = x
    return tokens, q_lse, q_tok


def draft_distribution(z_k, E, W, prev, T):
    """q over the vocabulary for one position: softmax((z_k + E[prev] W)/T)."""
    y = (z_k + markov_bias(E, W, prev)) / T
    e, lse = softmax_rows(y)
    return np.exp(y - lse[:, None])


# --------------------------------------------------------------------------
# RNN sequential head (news article section 创新一, second stage: the RNN head
# keeps a recurrent state and so captures longer dependencies; explainer,
# Markov-head panel: an RNN head accumulates the prefix inside the block)
# --------------------------------------------------------------------------

def round_to(x, dtype: str) -> np.ndarray:
    """Round float64 values to the nearest bf16 ("bf16") or fp32 ("f32")
    value, ties to even, in one step; returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f32":
        return x.astype(np.float32).astype(np.float64)
    m, e = np.frexp(x)  # x = m 2^e, 0.5 <= |m| < 1: 8 significant bits kept
    out = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    tiny = np.abs(x) < 2.0 ** -126  # bf16 subnormals: spacing 2^-133
    out[tiny] = np.ldexp(np.rint(np.ldexp(x[tiny], 133)), -133)
    return out


def fma32(a, b, c) -> np.ndarray:
    """fp32 fused multiply-add a * b + c with a single rounding (IEEE 754),
    for fp32 operands.  The product is exact in float64; TwoSum gives the
    float64 sum's rounding error, which decides the fp32 rounding when the
    float64 sum lands exactly half-way between two fp32 values."""
    a, b, c = (np.asarray(t, dtype=np.float32).astype(np.float64) for t in (a, b, c))
    a, b, c = np.broadcast_arrays(a, b, c)
    p = a * b
    hi = p + c
    bv = hi - p
    lo = (p - (hi - bv)) + (c - bv)
    f = hi.astype(np.float32)
    d = hi - f.astype(np.float64)
    g = np.nextafter(f, np.where(d > 0, np.float32(np.inf), np.float32(-np.inf)))
    half = (d != 0) & (hi == (f.astype(np.float64) + g.astype(np.float64)) / 2)
    flip = half & (lo != 0) & (np.sign(lo) == np.sign(d))
    return np.where(flip, g, f)


def rnn_state(E, U, prev, s_prev, dtype: str) -> np.ndarray:
    """s = round(tanh(pre)) for a batch of requests: pre[n, j] starts from
    E[prev[n], j] (0 when prev < 0) and adds s_prev[n, i] * U[i, j] for
    i = 0..r-1 in fp32 fused multiply-adds; tanh in float64; rounded to the
    state type.  E: [V, r], U: [r, r], prev: [n], s_prev: [n, r]."""
    prev = np.asarray(prev, dtype=np.int64)
    r = E.shape[1]
    acc = np.zeros((prev.shape[0], r), dtype=np.float32)
    ok = prev >= 0
    acc[ok] = E[prev[ok]].astype(np.float32)
    for i in range(r):
        acc = fma32(s_prev[:, i : i + 1], U[i][None, :], acc)
    return round_to(np.tanh(acc.astype(np.float64)), dtype)


def rnn_states(E, U, anchor, tokens, dtype: str) -> np.ndarray:
    """The states s_0..s_{gamma-1} of given drafts: s_k from x_{k-1} (the
    anchor for k = 0) and s_{k-1}.  Returns [R, gamma, r] float64."""
    tokens = np.asarray(tokens, dtype=np.int64)
    R, G = tokens.shape
    S = np.zeros((R, G, E.shape[1]))
    s = np.zeros((R, E.shape[1]))
    for k in range(G):
        prev = np.asarray(anchor, dtype=np.int64) if k == 0 else tokens[:, k - 1]
        s = rnn_state(E, U, prev, s, dtype)
        S[:, k] = s
    return S


def draft_distribution_rows(z_k, rows, W, T):
    """q over the vocabulary for one position with bias rows @ W:
    softmax((z_k + rows W) / T)."""
    y = (z_k + np.asarray(rows, dtype=np.float64) @ W) / T
    e, lse = softmax_rows(y)
    return np.exp(y - lse[:, None])


def draft_sample_rnn(z, E, U, W, anchor, u_draft, T, dtype: str):
    """Semi-autoregressive draft with the RNN head: for k = 0..gamma-1,
    s_k = rnn_state(x_{k-1}, s_{k-1}), y = (z_k + s_k W) / T, q_k = softmax(y),
    x_k = inverse_cdf(q_k, u_k) (greedy when T == 0).  Returns tokens,
    q_lse, q_tok as draft_sample does, and the states S [R, gamma, r]."""
    R, G, V = z.shape
    tokens = np.zeros((R, G), dtype=np.int64)
    q_lse = np.zeros((R, G))
    q_tok = np.zeros((R, G))
    S = np.zeros((R, G, E.shape[1]))
    s = np.zeros((R, E.shape[1]))
    prev = np.asarray(anchor, dtype=np.int64).copy()
    for k in range(G):
        s = rnn_state(E, U, prev, s, dtype)
        S[:, k] = s
        y = z[:, k, :] + s @ W
        if T == 0.0:
            x = first_argmax(y)
            q_lse[:, k] = y[np.arange(R), x]
            q_tok[:, k] = 1.0
        else:
            y = y / T
            e, lse = softmax_rows(y)
            x = inverse_cdf(e, u_draft[:, k])
            q_lse[:, k] = lse
            q_tok[:, k] = np.exp(y[np.arange(R), x] - lse)
        tokens[:, k] = x
        prev = x
    return tokens, q_lse, q_tok, S


# --------------------------------------------------------------------------
# Confidence head, STS and survival (news article section 2.1; explainer
# survival panel)
# --------------------------------------------------------------------------

def confidence(h, w, E1, anchor, tokens, sts_t, c_in=None):
    """c_{r,k} = sigmoid((w . [h_{r,k}; E1[x_{k-1}]]) / t_k); a = cumprod_k c.

    h: [R, gamma, d], w: [d + r], E1: [V, r].  When c_in is given the head is
    skipped and only the survival product runs.  Returns (c, a) float64.
    """
    if c_in is None:
        R, G, d = h.shape
        c = np.zeros((R, G))
        for k in range(G):
            prev = anchor if k == 0 else tokens[:, k - 1]
            prev = np.asarray(prev, dtype=np.int64)
            emb = np.zeros((R, E1.shape[1]))
            ok = prev >= 0
            emb[ok] = E1[prev[ok]]
            s = h[:, k, :] @ w[:d] + emb @ w[d:]
            c[:, k] = 1.0 / (1.0 + np.exp(-s / sts_t[k]))
    else:
        c = np.asarray(c_in, dtype=np.float64)
    R, G = c.shape
    a = np.zeros((R, G))
    run = np.ones(R)
    for k in range(G):
        run = run * c[:, k]
        a[:, k] = run
    return c, a


# --------------------------------------------------------------------------
# Hardware-aware prefix scheduler (news article section 2.2 and challenge 2;
# explainer survival panel: E = R + sum a, rate = E / T(B))
# --------------------------------------------------------------------------

def to_fixed(a: np.ndarray) -> np.ndarray:
    """Nearest multiple of 2^-40 (ties to even), as int64 units."""
    return np.rint(np.asarray(a, dtype=np.float64) * float(1 << FIX_SHIFT)).astype(np.int64)


def schedule(a, sps, early_stop=True, max_B=0):
    """Greedy prefix scheduler.

    a: [R, gamma] survival values (the fp32 values, as float64); sps: [n]
    steps/s for B = 0..n-1.  Candidates are ordered by (a desc, request asc,
    position asc).  Returns dict(ell [R], row_off [R+1], B, E, i_star, theta).
    """
    a = np.asarray(a, dtype=np.float64)
    R, G = a.shape
    N = R * G
    rr, jj = np.meshgrid(np.arange(R), np.arange(G), indexing="ij")
    flat_a, flat_r, flat_j = a.ravel(), rr.ravel(), jj.ravel()
    order = np.lexsort((flat_j, flat_r, -flat_a))
    fx = to_fixed(flat_a[order])
    S = np.concatenate([[0], np.cumsum(fx)])  # S[i] = sum of the top i
    imax = N if max_B <= 0 else max(0, min(N, max_B - R))
    if R + imax >= len(sps):
        raise ValueError("SPS table shorter than the largest batch considered")
    theta = np.zeros(imax + 1)
    for i in range(imax + 1):
        e_i = float(R) + float(S[i]) * 2.0 ** -FIX_SHIFT
        theta[i] = e_i * float(sps[R + i])
    if early_stop:
        i_star = imax
        for i in range(imax):
            if not theta[i + 1] > theta[i]:
                i_star = i
                break
    else:
        i_star = int(np.argmax(theta))
    ell = np.bincount(flat_r[order[:i_star]], minlength=R).astype(np.int64)
    row_off = np.concatenate([[0], np.cumsum(1 + ell)]).astype(np.int64)
    E = float(R) + float(S[i_star]) * 2.0 ** -FIX_SHIFT
    return dict(ell=ell, row_off=row_off, B=int(R + i_star), E=E, i_star=int(i_star),
                theta=theta, order=order)


def schedule_capacity(a, K):
    """Capacity scheduling (news article, challenge 2): the verification
    capacity K (a batch size fixed before this step, e.g. the batch the global
    search chose on the survival values two steps earlier) is filled with the
    current candidates in the current order, so the batch is exactly the first
    i = min(max(K - R, 0), R * gamma) candidates.  Returns dict(ell, row_off,
    B, E, i_star)."""
    a = np.asarray(a, dtype=np.float64)
    R, G = a.shape
    N = R * G
    rr, jj = np.meshgrid(np.arange(R), np.arange(G), indexing="ij")
    order = np.lexsort((jj.ravel(), rr.ravel(), -a.ravel()))
    i = int(max(0, min(N, int(K) - R)))
    S = int(np.sum(to_fixed(a.ravel()[order[:i]])))
    ell = np.bincount(rr.ravel()[order[:i]], minlength=R).astype(np.int64)
    row_off = np.concatenate([[0], np.cumsum(1 + ell)]).astype(np.int64)
    E = float(R) + float(S) * 2.0 ** -FIX_SHIFT
    return dict(ell=ell, row_off=row_off, B=int(R + i), E=E, i_star=i)


# --------------------------------------------------------------------------
# Lossless verification (forum post, lossless proof; explainer lossless
# panel; tutorial section 五 acceptance rule)
# --------------------------------------------------------------------------

def _row_lse(target, rows, T, chunk=256):
    """Natural-log normaliser of target[rows] / T (row maximum when greedy)."""
    out = np.zeros(len(rows))
    for s in range(0, len(rows), chunk):
        blk = target[rows[s : s + chunk]]
        if T == 0.0:
            out[s : s + chunk] = np.max(blk, axis=1)
        else:
            _, l = softmax_rows(blk / T)
            out[s : s + chunk] = l
    return out


def verify(z, E, W, anchor, tokens, T, ell, row_off, target, u_acc, u_fin, states=None):
    """Rejection-sampling (or greedy) verification of the scheduled prefixes.

    With states ([R, gamma, r], the RNN head's) the draft distribution of
    position j is rebuilt with the bias states[r, j] W instead of E[x_{j-1}] W.

    target: [B_rows, V]; the rows of request r are row_off[r] + j for
    j = 0..ell[r]; row j is the target distribution for draft position j+1
    and row ell[r] the bonus row.  Returns dict(n_acc [R], out_tokens
    [R, gamma+1] (-1 padded), p_lse (dict row -> lse, or row maximum when
    greedy), final_kind [R] (0 bonus, 1 residual, 2 residual mass zero so
    p is used), final_row [R]).
    """
    R, G, V = z.shape
    anchor = np.asarray(anchor, dtype=np.int64)
    tokens = np.asarray(tokens, dtype=np.int64)
    ell = np.asarray(ell, dtype=np.int64)
    row_off = np.asarray(row_off, dtype=np.int64)
    rows = np.concatenate([row_off[r] + np.arange(ell[r] + 1) for r in range(R)])
    p_lse = dict(zip(rows.tolist(), _row_lse(target, rows, T).tolist()))

    # Sequential acceptance over positions, vectorised over requests.
    n_acc = ell.copy()
    decided = np.zeros(R, dtype=bool)
    for j in range(G):
        idx = np.nonzero((~decided) & (j < ell))[0]
        if idx.size == 0:
            continue
        trow = target[row_off[idx] + j]
        x = tokens[idx, j]
        if T == 0.0:
            acc = first_argmax(trow) == x
        else:
            y = trow / T
            _, lse = softmax_rows(y)
            p_x = np.exp(y[np.arange(idx.size), x] - lse)
            if states is None:
                prev = anchor[idx] if j == 0 else tokens[idx, j - 1]
                q = draft_distribution(z[idx, j, :], E, W, prev, T)
            else:
                q = draft_distribution_rows(z[idx, j, :], states[idx, j, :], W, T)
            q_x = q[np.arange(idx.size), x]
            acc = u_acc[idx, j] < p_x / q_x
        rej = idx[~acc]
        n_acc[rej] = j
        decided[rej] = True

    out = -np.ones((R, G + 1), dtype=np.int64)
    for r in range(R):
        out[r, : n_acc[r]] = tokens[r, : n_acc[r]]
    final_row = row_off[:R] + n_acc
    rejected = n_acc < ell
    kind = np.where(rejected, 1, 0).astype(np.int64)
    final_tok = np.zeros(R, dtype=np.int64)
    if T == 0.0:
        final_tok = first_argmax(target[final_row])
    else:
        y = target[final_row] / T
        _, lse = softmax_rows(y)
        p = np.exp(y - lse[:, None])
        w = p.copy()
        ridx = np.nonzero(rejected)[0]
        if ridx.size:
            j = n_acc[ridx]
            if states is None:
                prev = np.where(j == 0, anchor[ridx], tokens[ridx, np.maximum(j - 1, 0)])
                q = draft_distribution(z[ridx, j, :], E, W, prev, T)
            else:
                q = draft_distribution_rows(z[ridx, j, :], states[ridx, j, :], W, T)
            res = np.maximum(0.0, p[ridx] - q)
            zero = ~(np.sum(res, axis=1) > 0.0)
            res[zero] = p[ridx[zero]]
            kind[ridx[zero]] = 2
            w[ridx] = res
        final_tok = inverse_cdf(w, np.asarray(u_fin, dtype=np.float64))
    out[np.arange(R), n_acc] = final_tok
    return dict(n_acc=n_acc, out_tokens=out, p_lse=p_lse, final_kind=kind,
                final_row=final_row)


def final_weights(z, E, W, anchor, tokens, T, target_row, j, r, rejected, states=None):
    """The distribution the final token of request r is drawn from
    (residual when rejected at position j+1, else the bonus row's p);
    used by the tests to classify near-ties.  states: as in verify."""
    y = target_row[None, :] / T
    e, lse = softmax_rows(y)
    p = np.exp(y - lse[:, None])
    if not rejected:
        return p[0]
    if states is None:
        prev = np.array([anchor[r] if j == 0 else tokens[r, j - 1]])
        q = draft_distribution(z[r : r + 1, j, :], E, W, prev, T)
    else:
        q = draft_distribution_rows(z[r : r + 1, j, :], states[r : r + 1, j, :], W, T)
    w = np.maximum(0.0, p - q)
    return w[0] if np.sum(w) > 0 else p[0]
