"""Pins for the CPU oracle: values printed on the pages, closed forms,
invariants and brute force on tiny inputs.  None of these re-derives a value
from the oracle's own formula; each would fail under a plausible slip (a
dropped bias term, a swapped p/q, an off-by-one position, a missing +R)."""

import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle  # noqa: F401
import oracle.dspark_oracle as numpy_oracle
from oracle import native as cpp_oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(params=["numpy", "cpp"], scope="module")
def orc(request):
    """Both oracles: the numpy restatement and the plain C++ one."""
    if request.param == "cpp":
        cpp_oracle.build()
        return cpp_oracle
    return numpy_oracle


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def uni24(rng, shape):
    return rng.integers(0, 1 << 24, size=shape).astype(np.float64) * 2.0 ** -24


# ---------------------------------------------------------------- Markov head

def test_markov_two_token_toy(orc):
    g = gold("markov_two_token.json")
    # V = 2, rank 1: E[A] = 1, W = (ln 9, 0): the previous token A adds ln 9 to A.
    E = np.array([[1.0], [0.0]])
    W = np.array([[math.log(9.0), 0.0]])
    z = np.array(g["base_logits"]).reshape(1, 1, 2)
    q = orc.draft_distribution(z[:, 0, :], E, W, np.array([0]), 1.0)[0]
    assert np.allclose(q, g["q_after"], atol=1e-12, rtol=0)
    q0 = orc.draft_distribution(z[:, 0, :], E, W, np.array([-1]), 1.0)[0]
    assert np.allclose(q0, g["q_before"], atol=1e-15, rtol=0)
    # The sampled token, its probability and the normaliser: closed forms.
    for u, want in [(0.0, 0), (0.8999, 0), (0.9, 1), (0.99, 1)]:
        tok, lse, qt = orc.draft_sample(z, E, W, np.array([0]), np.array([[u]]), 1.0)
        assert tok[0, 0] == want
        assert abs(lse[0, 0] - math.log(10.0)) < 1e-12  # ln(e^{ln 9} + e^0)
        assert abs(qt[0, 0] - (0.9 if want == 0 else 0.1)) < 1e-12


def test_temperature_scales_logit_plus_bias(orc):
    E = np.array([[1.0], [0.0]])
    W = np.array([[math.log(9.0), 0.0]])
    z = np.zeros((1, 2))
    for T in (0.5, 0.7, 2.0):
        q = orc.draft_distribution(z, E, W, np.array([0]), T)[0]
        k = 9.0 ** (1.0 / T)
        assert abs(q[0] - k / (k + 1.0)) < 1e-12


def test_draft_feeds_previous_token_left_to_right(orc):
    # One-hot embedding (non-symmetric permutation) and a transition that
    # strongly favours perm[prev]; base logits zero.  The draft must follow
    # the chain anchor -> perm[anchor] -> perm[perm[anchor]] ...
    V = 6
    perm = np.array([3, 0, 5, 1, 2, 4])
    E = np.eye(V)[[2, 0, 1, 5, 3, 4]]  # row v of E is one-hot at emb_idx[v]
    emb_idx = np.argmax(E, axis=1)
    W = np.full((V, V), -30.0)
    for v in range(V):
        W[emb_idx[v], perm[v]] = 30.0
    G = 5
    z = np.zeros((2, G, V))
    u = np.full((2, G), 0.5)
    tok, _, qt = orc.draft_sample(z, E, W, np.array([1, 4]), u, 1.0)
    for r, a0 in enumerate([1, 4]):
        x = a0
        for k in range(G):
            x = perm[x]
            assert tok[r, k] == x
    assert np.all(qt > 1 - 1e-12)


def test_anchor_minus_one_disables_first_bias(orc):
    E = np.array([[1.0], [0.0]])
    W = np.array([[-50.0, 0.0]])
    z = np.array([[[2.0, 0.0]]])
    # with the anchor bias token 0 would be all but impossible
    tok_b, _, _ = orc.draft_sample(z, E, W, np.array([0]), np.array([[0.5]]), 1.0)
    tok_n, _, _ = orc.draft_sample(z, E, W, np.array([-1]), np.array([[0.5]]), 1.0)
    assert tok_b[0, 0] == 1 and tok_n[0, 0] == 0


def test_greedy_draft_lowest_index_on_ties(orc):
    z = np.array([[[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 0.0, 5.0]]])
    E = np.zeros((4, 1))
    W = np.zeros((1, 4))
    tok, lse, qt = orc.draft_sample(z, E, W, np.array([0]), np.zeros((1, 2)), 0.0)
    assert tok.tolist() == [[1, 0]]
    assert lse.tolist() == [[3.0, 5.0]] and qt.tolist() == [[1.0, 1.0]]


# ---------------------------------------------------------------- inverse CDF

def test_inverse_cdf_boundary_reading(orc):
    w = np.array([[1.0, 1.0, 1.0, 1.0]])
    # smallest v with C_v > u * S: at u*S exactly on a boundary, the next token
    assert orc.inverse_cdf(w, np.array([0.25]))[0] == 1
    assert orc.inverse_cdf(w, np.array([0.25 - 2 ** -24]))[0] == 0
    assert orc.inverse_cdf(w, np.array([0.0]))[0] == 0
    # zero-weight tokens are never drawn
    w2 = np.array([[0.0, 2.0, 0.0, 0.0, 2.0, 0.0]])
    got = [orc.inverse_cdf(w2, np.array([u]))[0] for u in (0.0, 0.49, 0.5, 0.99)]
    assert got == [1, 1, 4, 4]


def test_inverse_cdf_brute_force_small_vocab(orc):
    rng = np.random.default_rng(7)
    for V in range(1, 9):
        for _ in range(20):
            w = rng.integers(0, 5, size=V).astype(np.float64)
            if w.sum() == 0:
                w[rng.integers(V)] = 1.0
            S = w.sum()
            for k in range(0, 64):
                u = k / 64.0
                # explicit CDF table, integer arithmetic: first v with cum > u*S
                want, cum = None, 0.0
                for v in range(V):
                    cum += w[v]
                    if cum > u * S:
                        want = v
                        break
                assert orc.inverse_cdf(w[None, :], np.array([u]))[0] == want


def test_softmax_two_token_closed_form(orc):
    rng = np.random.default_rng(3)
    for _ in range(50):
        a, b = rng.normal(0, 5, size=2)
        e, lse = orc.softmax_rows(np.array([[a, b]]))
        want_lse = max(a, b) + math.log1p(math.exp(-abs(a - b)))
        assert abs(lse[0] - want_lse) < 1e-12
        p0 = math.exp(a - lse[0])
        assert abs(p0 - 1.0 / (1.0 + math.exp(b - a))) < 1e-12


# ---------------------------------------------------------------- confidence

def test_confidence_closed_forms_and_indexing(orc):
    # d = 1, rank 1.  Feature vector [h_k ; E1[x_{k-1}]].
    R, G, d, V = 1, 3, 1, 4
    h = np.array([[[1.0], [0.0], [0.0]]])
    E1 = np.array([[0.0], [1.0], [0.0], [2.0]])
    w = np.array([math.log(3.0), -math.log(3.0)])
    anchor = np.array([0])  # E1[0] = 0
    tokens = np.array([[1, 3, 2]])  # x_1 = 1 (E1 = 1), x_2 = 3 (E1 = 2)
    t = np.array([1.0, 1.0, 2.0])
    c, a = orc.confidence(h, w, E1, anchor, tokens, t)
    # k=1: s = ln3 -> 0.75 ; k=2: s = -ln3 (E1[x_1]=1) -> 0.25 ;
    # k=3: s = -2 ln3 (E1[x_2]=2), t=2 -> sigmoid(-ln3) = 0.25
    assert np.allclose(c[0], [0.75, 0.25, 0.25], atol=1e-15)
    assert np.allclose(a[0], [0.75, 0.1875, 0.046875], atol=1e-15)


def test_survival_chain_page_values(orc):
    g = gold("survival_chain.json")
    for case in g["cases"]:
        c = np.array([[case["c1"]] + g["conditionals_after_first"]])
        _, a = orc.confidence(None, None, None, None, None, None, c_in=c)
        assert np.allclose(a[0], case["a"], rtol=1e-14, atol=0)
    g = gold("tutorial_worked_example.json")
    _, a = orc.confidence(None, None, None, None, None, None,
                             c_in=np.array([g["confidences"]]))
    assert np.allclose(a[0], g["survival_products"], rtol=1e-14, atol=0)


def test_survival_never_increases(orc):
    rng = np.random.default_rng(11)
    c = rng.uniform(0, 1, size=(64, 16))
    c[:, 3] = 1.0  # c rounding to one
    c[5, :] = 1.0
    _, a = orc.confidence(None, None, None, None, None, None, c_in=c)
    assert np.all(np.diff(a, axis=1) <= 0)
    assert np.all(a[5] == 1.0)


# ---------------------------------------------------------------- scheduler

def sps_from_cost_model(n, load=1.0):
    g = gold("scheduler_cost_model.json")["T_ms"]
    B = np.arange(n, dtype=np.float64)
    T = g["const"] + (g["lin0"] + g["lin_load"] * load) * B + g["quad_load"] * load * B * B
    return (1000.0 / T).astype(np.float32).astype(np.float64)


def brute_force_best(a, sps):
    """Enumerate every allocation l in {0..gamma}^R (prefixes per request);
    Theta(l) = (R + sum of the first l_r survival values of each request)
    * SPS[R + sum l].  Sums in the same 2^-40 integer units."""
    R, G = a.shape
    fx = np.rint(np.asarray(a) * 2.0 ** 40).astype(np.int64)
    best, arg = None, []
    for ell in itertools.product(range(G + 1), repeat=R):
        s = sum(int(fx[r, :l].sum()) for r, l in enumerate(ell))
        th = (float(R) + float(s) * 2.0 ** -40) * float(sps[R + sum(ell)])
        if best is None or th > best:
            best, arg = th, [ell]
        elif th == best:
            arg.append(ell)
    return best, arg


def random_survival(rng, R, G):
    c = rng.uniform(0.05, 1.0, size=(R, G))
    return np.cumprod(c, axis=1).astype(np.float32).astype(np.float64)


def unimodal(theta):
    i = int(np.argmax(theta))
    return np.all(np.diff(theta[: i + 1]) > 0) and np.all(np.diff(theta[i:]) <= 0)


@pytest.mark.parametrize("R,G", [(1, 4), (2, 3), (3, 2), (2, 4), (3, 3)])
def test_scheduler_brute_force(orc, R, G):
    rng = np.random.default_rng(100 * R + G)
    n_uni = 0
    for trial in range(40):
        a = random_survival(rng, R, G)
        if trial % 2 == 0:
            sps = sps_from_cost_model(R * (G + 1) + 1, load=rng.uniform(0.2, 30.0))
        else:
            sps = rng.uniform(1.0, 100.0, size=R * (G + 1) + 1)
        best, args = brute_force_best(a, sps)
        glob = orc.schedule(a, sps, early_stop=False)
        assert glob["theta"][glob["i_star"]] == best
        if len(args) == 1:
            assert tuple(glob["ell"].tolist()) == args[0]
        es = orc.schedule(a, sps, early_stop=True)
        if unimodal(es["theta"]):
            n_uni += 1
            assert es["theta"][es["i_star"]] == best
            assert es["i_star"] == glob["i_star"]
        # prefix property: survival never increases within a request, so the
        # chosen set is the first l_r positions of each request.
        top = es["order"][: es["i_star"]]
        for r in range(R):
            js = sorted(int(o % G) for o in top if o // G == r)
            assert js == list(range(len(js)))
    assert n_uni > 0


def test_scheduler_early_stop_differs_on_sawtooth(orc):
    # One request, four candidates of 0.9.  SPS dips at B = 2 then recovers:
    # early stop keeps nothing, global search keeps all four.
    a = np.array([[0.9, 0.81, 0.729, 0.6561]], dtype=np.float32).astype(np.float64)
    sps = np.array([0.0, 100.0, 40.0, 60.0, 70.0, 80.0])
    es = orc.schedule(a, sps, early_stop=True)
    gl = orc.schedule(a, sps, early_stop=False)
    assert es["ell"].tolist() == [0] and es["B"] == 1 and es["E"] == 1.0
    assert gl["ell"].tolist() == [4] and gl["B"] == 5
    assert abs(gl["E"] - (1.0 + a.sum())) < 1e-9


def test_scheduler_plateau_stops(orc):
    # Throughput that stays flat is not rising: stop (strict comparison).
    a = np.zeros((1, 3))
    sps = np.full(5, 10.0)
    es = orc.schedule(a, sps, early_stop=True)
    assert es["i_star"] == 0 and es["ell"].tolist() == [0]


def test_scheduler_tie_order_request_then_position(orc):
    a = np.full((3, 2), 0.5)
    sps = 1000.0 / (1.0 + 0.0 * np.arange(10))  # constant rate: only E matters
    for i_cap, want in [(1, [1, 0, 0]), (2, [2, 0, 0]), (3, [2, 1, 0]), (5, [2, 2, 1])]:
        out = orc.schedule(a, sps, early_stop=False, max_B=3 + i_cap)
        assert out["ell"].tolist() == want
        assert out["row_off"].tolist() == [0, 1 + want[0], 2 + want[0] + want[1],
                                            3 + sum(want)]


def test_scheduler_sps_too_short_is_an_error(orc):
    with pytest.raises(ValueError):
        orc.schedule(np.full((2, 2), 0.5), np.ones(6), early_stop=True)


def test_fixed_point_rounds_half_to_even(orc):
    u = 2.0 ** -40
    assert orc.to_fixed(np.array([0.5 * u, 1.5 * u, 2.5 * u, 1.0])).tolist() == \
        [0, 2, 2, 1 << 40]


# ---------------------------------------------------------------- verification

def _two_token_step(orc, q, p, n, rng):
    """n independent one-position steps with draft q and target p (V = 2)."""
    z = np.log(np.array(q)).reshape(1, 1, 2).repeat(n, axis=0)
    E = np.zeros((2, 1))
    W = np.zeros((1, 2))
    anchor = np.zeros(n, dtype=np.int64)
    tok, _, _ = orc.draft_sample(z, E, W, anchor, uni24(rng, (n, 1)), 1.0)
    target = np.tile(np.log(np.array(p)), (2 * n, 1))  # row 0: position 1, row 1: bonus
    ell = np.ones(n, dtype=np.int64)
    row_off = np.arange(n + 1, dtype=np.int64) * 2
    out = orc.verify(z, E, W, anchor, tok, 1.0, ell, row_off, target,
                        uni24(rng, (n, 1)), uni24(rng, (n,)))
    return tok, out


@pytest.mark.parametrize("qi", [0, 1, 2, 3])
def test_lossless_marginal_chi_square(orc, qi):
    g = gold("lossless_two_token.json")
    p = np.array(g["p"])
    q = np.array(g["q_cases"][qi])
    n = g["trials"]
    rng = np.random.default_rng(2024 + qi)
    tok, out = _two_token_step(orc, q, p, n, rng)
    first = out["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=2).astype(np.float64)
    expect = n * p
    chi2 = float(np.sum((counts - expect) ** 2 / expect))
    assert chi2 < 10.828  # chi-square, 1 dof, alpha = 1e-3
    # acceptance rate equals sum_x min(p, q) within 4 sigma
    acc = float(np.mean(out["n_acc"] == 1))
    a_true = float(np.minimum(p, q).sum())
    sd = math.sqrt(a_true * (1 - a_true) / n) + 1e-12
    assert abs(acc - a_true) <= 4 * sd + 1e-12
    # the failure mass is the complement, sum_x max(0, p - q)
    assert abs((1 - acc) - float(np.maximum(0.0, p - q).sum())) <= 4 * sd + 1e-12
    # emitted count: accepted -> bonus token too (2), rejected -> 1
    assert np.all((out["out_tokens"][:, 1] >= 0) == (out["n_acc"] == 1))


def test_identity_q_equals_p_accepts_everything(orc):
    rng = np.random.default_rng(5)
    R, G, V = 8, 4, 16
    z = rng.normal(0, 2, size=(R, G, V))
    E = rng.normal(0, 0.3, size=(V, 3))
    W = rng.normal(0, 0.3, size=(3, V))
    anchor = rng.integers(0, V, size=R)
    tok, _, _ = orc.draft_sample(z, E, W, anchor, uni24(rng, (R, G)), 1.0)
    # target row j = exactly the draft's logits for position j+1
    target = np.zeros((R * (G + 1), V))
    prev = anchor.copy()
    for j in range(G):
        target[np.arange(R) * (G + 1) + j] = z[:, j, :] + orc.markov_bias(E, W, prev)
        prev = tok[:, j]
    target[np.arange(R) * (G + 1) + G] = rng.normal(0, 2, size=(R, V))
    ell = np.full(R, G)
    row_off = np.arange(R + 1) * (G + 1)
    out = orc.verify(z, E, W, anchor, tok, 1.0, ell, row_off, target,
                        uni24(rng, (R, G)), uni24(rng, (R,)))
    assert out["n_acc"].tolist() == [G] * R
    assert np.all(out["out_tokens"][:, :G] == tok)
    assert np.all(out["final_kind"] == 0)
    # sum_x min(p, q) = 1 when q = p
    q = orc.draft_distribution(z[:, 0, :], E, W, anchor, 1.0)
    assert np.allclose(np.minimum(q, q).sum(axis=1), 1.0, atol=1e-12)


def test_greedy_verify_argmax_match(orc):
    V, G = 5, 3
    z = np.zeros((3, G, V))
    E = np.zeros((V, 1))
    W = np.zeros((1, V))
    anchor = np.zeros(3, dtype=np.int64)
    tokens = np.array([[1, 2, 3], [1, 2, 3], [4, 4, 4]])
    rows = []
    # request 0: rows argmax 1, 2, 0 (mismatch at position 3), bonus unused
    for am in (1, 2, 0, 4):
        rows.append(np.eye(V)[am] * 3.0)
    # request 1: all three match, bonus row argmax 0 (tie 0/3 -> lowest index)
    for am in (1, 2, 3):
        rows.append(np.eye(V)[am] * 3.0)
    rows.append(np.array([7.0, 0.0, 0.0, 7.0, 0.0]))
    # request 2: only two verified (l = 2); second mismatches
    for am in (4, 1, 2):
        rows.append(np.eye(V)[am] * 3.0)
    target = np.array(rows)
    ell = np.array([3, 3, 2])
    row_off = np.array([0, 4, 8, 11])
    out = orc.verify(z, E, W, anchor, tokens, 0.0, ell, row_off, target,
                        np.zeros((3, G)), np.zeros(3))
    assert out["n_acc"].tolist() == [2, 3, 1]
    assert out["out_tokens"].tolist() == [[1, 2, 0, -1], [1, 2, 3, 0], [4, 1, -1, -1]]


def test_verify_rejection_never_accepts_zero_target_mass(orc):
    # p(x) = 0 for the drafted token: strict u < p/q never accepts, even u = 0
    z = np.array([[[0.0, 0.0]]])
    E = np.zeros((2, 1))
    W = np.zeros((1, 2))
    target = np.array([[0.0, -np.inf], [0.0, 0.0]])
    out = orc.verify(z, E, W, np.array([0]), np.array([[1]]), 1.0, np.array([1]),
                        np.array([0, 2]), target, np.array([[0.0]]), np.array([0.7]))
    assert out["n_acc"].tolist() == [0]
    assert out["out_tokens"][0].tolist() == [0, -1]


# ------------------------------------------- verification branches, closed forms

def _chi2_two(counts, p):
    n = counts.sum()
    expect = n * np.asarray(p)
    return float(np.sum((counts - expect) ** 2 / expect))


def test_verify_at_temperature_half_two_token(orc):
    """T = 0.5 on V = 2 (forum post, lossless proof; explainer, lossless panel;
    the temperature reading): the target row t = (0, ln 4) gives
    p = softmax(t / T) = (1/17, 16/17) (p = (0.2, 0.8) if the row were not
    divided by T), the draft q = (1/2, 1/2).  Acceptance = sum min(p, q) =
    1/17 + 1/2, the emitted marginal is p, the bonus token after an
    acceptance follows the bonus row's p, and the row's normaliser is
    ln(1 + 16)."""
    T, n = 0.5, 400_000
    rng = np.random.default_rng(99)
    p = np.array([1.0, 16.0]) / 17.0
    z = np.zeros((n, 1, 2))
    E, W = np.zeros((2, 1)), np.zeros((1, 2))
    anchor = np.zeros(n, dtype=np.int64)
    tok = rng.integers(0, 2, size=(n, 1))  # x_1 ~ q = (1/2, 1/2)
    target = np.tile(np.array([0.0, math.log(4.0)]), (2 * n, 1))  # position 1, bonus
    out = orc.verify(z, E, W, anchor, tok, T, np.ones(n, dtype=np.int64),
                     np.arange(n + 1, dtype=np.int64) * 2, target, uni24(rng, (n, 1)),
                     uni24(rng, (n,)))
    acc = float(np.mean(out["n_acc"] == 1))
    a_true = float(np.minimum(p, 0.5).sum())
    assert abs(acc - a_true) <= 4 * math.sqrt(a_true * (1 - a_true) / n)
    first = out["out_tokens"][:, 0]
    assert _chi2_two(np.bincount(first, minlength=2).astype(np.float64), p) < 10.828
    # after an acceptance the bonus token is drawn from the bonus row's p
    bonus = out["out_tokens"][out["n_acc"] == 1, 1]
    assert _chi2_two(np.bincount(bonus, minlength=2).astype(np.float64), p) < 10.828
    for row in (0, 1, 2 * n - 1):
        assert abs(out["p_lse"][row] - math.log(17.0)) < 1e-12


def test_rejection_at_second_position_uses_the_previous_token(orc):
    """gamma = 2; position 1 is always accepted (draft and target rows equal),
    position 2's draft depends on x_1 through the Markov bias: E = (1, -1),
    W = (-ln3/2, ln3/2), so q_2 = (1/4, 3/4) after x_1 = 0 and (3/4, 1/4) after
    x_1 = 1 -- in both cases the over-drafted token (the one rejections hit) is
    not x_1.  With p_2 = (0.6, 0.4) the residual max(0, p_2 - q_2) is a point
    mass on x_1, and the token emitted at position 2 must follow p_2 after
    either x_1 (the residual built from q_2 at x_2's bias instead would emit
    the other token).  Acceptance at position 2: sum min(p_2, q_2) = 0.65."""
    n = 300_000
    rng = np.random.default_rng(2025)
    p2 = np.array([0.6, 0.4])
    E = np.array([[1.0], [-1.0]])
    W = np.array([[-math.log(3.0) / 2, math.log(3.0) / 2]])
    z = np.zeros((n, 2, 2))
    anchor = np.full(n, -1, dtype=np.int64)  # no bias at position 1
    x1 = rng.integers(0, 2, size=n)
    q2_after = {0: np.array([0.25, 0.75]), 1: np.array([0.75, 0.25])}
    u = rng.random(n)
    x2 = np.where(x1 == 0, (u >= 0.25).astype(np.int64), (u >= 0.75).astype(np.int64))
    tok = np.stack([x1, x2], axis=1)
    rows = np.zeros((n, 3, 2))
    rows[:, 1, :] = np.log(p2)
    out = orc.verify(z, E, W, anchor, tok, 1.0, np.full(n, 2, dtype=np.int64),
                     np.arange(n + 1, dtype=np.int64) * 3, rows.reshape(3 * n, 2),
                     uni24(rng, (n, 2)), uni24(rng, (n,)))
    assert np.all(out["n_acc"] >= 1)  # position 1: p = q, so u < 1 always accepts
    second = out["out_tokens"][:, 1]
    for v in (0, 1):
        sel = x1 == v
        acc = float(np.mean(out["n_acc"][sel] == 2))
        a_true = float(np.minimum(p2, q2_after[v]).sum())
        assert abs(acc - a_true) <= 4 * math.sqrt(a_true * (1 - a_true) / sel.sum())
        counts = np.bincount(second[sel], minlength=2).astype(np.float64)
        assert _chi2_two(counts, p2) < 10.828
        rej = sel & (out["n_acc"] == 1)
        assert np.all(second[rej] == v) and np.all(out["final_kind"][rej] == 1)


def test_residual_with_zero_mass_draws_from_p(orc):
    """A rejection whose residual max(0, p - q) is zero everywhere (the
    reading for this case: draw from p).  Target row (0, -inf): p = (1, 0).
    Draft logits (0, -744): q = (1, e^-744), a subnormal.  The drafted token
    1 has p = 0, so it is rejected even at u = 0; p - q is (0, -e^-744), so
    the residual mass is 0 and the final token is drawn from p: token 0."""
    z = np.array([[[0.0, -744.0]]])
    E, W = np.zeros((2, 1)), np.zeros((1, 2))
    target = np.array([[0.0, -np.inf], [0.0, 0.0]])
    for uf in (0.0, 0.5, 1.0 - 2.0 ** -24):
        out = orc.verify(z, E, W, np.array([-1]), np.array([[1]]), 1.0, np.array([1]),
                         np.array([0, 2]), target, np.array([[0.0]]), np.array([uf]))
        assert out["n_acc"].tolist() == [0]
        assert out["out_tokens"][0].tolist() == [0, -1]
        assert out["final_kind"].tolist() == [2]


def test_final_weights_closed_forms(orc):
    """The distribution the final token is drawn from: the residual at the
    rejected position (with that position's previous token), the bonus row's
    p when all were accepted, p when the residual mass is zero."""
    E = np.array([[1.0], [-1.0]])
    W = np.array([[-math.log(3.0) / 2, math.log(3.0) / 2]])
    z = np.zeros((1, 2, 2))
    tokens = np.array([[0, 1]])
    row = np.log(np.array([0.6, 0.4]))
    # rejected at position 2 (j = 1): q_2 after x_1 = 0 is (1/4, 3/4)
    w = orc.final_weights(z, E, W, np.array([-1]), tokens, 1.0, row, 1, 0, True)
    assert np.allclose(w, [0.35, 0.0], atol=1e-12, rtol=0)
    # rejected at position 1 (j = 0) after anchor 1: q_1 = (3/4, 1/4)
    w = orc.final_weights(z, E, W, np.array([1]), tokens, 1.0, row, 0, 0, True)
    assert np.allclose(w, [0.0, 0.15], atol=1e-12, rtol=0)
    # all accepted: the bonus row's p, at the temperature
    w = orc.final_weights(z, E, W, np.array([-1]), tokens, 0.5, np.array([0.0, math.log(4.0)]),
                          2, 0, False)
    assert np.allclose(w, [1 / 17, 16 / 17], atol=1e-12, rtol=0)
    # zero residual mass: p
    z0 = np.array([[[0.0, -744.0]]])
    w = orc.final_weights(z0, np.zeros((2, 1)), np.zeros((1, 2)), np.array([-1]), np.array([[1]]),
                          1.0, np.array([0.0, -np.inf]), 0, 0, True)
    assert w.tolist() == [1.0, 0.0]


# ------------------------------------------------ capacity (asynchronous) scheduling

@pytest.mark.parametrize("R,G", [(1, 4), (2, 3), (3, 2), (3, 4)])
def test_capacity_schedule_brute_force(orc, R, G):
    """News article, challenge 2: the capacity K is fixed before the step; the
    current candidates fill it in the current order.  For a fixed batch
    B = K the top-(K - R) prefix maximises E over every allocation with
    sum l = K - R (brute force over {0..gamma}^R); K outside [R, R(1+gamma)]
    is clamped."""
    rng = np.random.default_rng(7 * R + G)
    for _ in range(25):
        a = random_survival(rng, R, G)
        fx = np.rint(a * 2.0 ** 40).astype(np.int64)
        for K in range(R - 1, R * (G + 1) + 2):
            out = orc.schedule_capacity(a, K)
            i = max(0, min(R * G, K - R))
            assert out["B"] == R + i and out["i_star"] == i
            assert out["row_off"][-1] == out["B"]
            best, arg = None, []
            for ell in itertools.product(range(G + 1), repeat=R):
                if sum(ell) != i:
                    continue
                s = sum(int(fx[r, :l].sum()) for r, l in enumerate(ell))
                if best is None or s > best:
                    best, arg = s, [ell]
                elif s == best:
                    arg.append(ell)
            assert out["E"] == float(R) + float(best) * 2.0 ** -40
            if len(arg) == 1:
                assert tuple(out["ell"].tolist()) == arg[0]


def test_capacity_from_two_steps_earlier_is_the_global_batch(orc):
    """The capacity predicted from step t-2's survival values is the batch
    the global search picks on them; with those same values now, the
    capacity schedule reproduces the global search's lengths."""
    rng = np.random.default_rng(31)
    for _ in range(20):
        R, G = 3, 4
        a_old = random_survival(rng, R, G)
        sps = rng.uniform(1.0, 100.0, size=R * (G + 1) + 1)
        best, args = brute_force_best(a_old, sps)
        K = orc.schedule(a_old, sps, early_stop=False)["B"]
        assert R + sum(args[0]) == K
        glob = orc.schedule(a_old, sps, early_stop=False)
        cap = orc.schedule_capacity(a_old, K)
        assert cap["ell"].tolist() == glob["ell"].tolist() and cap["E"] == glob["E"]


def test_capacity_tie_order_request_then_position(orc):
    a = np.full((3, 2), 0.5)
    for K, want in [(4, [1, 0, 0]), (5, [2, 0, 0]), (6, [2, 1, 0]), (8, [2, 2, 1])]:
        assert orc.schedule_capacity(a, K)["ell"].tolist() == want


# ---------------------------------------------------------------- RNN head
# News article, innovation 1 (an RNN head keeps a recurrent state); the
# form s_k = tanh(E[x_{k-1}] + s_{k-1} U) is this library's reading.

def test_round_to_state_types(orc):
    """bf16 keeps 8 significant bits, ties to even, in one rounding from the
    double (no detour through fp32): 1/3 -> 171/512; 1 + 2^-8 (a tie) -> 1;
    1 + 3 * 2^-8 (a tie) -> 1 + 2^-6; 1 + 2^-8 + 2^-40 (above the tie by less
    than an fp32 ulp) -> 1 + 2^-7.  fp32: 1/3 -> 11184811 / 2^25."""
    x = np.array([1.0 / 3.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -40,
                  -0.75, 2.0 ** -130 * 1.75])
    want = [171.0 / 512.0, 1.0, 1.0 + 2.0 ** -6, 1.0 + 2.0 ** -7, -0.75, 2.0 ** -133 * 14.0]
    assert orc.round_to(x, "bf16").tolist() == want
    assert orc.round_to(np.array([1.0 / 3.0]), "f32").tolist() == [11184811.0 / 2.0 ** 25]


def test_rnn_head_without_recurrence_is_the_markov_head_on_tanh_rows(orc):
    """U = 0: s_k = round(tanh(E[x_{k-1}])) depends on the previous token
    only, so the RNN draft equals the (pinned) Markov draft on the table
    round(tanh(E)), token for token, for both state types and greedy."""
    rng = np.random.default_rng(77)
    R, G, V, r = 6, 5, 40, 8
    for dtype, T in (("bf16", 1.0), ("f32", 0.7), ("bf16", 0.0)):
        E = orc.round_to(rng.standard_normal((V, r)), dtype)
        W = orc.round_to(rng.standard_normal((r, V)) * 0.5, dtype)
        z = rng.standard_normal((R, G, V)) * 2.0
        anchor = rng.integers(-1, V, size=R)
        anchor[0] = -1
        u = uni24(rng, (R, G))
        tok, ql, qt, S = orc.draft_sample_rnn(z, E, np.zeros((r, r)), W, anchor, u, T, dtype)
        Et = orc.round_to(np.tanh(E), dtype)
        tok2, ql2, qt2 = orc.draft_sample(z, Et, W, anchor, u, T)
        assert np.array_equal(tok, tok2)
        assert np.allclose(ql, ql2, rtol=1e-12, atol=0) and np.allclose(qt, qt2, rtol=1e-12)
        prev = np.concatenate([anchor[:, None], tok[:, :-1]], axis=1)
        want = np.where((prev >= 0)[..., None], Et[np.maximum(prev, 0)], 0.0)
        assert np.array_equal(S, want)


def _rnn_three_token_case(U):
    """V = 3, r = 1, fp32 states, base scores 0 (token 2 at -inf).  The anchor
    is token 2 and the draws are forced to x_0 = 0, x_1 = 1 by the uniforms.
    E is chosen so that the states are s_0 = 0.5, s_1 = 0.6, s_2 = 0.8 when
    the recurrence adds s_{k-1} * U; W gives token 1 the bias s * ln 9 / 0.8,
    so at the third position token 1 gains ln 9 over token 0: the explainer's
    Markov-head experiment (scores 0 / 0, +ln 9: 50% / 50% becomes 90% / 10%)."""
    E = np.array([[math.atanh(0.6) - 0.5 * U], [math.atanh(0.8) - 0.6 * U], [math.atanh(0.5)]])
    E = E.astype(np.float32).astype(np.float64)
    W = np.array([[0.0, math.log(9.0) / 0.8, 0.0]])
    z = np.zeros((1, 3, 3))
    z[..., 2] = -np.inf
    return E, W, z


@pytest.mark.parametrize("u_last,want", [(0.0999, 0), (0.1001, 1)])
def test_rnn_head_explainer_ratio_through_the_recurrence(orc, u_last, want):
    U = 0.7
    E, W, z = _rnn_three_token_case(U)
    u = np.array([[0.0, 0.999999, u_last]])
    tok, ql, qt, S = orc.draft_sample_rnn(z, E, np.array([[U]]), W, np.array([2]), u, 1.0, "f32")
    assert tok[0].tolist() == [0, 1, want]
    assert np.allclose(S[0, :, 0], [0.5, 0.6, 0.8], atol=2e-7, rtol=0)
    assert abs(qt[0, 2] - (0.1 if want == 0 else 0.9)) < 1e-6
    assert abs(ql[0, 2] - math.log(10.0)) < 1e-6  # ln(e^0 + e^{ln 9})
    # without the recurrence term the third state is not 0.8: the 90% is gone
    _, _, qt0, _ = orc.draft_sample_rnn(z, E, np.zeros((1, 1)), W, np.array([2]), u, 1.0, "f32")
    assert abs(qt0[0, 2] - qt[0, 2]) > 1e-2


def test_rnn_head_remembers_the_token_two_back(orc):
    """With U != 0 the third position's distribution depends on x_0 even with
    x_1 fixed; with U = 0 (a one-token memory) it does not."""
    rng = np.random.default_rng(5)
    V, r = 4, 8
    E = orc.round_to(rng.standard_normal((V, r)), "f32")
    W = orc.round_to(rng.standard_normal((r, V)), "f32")
    Um = orc.round_to(rng.standard_normal((r, r)) * 0.6, "f32")
    z = np.zeros((2, 3, V))
    anchor = np.array([3, 3])
    tokens = np.array([[0, 2, 0], [1, 2, 0]])  # same x_1, different x_0
    for U, differ in ((Um, True), (np.zeros((r, r)), False)):
        S = orc.rnn_states(E, U, anchor, tokens, "f32")
        q = orc.draft_distribution_rows(z[:, 2, :], S[:, 2, :], W, 1.0)
        assert (np.max(np.abs(q[0] - q[1])) > 1e-3) == differ
        assert np.array_equal(S[0, 0], S[1, 0])  # same anchor


@pytest.mark.parametrize("s", [math.log(3.0), -math.log(3.0)])
def test_verify_uses_the_rnn_state_of_the_rejected_position(orc, s):
    """gamma = 1, V = 2, r = 1, W = (0, 1): the draft q at the first position
    is built from the state s (not from E, which is zero here): q = (1/4, 3/4)
    for s = ln 3 and (3/4, 1/4) for s = -ln 3.  Drafts drawn from that q and
    verified against p = (0.6, 0.4) must emit p (forum post, lossless proof);
    a residual built from E's zero bias (q = (1/2, 1/2)) would emit
    (0.4, 0.6) for s = ln 3."""
    n = 200_000
    rng = np.random.default_rng(11)
    q = np.array([1.0, math.exp(s)]) / (1.0 + math.exp(s))
    x = (uni24(rng, n) >= q[0]).astype(np.int64)
    p = np.array([0.6, 0.4])
    rows = np.zeros((n, 2, 2))
    rows[:, 0, :] = np.log(p)
    states = np.full((n, 1, 1), s)
    out = orc.verify(np.zeros((n, 1, 2)), np.zeros((2, 1)), np.array([[0.0, 1.0]]),
                     np.full(n, 1, dtype=np.int64), x[:, None], 1.0, np.ones(n, dtype=np.int64),
                     np.arange(n + 1, dtype=np.int64) * 2, rows.reshape(2 * n, 2),
                     uni24(rng, (n, 1)), uni24(rng, (n,)), states=states)
    first = out["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=2).astype(np.float64)
    assert _chi2_two(counts, p) < 10.828
    acc = float(np.mean(out["n_acc"] == 1))
    a_true = float(np.minimum(p, q).sum())
    assert abs(acc - a_true) <= 4 * math.sqrt(a_true * (1 - a_true) / n)
    over = 0 if q[0] > p[0] else 1  # the over-drafted token is the one rejected
    rej = out["n_acc"] == 0
    assert np.all(x[rej] == over) and np.all(first[rej] == 1 - over)


def test_rnn_state_row_vector_times_U(orc):
    """The recurrence multiplies the state as a row vector, like E[x] W:
    pre_j = E[x][j] + sum_i s_i U[i][j].  r = 2: s_0 = (0.5, 0) from the anchor
    row (atanh 0.5, 0); the next row is 0 and U has one entry U[0][1] = c with
    c / 2 = atanh 0.75, so s_1 = (0, 0.75).  U's transpose would give s_1 = 0."""
    c = 2.0 * math.atanh(0.75)
    E = np.array([[0.0, 0.0], [math.atanh(0.5), 0.0]]).astype(np.float32).astype(np.float64)
    U = np.array([[0.0, c], [0.0, 0.0]]).astype(np.float32).astype(np.float64)
    S = orc.rnn_states(E, U, np.array([1]), np.array([[0, 0]]), "f32")
    assert np.allclose(S[0, 0], [0.5, 0.0], atol=1e-7, rtol=0)
    assert np.allclose(S[0, 1], [0.0, 0.75], atol=1e-7, rtol=0)
