"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these retypes the oracle's formulas: each checks the oracle's
*outputs* against a worked example printed on the pages, a closed form, an
exact enumeration, a library routine (scipy's softmax) or a property
(identical-to-greedy), so that a dropped term, a flipped inequality, a
transposed p/q or a wrong temperature fails at least one of them.
"""
import json
import os

import numpy as np
import pytest
from scipy import special, stats

import oracle
import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _f32_softmax(logits32, T=1.0):
    """softmax of the float32 logits the oracle actually receives (scipy)."""
    return special.softmax(np.asarray(logits32, np.float64) / T)


# ---------------------------------------------------------------------------
# P-toy: the printed V=5 example, 200k draws
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def toy():
    g = json.load(open(os.path.join(GOLD, "toy_pq.json")))
    inp = W.make_toy(g["draws"], seed=1000)
    res = oracle.verify_inputs(inp)
    return g, inp, res


def test_toy_accept_rate_is_one_minus_tvd(toy):
    g, inp, res = toy
    p, q = np.array(g["p"]), np.array(g["q"])
    alpha = 1.0 - 0.5 * np.abs(p - q).sum()
    assert alpha == pytest.approx(g["printed_one_minus_tvd"], abs=5e-4)
    n = g["draws"]
    sigma = np.sqrt(alpha * (1 - alpha) / n)
    acc = res["num_accepted"].mean()
    assert abs(acc - alpha) < 4 * sigma, (acc, alpha, sigma)
    assert abs(acc - g["printed_accept_rate"]) < 0.005


def test_toy_output_frequency_matches_p(toy):
    g, inp, res = toy
    p = np.array(g["p"])
    first = res["out_tokens"][:, 0]
    counts = np.bincount(first, minlength=5)
    n = counts.sum()
    chi = stats.chisquare(counts, p * n)
    assert chi.pvalue > 1e-3, chi
    freq = counts / n
    assert np.all(np.abs(freq - np.array(g["printed_observed_freq"])) < 0.005)


def test_toy_exact_intermediates(toy):
    g, inp, res = toy
    p, q = np.array(g["p"]), np.array(g["q"])
    px, qx, rm = oracle.position_probs(inp["target"][:4], inp["draft"][:4], "f32",
                                       inp["tokens"][:4], inp["temperature"][:4], inp["K"][:4])
    # residual mass = sum max(0, p - q) = 0.22, so alpha = sum min(p, q) = 0.78
    assert np.allclose(rm[:, 0], 0.22, atol=1e-6)
    # p(x), q(x) at the proposed token
    assert np.allclose(px[:, 0], p[inp["tokens"][:4, 0]], atol=1e-6)
    assert np.allclose(qx[:, 0], q[inp["tokens"][:4, 0]], atol=1e-6)
    r, code = oracle.final_distribution(inp["target"][0, 0], inp["draft"][0, 0], "f32", 1.0)
    assert code == 1
    assert np.allclose(r, np.array([0.20, 0.0, 0.0, 0.02, 0.0]) / 0.22, atol=1e-6)


# ---------------------------------------------------------------------------
# P-enum: exact enumeration of the output distribution over the uniform grid
# ---------------------------------------------------------------------------
def _first_token(tl, dl, x, u0, u1):
    V = tl.shape[-1]
    tgt = np.stack([tl, tl]).reshape(1, 2, V).astype(np.float32)
    drf = dl.reshape(1, 1, V).astype(np.float32)
    out = oracle.verify(tgt, drf, "f32", np.array([[x]], np.int32),
                        np.array([[u0, u1]], np.float32), np.ones(1, np.float32),
                        np.array([1], np.int32))
    return int(out["num_accepted"][0]), int(out["out_tokens"][0, 0])


def _count_below(pred):
    """Number of k in [0, 2^24) with pred(k * 2^-24) true, pred monotone (true, then false)."""
    lo, hi = 0, 1 << 24
    while lo < hi:
        mid = (lo + hi) // 2
        if pred(mid * 2.0 ** -24):
            lo = mid + 1
        else:
            hi = mid
    return lo


@pytest.mark.parametrize("case", ["v3", "toy"])
def test_enumerated_output_distribution_equals_p(case):
    if case == "v3":
        tl = np.array([0.3, -1.2, 1.1], np.float32)
        dl = np.array([1.4, 0.2, -0.5], np.float32)
    else:
        tl = np.log(W.TOY_P).astype(np.float32)
        dl = np.log(W.TOY_Q).astype(np.float32)
    V = len(tl)
    p = _f32_softmax(tl)
    q = _f32_softmax(dl)
    grid = float(1 << 24)
    A = np.zeros(V)
    for x in range(V):
        A[x] = _count_below(lambda u: _first_token(tl, dl, x, u, 0.5)[0] == 1) / grid
    # closed form of the accept probability per proposal: min(1, p/q)
    assert np.allclose(A, np.minimum(1.0, p / q), atol=2.0 / grid)
    xr = int(np.argmin(A))
    assert A[xr] < 1.0
    u_rej = 1.0 - 2.0 ** -24
    le = [_count_below(lambda u: _first_token(tl, dl, xr, u_rej, u)[1] <= y) for y in range(V)]
    R = np.diff(np.concatenate([[0], le])) / grid
    P = np.array([sum(q[x] * (A[x] * (y == x) + (1 - A[x]) * R[y]) for x in range(V))
                  for y in range(V)])
    assert np.allclose(P, p, atol=2.0 ** -21), (P, p)
    # the oracle's residual obeys q*min(1,p/q) + (sum max(0,p-q)) * r = p
    r, _ = oracle.final_distribution(tl, dl, "f32", 1.0)
    recon = q * np.minimum(1.0, p / q) + np.maximum(p - q, 0).sum() * r
    assert np.allclose(recon, p, atol=1e-15)


# ---------------------------------------------------------------------------
# P-softmax: the final distribution without a draft row is softmax(l / T)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T", [0.7, 1.0, 2.5])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_final_distribution_is_temperature_softmax(T, dtype):
    rng = np.random.default_rng(7)
    l32 = (rng.standard_normal(257) * 3).astype(np.float32)
    stored = W.f32_to_bf16_bits(l32) if dtype == "bf16" else l32
    exact = W.as_f32(stored, dtype)
    r, code = oracle.final_distribution(stored, None, dtype, T)
    assert code == 1
    # the library and the oracle receive T as float32
    assert np.allclose(r, _f32_softmax(exact, float(np.float32(T))), rtol=1e-12, atol=0)


def test_bonus_draw_frequency_is_softmax():
    """All proposals accepted (q == p and u < 1): the extra token comes from row K."""
    rng = np.random.default_rng(3)
    V, B, K = 6, 100_000, 2
    l = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    tgt = np.broadcast_to(l, (B, K + 1, V)).copy()
    drf = tgt[:, :K].copy()
    tok = np.zeros((B, K), np.int32)
    uni = W.uniform_grid(11, 77, B, K + 1)
    out = oracle.verify(tgt, drf, "f32", tok, uni, np.ones(B, np.float32), np.full(B, K, np.int32))
    assert np.all(out["num_accepted"] == K)
    counts = np.bincount(out["out_tokens"][:, K], minlength=V)
    assert stats.chisquare(counts, _f32_softmax(l[K]) * B).pvalue > 1e-3


# ---------------------------------------------------------------------------
# P-geo: i.i.d. alpha gives the truncated geometric law and E[tokens] formula
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("alpha", [0.3, 0.6, 0.9])
@pytest.mark.parametrize("K", [1, 4, 8])
def test_geometric_acceptance_law(alpha, K):
    B = 60_000
    inp = W.make_geometric(alpha, B, K, seed=int(alpha * 100) + K)
    res = oracle.verify_inputs(inp)
    n = res["num_accepted"]
    assert n.min() >= 0 and n.max() <= K
    probs = np.array([alpha ** j * (1 - alpha) for j in range(K)] + [alpha ** K])
    counts = np.bincount(n, minlength=K + 1)
    keep = probs * B > 5
    chi = stats.chisquare(counts[keep], probs[keep] * B * counts[keep].sum() /
                          (probs[keep] * B).sum())
    assert chi.pvalue > 1e-4, (alpha, K, chi)
    tokens = n + 1
    expect = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(tokens.mean() - expect) < 4 * tokens.std() / np.sqrt(B)


# ---------------------------------------------------------------------------
# P-alpha: acceptance of tested positions equals sum min(p, q) = 1 - residual
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,sd,T", [("bf16", 1.0, 1.0), ("f32", 1.5, 0.7)])
def test_expected_accepts_from_position_alpha(dtype, sd, T):
    B, K, V = 20000, 4, 48
    inp = W.make_host(B, K, V, dtype, 2.0, sd, T, seed=99)
    res = oracle.verify_inputs(inp)
    _, _, rm = oracle.position_probs(inp["target"], inp["draft"], dtype, inp["tokens"],
                                     inp["temperature"], inp["K"])
    alpha = 1.0 - rm                                     # [B, K]
    # with x_i ~ q and independent uniforms, position i accepts with probability
    # alpha_i independently: P(nacc >= n) = prod_{i<n} alpha_i
    tail = np.cumprod(alpha, axis=1)                     # P(nacc >= n), n = 1..K
    mean_b = tail.sum(axis=1)
    var_b = (tail * (2 * np.arange(1, K + 1) - 1)).sum(axis=1) - mean_b ** 2
    diff = res["num_accepted"].mean() - mean_b.mean()
    sigma = np.sqrt(var_b.sum()) / B
    assert abs(diff) < 5 * sigma, (diff, sigma, mean_b.mean())


# ---------------------------------------------------------------------------
# P-greedy: speculative greedy decoding equals target-only greedy decoding
# ---------------------------------------------------------------------------
def test_greedy_speculation_identical_to_target_greedy():
    rng = np.random.default_rng(5)
    V, K, steps = 7, 3, 60
    # next-token logit tables (previous token -> logits), coarse values force ties
    table_t = rng.integers(0, 3, size=(V, V)).astype(np.float32)
    table_d = np.where(rng.random((V, V)) < 0.3,
                       rng.integers(0, 3, size=(V, V)), table_t).astype(np.float32)
    seq = [0]
    while len(seq) < steps:
        xs, prev = [], seq[-1]
        for _ in range(K):
            prev = int(np.argmax(table_d[prev]))
            xs.append(prev)
        ctx = [seq[-1]] + xs
        tgt = np.stack([table_t[c] for c in ctx]).reshape(1, K + 1, V)
        drf = np.stack([table_d[c] for c in ctx[:K]]).reshape(1, K, V)
        out = oracle.verify(tgt, drf, "f32", np.array([xs], np.int32),
                            np.zeros((1, K + 1), np.float32), np.zeros(1, np.float32),
                            np.array([K], np.int32))
        n = int(out["num_accepted"][0])
        assert 0 <= n <= K
        seq += xs[:n] + [int(out["out_tokens"][0, n])]
    ref = [0]
    while len(ref) < len(seq):
        ref.append(int(np.argmax(table_t[ref[-1]])))
    assert seq == ref


# ---------------------------------------------------------------------------
# P-edge: special values and degenerate inputs
# ---------------------------------------------------------------------------
def _one(tl, dl, x, u, T=1.0, K=1):
    V = tl.shape[-1]
    tl = np.asarray(tl, np.float32).reshape(1, K + 1, V)
    dl = np.asarray(dl, np.float32).reshape(1, K, V)
    return oracle.verify(tl, dl, "f32", np.array(x, np.int32).reshape(1, K),
                         np.asarray(u, np.float32).reshape(1, K + 1),
                         np.array([T], np.float32), np.array([K], np.int32))


def test_zero_draft_probability_accepts_iff_target_positive():
    ninf = -np.inf
    t = np.array([[0.0, 1.0, -1.0], [0.0, 0.0, 0.0]])
    d = np.array([[0.0, ninf, 0.0]])
    for u in (0.0, 0.5, 1 - 2 ** -24):
        assert _one(t, d, [1], [u, 0.5])["num_accepted"][0] == 1
    t2 = np.array([[0.0, ninf, -1.0], [0.0, 0.0, 0.0]])
    assert _one(t2, d, [1], [0.0, 0.5])["num_accepted"][0] == 0


def test_identical_distributions_always_accept():
    rng = np.random.default_rng(1)
    t = rng.standard_normal((3, 11)).astype(np.float32)
    for u in (0.0, 0.3, 1 - 2 ** -24):
        r = _one(t, t[:2], [4, 9], [u, u, 0.2], K=2)
        assert r["num_accepted"][0] == 2
        assert list(r["out_tokens"][0, :2]) == [4, 9]


def test_uniform_zero_accepts_any_positive_target():
    t = np.array([[5.0, -30.0, 0.0], [0.0, 0.0, 0.0]])
    d = np.array([[-30.0, 5.0, 0.0]])
    assert _one(t, d, [1], [0.0, 0.1])["num_accepted"][0] == 1
    assert _one(t, d, [1], [2 ** -24, 0.1])["num_accepted"][0] == 0


def test_zero_drafts_samples_row_zero():
    tl = np.array([[[0.0, -np.inf, 2.0, 1.0]]], np.float32)
    B = 20_000
    tgt = np.broadcast_to(tl, (B, 1, 4)).copy()
    uni = W.uniform_grid(5, 9, B, 1)
    out = oracle.verify(tgt, np.zeros((B, 0, 4), np.float32), "f32", np.zeros((B, 0), np.int32),
                        uni, np.ones(B, np.float32), np.zeros(B, np.int32))
    assert np.all(out["num_accepted"] == 0)
    c = np.bincount(out["out_tokens"][:, 0], minlength=4)
    assert c[1] == 0                                     # -inf logit is never drawn
    assert stats.chisquare(c[[0, 2, 3]], _f32_softmax(tl[0, 0])[[0, 2, 3]] * B).pvalue > 1e-3


def test_unusable_inputs_give_minus_one():
    t = np.zeros((2, 4), np.float32)
    d = np.zeros((1, 4), np.float32)
    bad_t = t.copy(); bad_t[0, 2] = np.nan
    assert _one(bad_t, d, [0], [0.5, 0.5])["num_accepted"][0] == -1
    pinf = t.copy(); pinf[0, 1] = np.inf
    assert _one(pinf, d, [0], [0.5, 0.5])["num_accepted"][0] == -1
    allninf = t.copy(); allninf[1, :] = -np.inf
    assert _one(allninf, d, [0], [0.5, 0.5])["num_accepted"][0] == -1   # bonus row reached
    for T in (-1.0, np.nan, np.inf, 1e-40):
        assert _one(t, d, [0], [0.5, 0.5], T=T)["num_accepted"][0] == -1
    assert _one(t, d, [4], [0.5, 0.5])["num_accepted"][0] == -1
    assert _one(t, d, [-1], [0.5, 0.5])["num_accepted"][0] == -1
    assert _one(t, d, [0], [1.0, 0.5])["num_accepted"][0] == -1
    assert _one(t, d, [0], [0.5, -0.1])["num_accepted"][0] == -1
    r = _one(t, d, [0], [0.5, 0.5])
    assert r["num_accepted"][0] == 1 and list(r["out_tokens"][0]) [0] == 0


def test_rows_after_first_rejection_are_never_read():
    t = np.array([[5.0, -5.0], [np.nan, 0.0], [0.0, 0.0]], np.float32)
    d = np.array([[-5.0, 5.0], [np.nan, 0.0]], np.float32)
    # x_0 = 1 with p(1) << q(1): rejected for u = 0.9, NaN rows 1 and 2 never reached
    r = _one(t, d, [1, 0], [0.9, 0.9, 0.5], K=2)
    assert r["num_accepted"][0] == 0
    assert r["out_tokens"][0, 0] == 0 and r["out_tokens"][0, 1] == -1


def test_greedy_ties_take_lowest_index_and_ignore_uniforms():
    t = np.array([[1.0, 3.0, 3.0], [2.0, 2.0, 0.0]], np.float32)
    d = np.array([[0.0, 0.0, 9.0]], np.float32)
    r = _one(t, d, [1], [np.nan, np.nan], T=0.0)
    assert r["num_accepted"][0] == 1 and list(r["out_tokens"][0]) == [1, 0]
    r = _one(t, d, [2], [0.0, 0.0], T=0.0)
    assert r["num_accepted"][0] == 0 and list(r["out_tokens"][0]) == [1, -1]


def test_output_layout_and_padding():
    inp = W.make_host(6, np.array([0, 1, 2, 3, 1, 0], np.int32), 37, "bf16", 2.0, 1.0,
                      np.array([1, 0, 1, 0, 0.5, 0], np.float32), seed=4)
    res = oracle.verify_inputs(inp)
    for b in range(6):
        n = res["num_accepted"][b]
        row = res["out_tokens"][b]
        assert 0 <= n <= inp["K"][b]
        assert list(row[:n]) == list(inp["tokens"][b, :n])
        assert 0 <= row[n] < 37
        assert np.all(row[n + 1:] == -1)


# ---------------------------------------------------------------------------
# P-tie: the tie flag marks exactly the decisions whose uniform lies within
# 1e-6 of its threshold.  The pages state the rule as a comparison with
# min(1, p/q) (tech-tldr.com, section 受理判定の数理：修正版棄却サンプリング)
# and note that floating-point precision can change the outcome of such
# comparisons (issoh.co.jp, section 受理・棄却の規則と出力分布が変わらない理由,
# the vLLM caveat); parity exempts flagged sequences, so the flag must be set
# inside the band and clear outside it.  Thresholds here come from scipy's
# softmax of the float32 logits, not from the oracle.
# ---------------------------------------------------------------------------
TIE_T = np.array([[0.3, -1.2, 1.1, 0.2, -0.4],     # tested row 0
                  [0.9, 0.1, -0.6, 0.4, -1.3]], np.float32)   # bonus row 1
TIE_D = np.array([[1.4, 0.2, -0.5, 0.6, -0.9]], np.float32)
INSIDE = (-5e-7, 5e-7)      # within the 1e-6 band
OUTSIDE = (-2e-6, 2e-6)     # clear of it


def _tie_dists():
    p, q = _f32_softmax(TIE_T[0]), _f32_softmax(TIE_D[0])
    resid = np.maximum(p - q, 0.0)
    return p, q, np.cumsum(resid / resid.sum()), np.cumsum(_f32_softmax(TIE_T[1]))


def _near(u, delta):
    """The float32 uniform closest to u + delta (its distance from u stays
    within 0.3 of |delta|: float32 spacing below 1 is at most 6e-8)."""
    v = np.float32(u + delta)
    assert abs(float(v) - u - delta) < 0.3 * abs(delta)
    return v


@pytest.mark.parametrize("x", [3, 0])
def test_tie_flag_at_the_accept_threshold(x):
    p, q, cdf_r, cdf_b = _tie_dists()
    ratio = p[x] / q[x]
    assert 0.05 < ratio < 0.95
    u_final = 0.3     # far from every boundary of both final distributions
    assert min(np.min(np.abs(cdf_r - u_final)), np.min(np.abs(cdf_b - u_final))) > 0.05
    for delta in INSIDE + OUTSIDE:
        r = _one(TIE_T, TIE_D, [x], [_near(ratio, delta), u_final])
        assert r["num_accepted"][0] == (1 if delta < 0 else 0), delta
        assert bool(r["tie"][0]) == (delta in INSIDE), (x, delta)


def test_tie_flag_at_the_residual_cdf_boundaries():
    """Proposal 0 rejected (u = 0.999, far above p/q = 0.41); the residual
    has mass at tokens 2 and 4 only, so its one interior boundary C lies
    between them: just below C the token is 2 (C is its upper end), just
    above it the token is 4 (C is its lower end, token 3 holding no mass)."""
    p, q, cdf_r, _ = _tie_dists()
    C = cdf_r[2]
    assert 0.5 < C < 0.99 and cdf_r[3] == C
    for delta in INSIDE + OUTSIDE:
        r = _one(TIE_T, TIE_D, [0], [0.999, _near(C, delta)])
        assert r["num_accepted"][0] == 0
        assert r["out_tokens"][0, 0] == (2 if delta < 0 else 4), delta
        assert bool(r["tie"][0]) == (delta in INSIDE), delta


@pytest.mark.parametrize("j", [0, 1, 2, 3])
def test_tie_flag_at_the_bonus_cdf_boundaries(j):
    """Proposal 3 accepted (u = 0, far below p/q = 0.83): the bonus token is
    drawn from p of row 1; at each interior boundary C_j the token is j just
    below it and j + 1 just above it."""
    _, _, _, cdf_b = _tie_dists()
    C = cdf_b[j]
    for delta in INSIDE + OUTSIDE:
        r = _one(TIE_T, TIE_D, [3], [0.0, _near(C, delta)])
        assert r["num_accepted"][0] == 1
        assert r["out_tokens"][0, 1] == (j if delta < 0 else j + 1), (j, delta)
        assert bool(r["tie"][0]) == (delta in INSIDE), (j, delta)


def test_greedy_decisions_are_never_flagged():
    p, q, _, cdf_b = _tie_dists()
    for u in (p[3] / q[3], cdf_b[1], 0.0):
        r = _one(TIE_T, TIE_D, [2], [np.float32(u), np.float32(u)], T=0.0)
        assert not r["tie"][0]


def test_ties_are_rare_on_random_batches():
    """A uniform lands in a 2e-6-wide band around a threshold with
    probability 2e-6 per decision: a random batch of 20,000 sequences (about
    three decisions each) should flag well under 1e-4 of them."""
    B = 20000
    inp = W.make_host(B, 4, 48, "f32", 2.0, 1.0, 1.0, seed=2718)
    res = oracle.verify_inputs(inp)
    assert int(res["tie"].sum()) <= max(2, int(1e-4 * B))
