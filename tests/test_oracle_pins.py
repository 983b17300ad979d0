"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each test ties one oracle step to something other than the oracle itself: a
hand-worked example, a closed form printed on the pages, a brute-force enumeration,
a library routine, a Monte Carlo estimate of a probability the pages state, or an
invariant. Sources: "MagicPIG: LSH Sampling for Efficient LLM Generation"
(arXiv 2410.16179v2) and the authors' responses to reviews (paperhub page).
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------------
# hand-worked example (tests/golden)
# ----------------------------------------------------------------------------------

def test_golden_tiny_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "tiny_2d_worked_example.json")))
    keys = np.array(g["keys"], float)
    vals = np.array(g["values"], float)
    W = np.array(g["W"], float)
    q = np.array(g["q"], float)
    K, L, s, w, n0 = g["K"], g["L"], g["n_sink"], g["window"], g["n_prefill"]
    ex = g["expected"]
    tables = O.HeadTables(keys, W, K, L, s, n0)
    np.testing.assert_allclose(tables.center, ex["center"], atol=1e-15)
    np.testing.assert_array_equal(tables.codes, ex["key_codes"])
    r = O.decode_head(q, keys, vals, tables, n0, w)
    np.testing.assert_array_equal(r["q_code"], ex["q_code"])
    np.testing.assert_array_equal(r["S"], ex["S"])
    np.testing.assert_array_equal(r["T"], ex["T"])
    # arccos is ill-conditioned at cos = 1: a rounding of cos by 1 ulp moves p by ~1e-8
    np.testing.assert_allclose(r["p"], [float(Fraction(x)) for x in ex["p"]], atol=1e-7)
    np.testing.assert_allclose(r["u"], [float(Fraction(x)) for x in ex["u"]], rtol=1e-12)
    env = {"exp": math.exp, "sqrt": math.sqrt}
    wts = {int(i): eval(e, env) for i, e in ex["weights"].items()}
    tot = sum(wts.values())
    want = np.array([sum(wt * vals[i][0] for i, wt in wts.items()) / tot, 1.0])
    np.testing.assert_allclose(r["out"], want, rtol=1e-13)


# ----------------------------------------------------------------------------------
# a1 centering
# ----------------------------------------------------------------------------------

def test_center_is_known_mean_of_non_sink_prefill():
    rng = np.random.default_rng(5)
    d, s, n0 = 6, 4, 40
    a = rng.normal(size=d)
    half = rng.normal(size=((n0 - s) // 2, d))
    z = np.concatenate([half, -half])            # sums to zero over [s, n0)
    keys = np.concatenate([1e6 * rng.normal(size=(s, d)),   # sinks: must not enter the mean
                           a + z,
                           1e6 * rng.normal(size=(5, d))])  # appended later: must not enter
    np.testing.assert_allclose(O.center_of_keys(keys, s, n0), a, atol=1e-9)


# ----------------------------------------------------------------------------------
# a2 / a5 SimHash codes
# ----------------------------------------------------------------------------------

def test_codes_one_hot_projections_by_hand():
    # columns: e0, e1 | e2, e3 | -e0, e2  (K = 2, L = 3)
    W = np.zeros((4, 6))
    W[0, 0] = W[1, 1] = W[2, 2] = W[3, 3] = W[2, 5] = 1.0
    W[0, 4] = -1.0
    x = np.array([[1.0, -2.0, 3.0, -4.0],     # y = 1,-2 | 3,-4 | -1, 3
                  [-1.0, 2.0, -3.0, 4.0]])    # y = -1,2 | -3,4 | 1, -3
    codes = O.simhash_codes(x, W, K=2, L=3)
    # bit b of table t is column t*K + b
    np.testing.assert_array_equal(codes, [[0b01, 0b01, 0b10], [0b10, 0b10, 0b01]])


def test_codes_negation_is_complement_and_scale_invariant():
    rng = np.random.default_rng(1)
    d, K, L = 16, 5, 9
    W = rng.normal(size=(d, K * L))
    x = rng.normal(size=(50, d))
    c = rng.normal(size=d)
    codes = O.simhash_codes(x, W, K, L, center=c)
    mirrored = 2 * c - x                          # x - c  ->  -(x - c)
    np.testing.assert_array_equal(O.simhash_codes(mirrored, W, K, L, center=c),
                                  (2 ** K - 1) ^ codes)
    scaled = c + 7.5 * (x - c)
    np.testing.assert_array_equal(O.simhash_codes(scaled, W, K, L, center=c), codes)


@pytest.mark.parametrize("theta_deg,K", [(30, 3), (75, 2), (120, 1)])
def test_per_table_collision_rate_monte_carlo(theta_deg, K):
    """P[code_t(x) = code_t(y)] = (1 - theta/pi)^K over Gaussian hyperplanes
    (MagicPIG §2.2 SimHash). Each of L = 40000 tables is an independent draw."""
    rng = np.random.default_rng(theta_deg)
    d, L = 12, 40000
    th = math.radians(theta_deg)
    e0, e1 = np.eye(d)[0], np.eye(d)[1]
    x = np.array([e0, math.cos(th) * e0 + math.sin(th) * e1])
    W = rng.normal(size=(d, K * L))
    codes = O.simhash_codes(x, W, K, L)
    rate = np.mean(codes[0] == codes[1])
    want = (1 - th / math.pi) ** K
    sigma = math.sqrt(want * (1 - want) / L)
    assert abs(rate - want) < 4 * sigma, (rate, want, sigma)


def test_near_tie_mask_flags_small_projections():
    W = np.array([[1.0, 1.0], [0.0, 1e-7]])
    x = np.array([[1.0, -1.0]])     # y = 1, 1 - 1e-7
    x2 = np.array([[1e-7, 1.0]])    # y = 1e-7, ~1e-7: both tiny relative to |x||w|
    assert not O.near_ties(x, W).any()
    assert O.near_ties(x2, W).all()


def test_zero_projections_are_near_ties():
    """SimHash keeps the sign of a projection ([MagicPIG] §2.2); a projection that is
    exactly zero has none, so it is a near tie and its bit is never compared: a key
    equal to the center, a zero query, and a column orthogonal to the key."""
    W = np.array([[1.0, 0.0, 2.0], [0.0, 1.0, -1.0]])
    c = np.array([0.5, -0.25])
    assert O.near_ties(c[None, :], W, center=c).all()
    assert O.near_ties(np.zeros((1, 2)), W).all()
    np.testing.assert_array_equal(O.near_ties(np.array([[1.0, 2.0]]), W), [[False, False, True]])


def test_near_tie_band_is_relative_to_both_norms():
    """A near tie is a projection below 1e-5 of |x - c| |w_j|, so whether a sign is a
    near tie depends only on the angle between x - c and w_j: rescaling x - c or any
    column of W leaves the mask unchanged. Columns are built at chosen cosines with
    x - c: +-0.5e-5 (ties), +-2e-5 and 0.3 (not ties)."""
    rng = np.random.default_rng(12)
    d = 8
    c = rng.normal(size=d)
    xc = rng.normal(size=d)
    xh = xc / np.linalg.norm(xc)
    e = rng.normal(size=d)
    e -= (e @ xh) * xh
    e /= np.linalg.norm(e)
    cosines = [0.5e-5, -0.5e-5, 2e-5, -2e-5, 0.3]
    W = np.stack([cs * xh + math.sqrt(1 - cs * cs) * e for cs in cosines], axis=1)
    want = np.array([[True, True, False, False, False]])
    for sx in [1.0, 1e-3, 1e4]:
        for cols in [np.ones(5), np.array([1e-3, 1e4, 7.0, 0.02, 1e3])]:
            got = O.near_ties((c + sx * xc)[None, :], W * cols[None, :], center=c)
            np.testing.assert_array_equal(got, want, err_msg=f"x scale {sx}, column scales {cols}")


# ----------------------------------------------------------------------------------
# a7 collision / inclusion probability
# ----------------------------------------------------------------------------------

def test_collision_probability_special_angles():
    q = np.array([2.0, 1.0])
    kc = np.array([[4.0, 2.0], [-2.0, -1.0], [-1.0, 2.0], [1.0, 3.0], [0.0, 0.0]])
    # arccos is ill-conditioned at cos = +-1 (1 ulp of cos moves p by ~1e-8)
    np.testing.assert_allclose(O.collision_probability(q, kc), [1.0, 0.0, 0.5, 0.75, 0.5],
                               atol=1e-7)


@pytest.mark.parametrize("L,T", [(3, 2), (6, 2), (10, 2), (10, 1), (8, 3)])
def test_inclusion_probability_enumerates_table_patterns(L, T):
    """Brute force: sum over all 2^L patterns of per-table collisions (each table
    collides independently with x = p^K) with at least T collisions."""
    K = 2
    for p in [0.05, 0.3, 0.5, 0.71, 0.93, 1.0]:
        x = p ** K
        want = 0.0
        for pat in itertools.product([0, 1], repeat=L):
            h = sum(pat)
            if h >= T:
                want += x ** h * (1 - x) ** (L - h)
        got = O.inclusion_probability(np.array([p]), K, L, threshold=T)[0]
        assert got == pytest.approx(want, rel=1e-12, abs=1e-300)


def test_inclusion_probability_matches_binomial_tail_and_eq10():
    K, L = 10, 150
    p = np.linspace(0.02, 1.0, 200)
    u = O.inclusion_probability(p, K, L)
    x = p ** K
    np.testing.assert_allclose(u, stats.binom.sf(1, L, x), rtol=1e-9)
    # the printed closed form (Eq. 10) where it does not cancel
    big = L * x >= 1.0
    eq10 = 1 - (1 - x) ** L - L * x * (1 - x) ** (L - 1)
    np.testing.assert_allclose(u[big], eq10[big], rtol=1e-12)
    # T = 1 is the classic LSH retrieval probability 1 - (1 - p^K)^L (MagicPIG §2.2)
    u1 = O.inclusion_probability(p, K, L, threshold=1)
    np.testing.assert_allclose(u1, -np.expm1(L * np.log1p(-np.minimum(x, 1 - 1e-16))), rtol=1e-9)
    assert np.all(np.diff(u) >= 0)


def test_expected_budget_is_the_binomial_tail_at_half():
    # closed form of the author responses (0.5^K per table) is P[Bin(L, 0.5^K) >= 2]
    for K, L in [(8, 75), (9, 120), (10, 150)]:
        x = 0.5 ** K
        assert O.expected_budget(K, L) == pytest.approx(stats.binom.sf(1, L, x), rel=1e-12)


# ----------------------------------------------------------------------------------
# a6 sampled set: region and statistics
# ----------------------------------------------------------------------------------

def test_region_and_static_tokens():
    assert O.lsh_region(10, 2, 3) == (2, 7)
    np.testing.assert_array_equal(O.exact_tokens(10, 2, 3), [0, 1, 7, 8, 9])
    np.testing.assert_array_equal(O.sampled_set(np.full(10, 5), 10, 2, 3), [2, 3, 4, 5, 6])
    assert O.lsh_region(3, 4, 2) == (3, 3)
    np.testing.assert_array_equal(O.exact_tokens(3, 4, 2), [0, 1, 2])
    assert O.lsh_region(6, 4, 2) == (4, 4)
    np.testing.assert_array_equal(O.exact_tokens(6, 4, 2), [0, 1, 2, 3, 4, 5])


def test_budget_at_half_collision_probability_equals_closed_form():
    """Keys whose centered vectors are orthogonal to q have p = 1/2 exactly; the
    expected sampled fraction is then the pages' closed form
    1 - (1-0.5^K)^L - L 0.5^K (1-0.5^K)^(L-1)."""
    rng = np.random.default_rng(11)
    d, n, K, L, s, w = 12, 400, 3, 8, 4, 8
    q = np.eye(d)[0] * 1.7
    keys = np.concatenate([np.zeros((n, 1)), rng.normal(size=(n, d - 1))], axis=1)
    fr = []
    for _ in range(300):
        W = rng.normal(size=(d, K * L))
        t = O.HeadTables(keys, W, K, L, s, n)
        r = O.decode_head(q, keys, keys, t, n, w)
        fr.append(len(r["S"]) / (n - s - w))
        np.testing.assert_allclose(r["p"], 0.5, atol=1e-12)
    fr = np.array(fr)
    want = O.expected_budget(K, L)
    assert abs(fr.mean() - want) < 4 * fr.std(ddof=1) / math.sqrt(len(fr)), (fr.mean(), want)


def _cone(rng, d, n):
    mu = rng.normal(size=d)
    mu /= np.linalg.norm(mu)
    keys = 3 * mu + rng.normal(size=(n, d))
    keys[0] = -6 * mu
    q = -2 * mu + rng.normal(size=d)
    return keys, q


def test_expected_sample_size_equals_sum_of_inclusion_probabilities():
    """E_W |S| = sum_i u_i: u is the true inclusion probability of the sampling rule."""
    rng = np.random.default_rng(3)
    d, n, K, L, s, w = 10, 300, 3, 10, 4, 16
    keys, q = _cone(rng, d, n)
    sizes, usum = [], None
    for _ in range(400):
        W = rng.normal(size=(d, K * L))
        t = O.HeadTables(keys, W, K, L, s, n)
        r = O.decode_head(q, keys, keys, t, n, w)
        sizes.append(len(r["S"]))
        if usum is None:
            lo, hi = O.lsh_region(n, s, w)
            p = O.collision_probability(q, keys[lo:hi] - t.center)
            usum = O.inclusion_probability(p, K, L).sum()
    sizes = np.array(sizes, float)
    assert abs(sizes.mean() - usum) < 4 * sizes.std(ddof=1) / math.sqrt(len(sizes)), (sizes.mean(), usum)


def test_snis_numerator_and_denominator_are_unbiased():
    """Averaged over hash draws, sum_{S∪T} w~/u v and sum_{S∪T} w~/u are unbiased for
    the full sums (Eq. 9 with P[i in S] = u_i), so their ratio tends to Eq. 1."""
    rng = np.random.default_rng(7)
    d, n, K, L, s, w = 8, 200, 2, 12, 2, 6
    keys, q = _cone(rng, d, n)
    vals = rng.normal(size=(n, d))
    exact = O.exact_attention(q, keys, vals)
    ref = float((keys @ q).max() / math.sqrt(d))
    nums, dens = [], []
    for _ in range(1500):
        W = rng.normal(size=(d, K * L))
        t = O.HeadTables(keys, W, K, L, s, n)
        r = O.decode_head(q, keys, vals, t, n, w)
        num, den = O.snis_sums(q, keys, vals, r["S"], r["u"], r["T"], ref)
        nums.append(num)
        dens.append(den)
    nums, dens = np.array(nums), np.array(dens)
    full_logit = keys @ q / math.sqrt(d) - ref
    np.testing.assert_allclose(dens.mean(), np.exp(full_logit).sum(),
                               rtol=4 * dens.std(ddof=1) / math.sqrt(len(dens)) / dens.mean())
    ratio = nums.mean(0) / dens.mean()
    resid = nums - ratio[None, :] * dens[:, None]
    se = resid.std(axis=0, ddof=1) / math.sqrt(len(dens)) / dens.mean()
    assert np.all(np.abs(ratio - exact) < 4.5 * se + 1e-9), (ratio, exact, se)


# ----------------------------------------------------------------------------------
# a7 - a9 special cases that reduce to exact attention (Eq. 1)
# ----------------------------------------------------------------------------------

def test_every_key_sampled_when_K_is_zero_gives_exact_attention():
    rng = np.random.default_rng(2)
    d, n, L, s, w = 16, 97, 5, 4, 8
    keys, q = _cone(rng, d, n)
    vals = rng.normal(size=(n, d))
    t = O.HeadTables(keys, np.zeros((d, 0)), 0, L, s, n)
    r = O.decode_head(q, keys, vals, t, n, w)
    np.testing.assert_array_equal(r["S"], np.arange(s, n - w))
    np.testing.assert_allclose(r["u"], 1.0)
    want = softmax(keys @ q / math.sqrt(d)) @ vals
    np.testing.assert_allclose(r["out"], want, rtol=1e-12)
    np.testing.assert_allclose(O.exact_attention(q, keys, vals), want, rtol=1e-12)


def test_short_sequence_is_all_static_and_exact():
    rng = np.random.default_rng(4)
    d, n, K, L, s, w = 8, 50, 4, 6, 4, 64
    keys, q = _cone(rng, d, n)
    vals = rng.normal(size=(n, d))
    t = O.HeadTables(keys, rng.normal(size=(d, K * L)), K, L, s, n)
    r = O.decode_head(q, keys, vals, t, n, w)
    assert len(r["S"]) == 0 and len(r["T"]) == n
    np.testing.assert_allclose(r["out"], softmax(keys @ q / math.sqrt(d)) @ vals, rtol=1e-12)


def test_constant_keys_reduce_to_a_weighted_mean():
    """Degenerate head: every key equals the center, so every projection is zero (code 0
    in every table, all near ties), cos(q, k - c) is taken as 0 (p = 1/2) and all logits
    are equal. The sampled set is the whole region or nothing, depending on whether the
    query's code is 0 in at least two tables, and the output is the mean of the values
    with weight 1/u on the sampled tokens and 1 on the static ones."""
    rng = np.random.default_rng(21)
    d, n, K, L, s, w = 8, 120, 2, 6, 4, 16
    a = np.round(16 * rng.normal(size=d)) / 16   # few mantissa bits: the mean is exactly a
    keys = np.tile(a, (n, 1))
    vals = rng.normal(size=(n, d))
    W = rng.normal(size=(d, K * L))
    t = O.HeadTables(keys, W, K, L, s, n)
    assert np.all(t.codes == 0) and t.ties.all()
    u_half = O.inclusion_probability(np.array([0.5]), K, L)[0]
    seen = set()
    for _ in range(40):
        q = rng.normal(size=d)
        r = O.decode_head(q, keys, vals, t, n, w)
        region = np.arange(s, n - w)
        zero_tables = int(np.sum(r["q_code"] == 0))
        S = region if zero_tables >= 2 else region[:0]
        np.testing.assert_array_equal(r["S"], S)
        np.testing.assert_allclose(r["p"], 0.5)
        wts = np.ones(n)
        wts[S] = 1.0 / u_half
        wts[np.setdiff1d(region, S)] = 0.0
        np.testing.assert_allclose(r["out"], wts @ vals / wts.sum(), rtol=1e-12)
        seen.add(len(S) > 0)
    assert seen == {True, False}


def test_translation_of_all_keys_changes_nothing():
    """Softmax is translation invariant and keys are centered (MagicPIG §4.3)."""
    rng = np.random.default_rng(9)
    d, n, K, L, s, w = 16, 600, 4, 20, 4, 32
    keys, q = _cone(rng, d, n)
    vals = rng.normal(size=(n, d))
    W = rng.normal(size=(d, K * L))
    shift = 5 * rng.normal(size=d)
    a = O.decode_head(q, keys, vals, O.HeadTables(keys, W, K, L, s, n), n, w)
    b = O.decode_head(q, keys + shift, vals, O.HeadTables(keys + shift, W, K, L, s, n), n, w)
    np.testing.assert_array_equal(a["S"], b["S"])
    assert len(a["S"]) > 0
    np.testing.assert_allclose(a["u"], b["u"], rtol=1e-10)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-9)


def test_translation_invariance_covers_appended_tokens():
    """Tokens appended after the build are hashed with the prefill's center, so a shift
    of every key (prefill and appended) leaves all codes, the sampled set and the output
    of a decode step past the prefill unchanged (MagicPIG §4.3 "Data pre-processing")."""
    rng = np.random.default_rng(13)
    d, n0, n, K, L, s, w = 16, 500, 560, 4, 20, 4, 32
    keys, q = _cone(rng, d, n)
    vals = rng.normal(size=(n, d))
    W = rng.normal(size=(d, K * L))
    shift = 5 * rng.normal(size=d)
    ta = O.HeadTables(keys, W, K, L, s, n0, n_total=n)
    tb = O.HeadTables(keys + shift, W, K, L, s, n0, n_total=n)
    np.testing.assert_allclose(tb.center, ta.center + shift, rtol=1e-12)
    np.testing.assert_array_equal(ta.codes, tb.codes)
    a = O.decode_head(q, keys, vals, ta, n, w)
    b = O.decode_head(q, keys + shift, vals, tb, n, w)
    np.testing.assert_array_equal(a["S"], b["S"])
    assert np.any(a["S"] >= n0)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-9)


def test_centering_off_hashes_raw_keys_and_is_not_translation_invariant():
    """The centering ablation (c = 0): codes are the SimHash of the raw keys, so shifting
    every key by a vector changes them, while with centering the shift cancels
    (§4.3 "Data pre-processing": the center removes the common component)."""
    rng = np.random.default_rng(11)
    d, K, L, s, n0 = 16, 4, 6, 2, 300
    keys = rng.standard_normal((n0, d))
    W = rng.standard_normal((d, K * L))
    shift = 5.0 * rng.standard_normal(d)
    off = O.HeadTables(keys, W, K, L, s, n0, centering=False)
    assert np.all(off.center == 0)
    np.testing.assert_array_equal(off.codes, O.simhash_codes(keys, W, K, L))
    on_a = O.HeadTables(keys, W, K, L, s, n0)
    on_b = O.HeadTables(keys + shift, W, K, L, s, n0)
    np.testing.assert_array_equal(on_a.codes, on_b.codes)
    off_b = O.HeadTables(keys + shift, W, K, L, s, n0, centering=False)
    assert np.any(off_b.codes != off.codes)


# ----------------------------------------------------------------------------------
# invariances of the whole step
# ----------------------------------------------------------------------------------

def test_tables_are_exchangeable_and_hyperplanes_scale_free():
    """Relabelling the L tables (moving whole K-column blocks of W) or scaling any
    hyperplane by a positive factor changes no sign, so S, u and the output stay the
    same (SimHash depends on the hyperplanes' directions only, MagicPIG §2.2)."""
    rng = np.random.default_rng(23)
    d, n, K, L, s, w = 12, 400, 3, 9, 4, 16
    keys, q = _cone(rng, d, n)
    vals = rng.normal(size=(n, d))
    W = rng.normal(size=(d, K * L))
    base = O.decode_head(q, keys, vals, O.HeadTables(keys, W, K, L, s, n), n, w)
    assert len(base["S"]) > 0
    perm = rng.permutation(L)
    Wp = W.reshape(d, L, K)[:, perm, :].reshape(d, K * L)
    Ws = W * rng.uniform(0.01, 100.0, size=K * L)[None, :]
    for W2 in (Wp, Ws):
        r = O.decode_head(q, keys, vals, O.HeadTables(keys, W2, K, L, s, n), n, w)
        np.testing.assert_array_equal(r["S"], base["S"])
        np.testing.assert_allclose(r["u"], base["u"], rtol=1e-12)
        np.testing.assert_allclose(r["out"], base["out"], rtol=1e-12)


def test_decode_reads_only_the_visible_tokens():
    """A decode step over n tokens does not depend on keys or values at positions >= n."""
    rng = np.random.default_rng(29)
    d, n0, n, K, L, s, w = 12, 300, 340, 3, 10, 4, 16
    keys, q = _cone(rng, d, n + 20)
    vals = rng.normal(size=(n + 20, d))
    W = rng.normal(size=(d, K * L))
    t = O.HeadTables(keys, W, K, L, s, n0, n_total=n + 20)
    a = O.decode_head(q, keys, vals, t, n, w)
    keys2, vals2 = keys.copy(), vals.copy()
    keys2[n:] = 100.0 * rng.normal(size=(20, d))
    vals2[n:] = 100.0 * rng.normal(size=(20, d))
    t2 = O.HeadTables(keys2, W, K, L, s, n0, n_total=n + 20)
    b = O.decode_head(q, keys2, vals2, t2, n, w)
    np.testing.assert_array_equal(a["S"], b["S"])
    np.testing.assert_array_equal(a["out"], b["out"])


def test_inclusion_probability_orders_with_K_L_and_T():
    """More tables raise u, more bits per table and a higher threshold lower it
    (P[Bin(L, p^K) >= T] is increasing in L and p, decreasing in K and T)."""
    p = np.linspace(0.05, 0.95, 19)
    u = lambda K, L, T: O.inclusion_probability(p, K, L, threshold=T)  # noqa: E731
    assert np.all(u(4, 20, 2) < u(4, 21, 2))
    assert np.all(u(5, 20, 2) < u(4, 20, 2))
    assert np.all(u(4, 20, 3) < u(4, 20, 2))
    assert np.all(np.diff(u(6, 50, 3)) > 0)


# ----------------------------------------------------------------------------------
# brute force on tiny inputs: the step written with loops and the math module
# ----------------------------------------------------------------------------------

def _brute_force_step(q, keys, vals, W, K, L, s, w, n0, n, T=2):
    """One decode step from the definitions, element by element, no numpy: the mean
    key over [s, n0); bit b of table t = [<x - c, W[:, tK + b]> > 0]; sampled iff
    >= T tables agree with the query; weights e^{q.k/sqrt d} / u on S, e^{q.k/sqrt d}
    on the sinks and the window; u = sum_{j >= T} C(L, j) x^j (1 - x)^(L - j)."""
    d = len(q)
    c = [sum(keys[i][j] for i in range(s, n0)) / (n0 - s) for j in range(d)]

    def code(x, center):
        out = []
        for t in range(L):
            v = 0
            for b in range(K):
                y = sum((x[j] - center[j]) * W[j][t * K + b] for j in range(d))
                v |= (1 if y > 0 else 0) << b
            out.append(v)
        return out

    qc = code(q, [0.0] * d)
    lo, hi = min(s, n), max(min(s, n), n - w)
    num, den = [0.0] * d, 0.0
    M = max(sum(q[j] * keys[i][j] for j in range(d)) / math.sqrt(d) for i in range(n))
    S = []
    for i in range(n):
        z = sum(q[j] * keys[i][j] for j in range(d)) / math.sqrt(d)
        wt = math.exp(z - M)
        if lo <= i < hi:
            kc = code(keys[i], c)
            if sum(1 for t in range(L) if kc[t] == qc[t]) < T:
                continue
            S.append(i)
            kd = [keys[i][j] - c[j] for j in range(d)]
            nq = math.sqrt(sum(v * v for v in q))
            nk = math.sqrt(sum(v * v for v in kd))
            cs = sum(q[j] * kd[j] for j in range(d)) / (nq * nk) if nq * nk > 0 else 0.0
            p = 1.0 - math.acos(max(-1.0, min(1.0, cs))) / math.pi
            x = p ** K
            u = sum(math.comb(L, j) * x ** j * (1 - x) ** (L - j) for j in range(T, L + 1))
            wt /= u
        den += wt
        for j in range(d):
            num[j] += wt * vals[i][j]
    return S, [v / den for v in num]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_whole_step_equals_brute_force_on_tiny_inputs(seed):
    rng = np.random.default_rng(100 + seed)
    d, n0, n, K, L, s, w = 5, 37, 41, 2, 4, 2, 5
    keys, q = _cone(rng, d, n)
    vals = rng.normal(size=(n, d))
    W = rng.normal(size=(d, K * L))
    t = O.HeadTables(keys, W, K, L, s, n0, n_total=n)
    r = O.decode_head(q, keys, vals, t, n, w)
    S, out = _brute_force_step(q.tolist(), keys.tolist(), vals.tolist(), W.tolist(), K, L, s, w, n0, n)
    assert len(S) > 0
    np.testing.assert_array_equal(r["S"], S)
    np.testing.assert_allclose(r["out"], out, rtol=1e-12)



# ----------------------------------------------------------------------------------
# the centered-query reading (query hashed as q - c)
# ----------------------------------------------------------------------------------

def test_centered_query_sampling_rule_matches_its_inclusion_probability():
    """With q - c hashed, each key is sampled with probability u_i computed from
    p = 1 - theta(q - c, k - c)/pi, the pair of vectors whose signs are compared: the
    frequency of every key over independent hash draws agrees with that u_i (and, for
    the keys where the readings differ most, not with the u of the uncentered query)."""
    rng = np.random.default_rng(31)
    d, n, K, L, s, w = 10, 300, 3, 10, 4, 16
    keys, q = _cone(rng, d, n)
    lo, hi = O.lsh_region(n, s, w)
    draws = 600
    hits = np.zeros(hi - lo)
    center = None
    for _ in range(draws):
        W = rng.normal(size=(d, K * L))
        t = O.HeadTables(keys, W, K, L, s, n)
        center = t.center
        r = O.decode_head(q, keys, keys, t, n, w, center_query=True)
        hits[r["S"] - lo] += 1
    freq = hits / draws
    u_cq = O.inclusion_probability(O.collision_probability(q - center, keys[lo:hi] - center), K, L)
    u_raw = O.inclusion_probability(O.collision_probability(q, keys[lo:hi] - center), K, L)
    se = np.sqrt(np.maximum(u_cq * (1 - u_cq), 1e-4) / draws)
    assert np.all(np.abs(freq - u_cq) < 5 * se), np.max(np.abs(freq - u_cq) / se)
    far = np.argsort(-np.abs(u_cq - u_raw))[:5]
    assert np.all(np.abs(freq[far] - u_raw[far]) > 5 * se[far])


def test_centered_query_sets_are_invariant_to_a_common_shift():
    """Shifting every key and the query by one vector leaves q - c and k - c, hence the
    codes, the sampled set and u, unchanged in the centered-query reading (but not the
    logits, which use the raw vectors)."""
    rng = np.random.default_rng(37)
    d, n, K, L, s, w = 16, 600, 4, 20, 4, 32
    keys, q = _cone(rng, d, n)
    vals = rng.normal(size=(n, d))
    W = rng.normal(size=(d, K * L))
    shift = 5 * rng.normal(size=d)
    a = O.decode_head(q, keys, vals, O.HeadTables(keys, W, K, L, s, n), n, w, center_query=True)
    b = O.decode_head(q + shift, keys + shift, vals, O.HeadTables(keys + shift, W, K, L, s, n), n, w,
                      center_query=True)
    np.testing.assert_array_equal(a["q_code"], b["q_code"])
    np.testing.assert_array_equal(a["S"], b["S"])
    assert len(a["S"]) > 0
    np.testing.assert_allclose(a["u"], b["u"], rtol=1e-10)


def test_each_key_is_sampled_with_its_inclusion_probability():
    """Per key, not only in the sum: over independent hash draws every key of the LSH
    region is sampled with frequency u_i (the uncentered query's p with the centered
    key), and the keys where the two query readings differ most reject the other one."""
    rng = np.random.default_rng(41)
    d, n, K, L, s, w = 10, 300, 3, 10, 4, 16
    keys, q = _cone(rng, d, n)
    lo, hi = O.lsh_region(n, s, w)
    draws = 600
    hits = np.zeros(hi - lo)
    center = None
    for _ in range(draws):
        W = rng.normal(size=(d, K * L))
        t = O.HeadTables(keys, W, K, L, s, n)
        center = t.center
        r = O.decode_head(q, keys, keys, t, n, w)
        hits[r["S"] - lo] += 1
    freq = hits / draws
    u = O.inclusion_probability(O.collision_probability(q, keys[lo:hi] - center), K, L)
    u_other = O.inclusion_probability(O.collision_probability(q - center, keys[lo:hi] - center), K, L)
    se = np.sqrt(np.maximum(u * (1 - u), 1e-4) / draws)
    assert np.all(np.abs(freq - u) < 5 * se), np.max(np.abs(freq - u) / se)
    far = np.argsort(-np.abs(u - u_other))[:5]
    assert np.all(np.abs(freq[far] - u_other[far]) > 5 * se[far])
