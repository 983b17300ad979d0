"""Plain CPU oracle of LSH-sampled decode attention (MagicPIG), float64.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's CPU
baseline may import this module. The product path never calls it, and it shares no
code with the CUDA library: no kernels, headers, helpers or tables.

Every function restates one step of "MagicPIG: LSH Sampling for Efficient LLM
Generation" (arXiv 2410.16179v2, cited below as [MagicPIG]) in numpy float64, slowly
and in the pages' order. Steps the pages leave open take the plainest reading; each
such reading is marked READING in the docstring.

Notation: d head dim, n tokens, K bits per table, L tables, hyperplane column
j = t*K + b for table t and bit b, sinks s, window w.
"""
from __future__ import annotations

import math

import numpy as np

NEAR_TIE_REL = 1e-5   # a projection with |y| <= 1e-5 * ||x|| * ||w_j|| is a near tie
THRESHOLD = 2         # [MagicPIG] §4.3 "Hash function selection": at least two tables


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ----------------------------------------------------------------------------------
# a1: centering
# ----------------------------------------------------------------------------------

def center_of_keys(keys, n_sink: int, n_prefill: int) -> np.ndarray:
    """Mean key used for centering, [MagicPIG] §4.3 "Data pre-processing".

    READING: the mean runs over the non-sink prefill tokens [n_sink, n_prefill) and is
    kept fixed for tokens appended later (the page averages all keys once, before the
    tables are built; averaging again each step would change every stored code).
    Returns float64 [d]; zeros if the range is empty.
    """
    k = _f64(keys)
    lo, hi = min(n_sink, n_prefill), n_prefill
    if hi <= lo:
        return np.zeros(k.shape[-1])
    return k[lo:hi].mean(axis=0)


# ----------------------------------------------------------------------------------
# a2 / a5: SimHash codes
# ----------------------------------------------------------------------------------

def projections(x, W, center=None) -> np.ndarray:
    """Random projections y = (x - center) W of rows x [n, d] onto the K·L columns
    of W [d, K·L] ([MagicPIG] §2.2 SimHash; Algorithm 1 'Encode'). float64 [n, K·L]."""
    x = _f64(x)
    if center is not None:
        x = x - _f64(center)[None, :]
    return x @ _f64(W)


def near_ties(x, W, center=None) -> np.ndarray:
    """Mask [n, K·L] of projections with |y| <= 1e-5 * ||x - center|| * ||W[:, j]||.
    These sign decisions are too close to zero to be reproduced bit-exactly by
    fp32 arithmetic, so comparisons exclude them (and count them).

    READING: the band is closed, so an exact zero projection is always a near tie,
    also when x equals the center (both sides zero). SimHash keeps the sign of the
    projection ([MagicPIG] §2.2), which a zero projection does not have; its bit is a
    convention of each implementation and is not compared."""
    x = _f64(x)
    if center is not None:
        x = x - _f64(center)[None, :]
    y = x @ _f64(W)
    bound = NEAR_TIE_REL * np.linalg.norm(x, axis=1)[:, None] * np.linalg.norm(_f64(W), axis=0)[None, :]
    return np.abs(y) <= bound


def simhash_codes(x, W, K: int, L: int, center=None) -> np.ndarray:
    """L packed K-bit SimHash codes per row, [MagicPIG] §2.2 and §4.3 "Hash function
    selection": each table projects onto K random directions and keeps the signs.

    READING: bit b of table t is 1 iff projection column j = t*K + b is > 0 (a zero
    projection gives 0); the code of table t is sum_b bit_b * 2^b.
    Returns int64 [n, L].
    """
    y = projections(x, W, center)
    n = y.shape[0]
    codes = np.zeros((n, L), dtype=np.int64)
    for t in range(L):
        for b in range(K):
            codes[:, t] |= (y[:, t * K + b] > 0).astype(np.int64) << b
    return codes


# ----------------------------------------------------------------------------------
# a6: match counts and the sampled set
# ----------------------------------------------------------------------------------

def lsh_region(n: int, n_sink: int, window: int) -> tuple[int, int]:
    """Token range [lo, hi) that is LSH-sampled: everything but the first n_sink
    tokens and the last `window` tokens ([MagicPIG] §4.4 "On-device cache"; §5.1
    Baselines: 4 initial tokens and a local window are kept exactly). Empty when
    n <= n_sink + window."""
    lo = min(n_sink, n)
    hi = max(lo, n - window)
    return lo, hi


def exact_tokens(n: int, n_sink: int, window: int) -> np.ndarray:
    """Static tokens attended with u = 1: sinks [0, s) and the window [n-w, n)."""
    lo, hi = lsh_region(n, n_sink, window)
    return np.concatenate([np.arange(0, lo), np.arange(hi, n)]).astype(np.int64)


def match_counts(key_codes, q_code) -> np.ndarray:
    """Number of tables in which each key's code equals the query's code."""
    kc = np.asarray(key_codes)
    qc = np.asarray(q_code)
    return (kc == qc[None, :]).sum(axis=1)


def sampled_set(counts, n: int, n_sink: int, window: int, threshold: int = THRESHOLD) -> np.ndarray:
    """S = {i in the LSH region : count_i >= threshold}, ascending ([MagicPIG] §4.3:
    a key is sampled only if it shares the query's code in at least two tables).
    `counts` covers tokens [0, n)."""
    lo, hi = lsh_region(n, n_sink, window)
    c = np.asarray(counts)[lo:hi]
    return (np.nonzero(c >= threshold)[0] + lo).astype(np.int64)


# ----------------------------------------------------------------------------------
# a7: collision and inclusion probabilities
# ----------------------------------------------------------------------------------

def collision_probability(q, kc) -> np.ndarray:
    """Per-hyperplane collision probability p = 1 - arccos(cos(q, k))/pi
    ([MagicPIG] §2.2 SimHash; Eq. 10 and Eq. 11).

    READING: k is the centered key k_i - c, the vector that was hashed (§4.3 "Data
    pre-processing"); Algorithm 1 prints p = 1 - w/(|q||K_S|) without the arccos,
    which contradicts Eq. 10/11, so Eq. 10/11 is followed. A zero-norm vector gives
    cos = 0 (p = 1/2). kc: [m, d]; returns float64 [m].
    """
    q = _f64(q)
    kc = _f64(kc)
    qn = np.linalg.norm(q)
    kn = np.linalg.norm(kc, axis=1)
    dots = kc @ q
    denom = qn * kn
    cos = np.where(denom > 0, dots / np.where(denom > 0, denom, 1.0), 0.0)
    cos = np.clip(cos, -1.0, 1.0)
    return 1.0 - np.arccos(cos) / math.pi


def _log_binom(L: int, j: int) -> float:
    return math.lgamma(L + 1) - math.lgamma(j + 1) - math.lgamma(L - j + 1)


def inclusion_probability(p, K: int, L: int, threshold: int = THRESHOLD) -> np.ndarray:
    """Probability that a key is sampled, [MagicPIG] Eq. 10 / Eq. 11:
    u = 1 - (1 - p^K)^L - L p^K (1 - p^K)^(L-1), i.e. P[Binomial(L, x) >= 2] with
    x = p^K the chance that one table's K bits all agree.

    Evaluated stably: when L*x is small the closed form cancels catastrophically, so
    the tail sum_{j >= T} C(L, j) x^j (1-x)^(L-j) is added term by term in log space
    until the terms fall below 1e-18 of the sum; otherwise the closed form
    1 - sum_{j < T} C(L, j) x^j (1-x)^(L-j) is used. Returns float64 like p.
    """
    p = _f64(p)
    flat = p.reshape(-1)
    out = np.empty_like(flat)
    T = int(threshold)
    for idx, pi in enumerate(flat):
        x = float(pi) ** K
        if x <= 0.0:
            out[idx] = 0.0 if T > 0 else 1.0
            continue
        if x >= 1.0:
            out[idx] = 1.0 if T <= L else 0.0
            continue
        if T <= 0:
            out[idx] = 1.0
            continue
        if T > L:
            out[idx] = 0.0
            continue
        lx, l1x = math.log(x), math.log1p(-x)
        if L * x <= 0.5 * T:
            total = 0.0
            for j in range(T, L + 1):
                term = math.exp(_log_binom(L, j) + j * lx + (L - j) * l1x)
                total += term
                if term < 1e-18 * total:
                    break
            out[idx] = total
        else:
            head = sum(math.exp(_log_binom(L, j) + j * lx + (L - j) * l1x) for j in range(T))
            out[idx] = 1.0 - head
    return out.reshape(p.shape)


def expected_budget(K: int, L: int) -> float:
    """Expected sampled fraction B/n = 1 - (1-0.5^K)^L - L 0.5^K (1-0.5^K)^(L-1) when
    every table collides with probability 0.5^K (author responses on (K, L) and the
    computation budget, 'Theoretically' paragraph)."""
    x = 0.5 ** K
    return 1.0 - (1.0 - x) ** L - L * x * (1.0 - x) ** (L - 1)


# ----------------------------------------------------------------------------------
# a7 - a9: the estimator
# ----------------------------------------------------------------------------------

def snis_logits(q, keys, S, u_S, T) -> tuple[np.ndarray, np.ndarray]:
    """Logits of [MagicPIG] Algorithm 1 / Eq. 11: q k_i / sqrt(d) - log u_i for the
    sampled keys S and q k_i / sqrt(d) for the static tokens T (u = 1).

    READING: raw (uncentered) keys in the logits for both S and T, as Algorithm 1
    writes them; softmax is translation invariant so this equals the centered form.
    Returns (indices, logits) with S first, then T.
    """
    q = _f64(q)
    k = _f64(keys)
    S = np.asarray(S, dtype=np.int64)
    T = np.asarray(T, dtype=np.int64)
    d = q.shape[0]
    idx = np.concatenate([S, T])
    logit = (k[idx] @ q) / math.sqrt(d)
    logit[: len(S)] -= np.log(_f64(u_S))
    return idx, logit


def snis_attention(q, keys, values, S, u_S, T) -> np.ndarray:
    """Self-normalized importance-sampling attention output, [MagicPIG] Eq. 9 / Eq. 11
    and Algorithm 1: softmax of the corrected logits over S ∪ T applied to V."""
    idx, logit = snis_logits(q, keys, S, u_S, T)
    if len(idx) == 0:
        return np.zeros(_f64(values).shape[-1])
    m = logit.max()
    e = np.exp(logit - m)
    return (e[:, None] * _f64(values)[idx]).sum(axis=0) / e.sum()


def snis_sums(q, keys, values, S, u_S, T, ref: float) -> tuple[np.ndarray, float]:
    """Numerator and denominator of Eq. 9 scaled by exp(-ref): (sum w~_i/u_i v_i,
    sum w~_i/u_i) over S ∪ T. Used to check that they are unbiased estimates."""
    idx, logit = snis_logits(q, keys, S, u_S, T)
    e = np.exp(logit - ref)
    return (e[:, None] * _f64(values)[idx]).sum(axis=0), float(e.sum())


def exact_attention(q, keys, values) -> np.ndarray:
    """o = Softmax(q K^T / sqrt(d)) V, [MagicPIG] §2.1 Eq. 1."""
    q = _f64(q)
    k = _f64(keys)
    logit = k @ q / math.sqrt(q.shape[0])
    e = np.exp(logit - logit.max())
    return (e[:, None] * _f64(values)).sum(axis=0) / e.sum()


# ----------------------------------------------------------------------------------
# composition: one query head, one decode step ([MagicPIG] Algorithm 1)
# ----------------------------------------------------------------------------------

class HeadTables:
    """Codes of every token of one KV head, as the tables would index them.

    Built from the prefill keys [0, n_prefill) with center c = mean over
    [n_sink, n_prefill); tokens appended later are hashed with the same c.
    """

    def __init__(self, keys, W, K: int, L: int, n_sink: int, n_prefill: int,
                 n_total: int | None = None, centering: bool = True):
        keys = _f64(keys)
        n_total = keys.shape[0] if n_total is None else n_total
        self.K, self.L, self.n_sink = K, L, n_sink
        self.W = _f64(W)
        # centering=False is the pages' ablation without the data pre-processing step:
        # keys are hashed as they are (c = 0), and p uses cos(q, k)
        self.center = center_of_keys(keys, n_sink, n_prefill) if centering else np.zeros(keys.shape[1])
        self.codes = simhash_codes(keys[:n_total], self.W, K, L, self.center)
        self.ties = near_ties(keys[:n_total], self.W, self.center)


def decode_head(q, keys, values, tables: HeadTables, n: int, window: int,
                threshold: int = THRESHOLD, key_codes=None, q_code=None, center_query: bool = False) -> dict:
    """One decode step for one query head ([MagicPIG] Algorithm 1 with the on-device
    cache of §4.4): encode q, query the tables, weight the sampled keys by -log u,
    attend exactly over sinks and window.

    READING: the query is hashed uncentered (only keys are centered in §4.3), and the
    collision probability is that of q with the centered key. With center_query the
    other reading is taken: q - c is hashed and p is the collision probability of
    q - c with k - c, the pair of vectors whose signs are compared. The logits use
    the raw q and k in both readings. `key_codes` / `q_code` may be given to run the
    later steps on codes computed elsewhere (stage-wise checks). Returns a dict with
    the intermediate results.
    """
    q = _f64(q)
    K, L, s = tables.K, tables.L, tables.n_sink
    qh = q - tables.center if center_query else q   # the vector that is hashed
    qc = simhash_codes(qh[None, :], tables.W, K, L)[0] if q_code is None else np.asarray(q_code)
    kc = tables.codes[:n] if key_codes is None else np.asarray(key_codes)[:n]
    counts = match_counts(kc, qc)
    S = sampled_set(counts, n, s, window, threshold)
    T = exact_tokens(n, s, window)
    k64 = _f64(keys)[:n]
    p = collision_probability(qh, k64[S] - tables.center[None, :])
    u = inclusion_probability(p, K, L, threshold)
    o = snis_attention(q, k64, _f64(values)[:n], S, u, T)
    return {"q_code": qc, "counts": counts, "S": S, "T": T, "p": p, "u": u, "out": o}
