"""Mutation check of the oracle's pins.

Each case plants one plausible mistake in the CPU oracle (a dropped term, a wrong
sign, an off-by-one index, a transposed operand, the other reading of an ambiguous
step), for the duration of the case only, and runs the pins of
`test_oracle_pins.py` until one fails. Every mistake must be caught by at least one
pin: one that no pin notices could sit in the oracle unseen. Mistakes are planted in
the oracle only, on the CPU.
"""
import inspect
import itertools
import math

import numpy as np
import pytest

import oracle
import oracle.magicpig_oracle as M
import test_oracle_pins as PINS

ORIG = {name: getattr(M, name) for name in dir(M) if callable(getattr(M, name)) and not name.startswith("__")}


def _pin_cases():
    """(name, function, kwargs) for every pin, parametrizations expanded, in file order."""
    for name, fn in list(vars(PINS).items()):
        if not (name.startswith("test_") and inspect.isfunction(fn)):
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names = [a.strip() for a in mark.args[0].split(",")] if isinstance(mark.args[0], str) \
                else list(mark.args[0])
            grid = []
            for v in mark.args[1]:
                v = v.values if hasattr(v, "values") else v
                grid.append(dict(zip(names, v if len(names) > 1 else (v,))))
            grids.append(grid)
        for combo in itertools.product(*grids):
            kw = {}
            for c in combo:
                kw.update(c)
            yield name, fn, kw


PIN_CASES = list(_pin_cases())


# ----------------------------------------------------------------------------------
# planted mistakes, one per case: {oracle function name: replacement}
# ----------------------------------------------------------------------------------

def _codes_by_column(col):
    """simhash_codes with bit b of table t taken from column col(t, b, K, L)."""
    def simhash_codes(x, W, K, L, center=None):
        y = M.projections(x, W, center)
        codes = np.zeros((y.shape[0], L), dtype=np.int64)
        for t in range(L):
            for b in range(K):
                codes[:, t] |= (y[:, col(t, b, K, L)] > 0).astype(np.int64) << b
        return codes
    return simhash_codes


def _codes_negative_side(x, W, K, L, center=None):
    y = M.projections(x, W, center)
    codes = np.zeros((y.shape[0], L), dtype=np.int64)
    for t in range(L):
        for b in range(K):
            codes[:, t] |= (y[:, t * K + b] < 0).astype(np.int64) << b
    return codes


def _logits_plus_log_u(q, keys, S, u_S, T):
    idx, logit = ORIG["snis_logits"](q, keys, S, u_S, T)
    logit[: len(S)] += 2.0 * np.log(np.asarray(u_S, float))
    return idx, logit


def _logits_unscaled(q, keys, S, u_S, T):
    idx, logit = ORIG["snis_logits"](q, keys, S, u_S, T)
    d = np.asarray(q).shape[0]
    logit[: len(S)] += np.log(np.asarray(u_S, float))
    logit *= math.sqrt(d)
    logit[: len(S)] -= np.log(np.asarray(u_S, float))
    return idx, logit


def _logits_without_static(q, keys, S, u_S, T):
    idx, logit = ORIG["snis_logits"](q, keys, S, u_S, [])
    return idx, logit


def _u_closed_form_as_printed(p, K, L, threshold=M.THRESHOLD):
    if threshold != 2:
        return ORIG["inclusion_probability"](p, K, L, threshold)
    x = np.asarray(p, float) ** K
    return 1.0 - (1.0 - x) ** L - L * x * (1.0 - x) ** (L - 1)


def _decode_head_p_from_raw_keys(q, keys, values, tables, n, window, threshold=M.THRESHOLD, key_codes=None,
                                 q_code=None, center_query=False):
    r = ORIG["decode_head"](q, keys, values, tables, n, window, threshold, key_codes, q_code, center_query)
    k64 = np.asarray(keys, float)[:n]
    qh = np.asarray(q, float) - (tables.center if center_query else 0.0)
    p = M.collision_probability(qh, k64[r["S"]])
    u = M.inclusion_probability(p, tables.K, tables.L, threshold)
    out = M.snis_attention(q, k64, np.asarray(values, float)[:n], r["S"], u, r["T"])
    return {**r, "p": p, "u": u, "out": out}


def _decode_head_centered_query(q, keys, values, tables, n, window, threshold=M.THRESHOLD, key_codes=None,
                                q_code=None, center_query=False):
    qc = M.simhash_codes(np.asarray(q, float)[None, :], tables.W, tables.K, tables.L, tables.center)[0]
    return ORIG["decode_head"](q, keys, values, tables, n, window, threshold, key_codes, qc, center_query)


def _decode_head_centered_hash_raw_p(q, keys, values, tables, n, window, threshold=M.THRESHOLD, key_codes=None,
                                     q_code=None, center_query=False):
    """Centered-query reading with p taken from the raw query."""
    if not center_query:
        return ORIG["decode_head"](q, keys, values, tables, n, window, threshold, key_codes, q_code)
    qc = M.simhash_codes(np.asarray(q, float)[None, :], tables.W, tables.K, tables.L, tables.center)[0]
    return ORIG["decode_head"](q, keys, values, tables, n, window, threshold, key_codes, qc, False)


class _TablesAppendedUncentered(ORIG["HeadTables"]):
    """Appended tokens hashed without the center."""

    def __init__(self, keys, W, K, L, n_sink, n_prefill, n_total=None, centering=True):
        super().__init__(keys, W, K, L, n_sink, n_prefill, n_total, centering)
        nt = self.codes.shape[0]
        if nt > n_prefill:
            self.codes[n_prefill:] = M.simhash_codes(np.asarray(keys, float)[n_prefill:nt], self.W, K, L)


MUTANTS = {
    # a1 centering
    "center includes the sinks": {"center_of_keys": lambda keys, s, n0: ORIG["center_of_keys"](keys, 0, n0)},
    "center includes appended keys": {
        "center_of_keys": lambda keys, s, n0: ORIG["center_of_keys"](keys, s, np.asarray(keys).shape[0])},
    # a2 / a5 hashing
    "projection ignores the center": {"projections": lambda x, W, center=None: ORIG["projections"](x, W, None)},
    "projection adds the center": {
        "projections": lambda x, W, center=None: ORIG["projections"](x, W, None if center is None
                                                                    else -np.asarray(center, float))},
    "bits of a table reversed": {"simhash_codes": _codes_by_column(lambda t, b, K, L: t * K + (K - 1 - b))},
    "table and bit indices transposed": {"simhash_codes": _codes_by_column(lambda t, b, K, L: b * L + t)},
    "bit set on the negative side": {"simhash_codes": _codes_negative_side},
    "near-tie band without the column norm": {
        "near_ties": lambda x, W, center=None: np.abs(M.projections(x, W, center)) < M.NEAR_TIE_REL * np.linalg.norm(
            np.asarray(x, float) - (0 if center is None else np.asarray(center, float)[None, :]), axis=1)[:, None]},
    "near-tie band open (exact zeros compared)": {
        "near_ties": lambda x, W, center=None: (lambda x0: np.abs(x0 @ np.asarray(W, float)) < M.NEAR_TIE_REL
                                                * np.linalg.norm(x0, axis=1)[:, None]
                                                * np.linalg.norm(np.asarray(W, float), axis=0)[None, :])(
            np.asarray(x, float) - (0 if center is None else np.asarray(center, float)[None, :]))},
    "query hashed centered": {"decode_head": _decode_head_centered_query},
    "centered query with p from the raw query": {"decode_head": _decode_head_centered_hash_raw_p},
    "appended tokens hashed uncentered": {"HeadTables": _TablesAppendedUncentered},
    # a6 match and region
    "query codes shifted by one table": {
        "match_counts": lambda kc, qc: ORIG["match_counts"](kc, np.roll(np.asarray(qc), 1))},
    "strict threshold": {
        "sampled_set": lambda c, n, s, w, threshold=M.THRESHOLD: ORIG["sampled_set"](c, n, s, w, threshold + 1)},
    "sinks in the sampled region": {"lsh_region": lambda n, s, w: (0, max(0, n - w))},
    "window one token short": {
        "lsh_region": lambda n, s, w: (min(s, n), max(min(s, n), min(n, n - w + 1)))},
    # a7 probabilities
    "p linear in the cosine": {  # (1 + cos)/2 instead of 1 - theta/pi
        "collision_probability": lambda q, kc:
        (1.0 + np.cos(math.pi * (1.0 - ORIG["collision_probability"](q, kc)))) / 2.0},
    "p from the raw keys": {"decode_head": _decode_head_p_from_raw_keys},
    "u forgets the one-table term": {
        "inclusion_probability": lambda p, K, L, threshold=M.THRESHOLD:
        ORIG["inclusion_probability"](p, K, L, max(1, threshold - 1))},
    "u with x = p^L": {
        "inclusion_probability": lambda p, K, L, threshold=M.THRESHOLD:
        ORIG["inclusion_probability"](p, L, L, threshold)},
    "u from the printed closed form (cancels)": {"inclusion_probability": _u_closed_form_as_printed},
    "budget forgets the one-table term": {"expected_budget": lambda K, L: 1.0 - (1.0 - 0.5 ** K) ** L},
    # a7 - a9 estimator
    "logit adds log u": {"snis_logits": _logits_plus_log_u},
    "logit without 1/sqrt(d)": {"snis_logits": _logits_unscaled},
    "static tokens dropped": {"snis_logits": _logits_without_static},
    "exact attention without 1/sqrt(d)": {
        "exact_attention": lambda q, k, v: ORIG["exact_attention"](np.asarray(q, float) * math.sqrt(len(q)), k, v)},
}


def _first_failing_pin():
    for name, fn, kw in PIN_CASES:
        try:
            fn(**kw)
        except AssertionError:
            return f"{name}{kw if kw else ''}"
    return None


def test_every_pin_passes_on_the_oracle_as_it_is():
    assert len(PIN_CASES) >= 20
    assert _first_failing_pin() is None


@pytest.mark.parametrize("mistake", sorted(MUTANTS))
def test_planted_mistake_is_caught(mistake, monkeypatch):
    for fname, repl in MUTANTS[mistake].items():
        monkeypatch.setattr(M, fname, repl)
        monkeypatch.setattr(oracle, fname, repl, raising=False)
    with np.errstate(all="ignore"):
        caught = _first_failing_pin()
    assert caught is not None, f"no pin notices: {mistake}"
    print(f"\n[{mistake}] caught by {caught}")
