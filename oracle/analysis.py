"""Closed forms for the SANTA / S2ANTA estimators (float64, numpy).

TEST INFRASTRUCTURE ONLY.  These formulas come from "Stochastic Sparse
Attention for Memory-Bound Inference":

* mean of every variant is the exact attention output mu = sum_n p_n V_n
  (App. A, Prop. A.2 and A.4);
* i.i.d. covariance trace tr(Sigma)/S with
  tr(Sigma) = sum_n p_n |V_n|^2 - |mu|^2 (App. A.2, Prop. A.3; App. M);
* independent stratified variance trace (1/S^2) sum_m tr(Sigma_m), Sigma_m
  the value covariance of the within-stratum distribution (App. A.5,
  Thm. A.6; App. M);
* systematic variance by replicates (App. M), and exactly as the integral
  over the shared offset u of the squared deviation of the estimate, which is
  constant between the offsets where a threshold (j + u)/S crosses a CDF edge
  (Sec. 2.1 systematic sampling; the paper gives no closed form);
* vector Bernstein tail for i.i.d. SANTA (App. B, Thm. B.1);
* expected number of distinct keys drawn (App. L, App. M.1 item 1) for the
  i.i.d., stratified and systematic samplers, and the expected share of V
  rows a causal prefill pass of i.i.d. SANTA reads (App. F, Table 9).

Strata follow Sec. 2.1: I_m = [m/S, (m+1)/S), with the inverse CDF of App. A.4.
"""
from __future__ import annotations

import math

import numpy as np


def cdf(p: np.ndarray) -> np.ndarray:
    return np.cumsum(np.asarray(p, dtype=np.float64))


def exact_mean(p: np.ndarray, V: np.ndarray) -> np.ndarray:
    return np.asarray(p, np.float64) @ np.asarray(V, np.float64)


def iid_variance_trace(p: np.ndarray, V: np.ndarray, S: int) -> float:
    V = np.asarray(V, np.float64)
    mu = exact_mean(p, V)
    tr = float(np.dot(p, np.einsum("nd,nd->n", V, V)) - mu @ mu)
    return tr / S


def iid_coordinate_variance(p: np.ndarray, V: np.ndarray, S: int) -> np.ndarray:
    """Diagonal of Sigma / S (per output coordinate)."""
    V = np.asarray(V, np.float64)
    mu = exact_mean(p, V)
    return (np.asarray(p) @ (V * V) - mu * mu) / S


def stratum_weights(p: np.ndarray, S: int) -> np.ndarray:
    """w[m, n] = S * |I_m intersect [F(n-1), F(n))| : the distribution of
    F^-1(T) for T uniform on stratum I_m (rows sum to 1)."""
    F = cdf(p)
    Fl = np.concatenate([[0.0], F[:-1]])
    m = np.arange(S, dtype=np.float64)
    lo = np.maximum(Fl[None, :], (m / S)[:, None])
    hi = np.minimum(F[None, :], ((m + 1) / S)[:, None])
    return S * np.clip(hi - lo, 0.0, None)


def stratified_mean(p: np.ndarray, V: np.ndarray, S: int) -> np.ndarray:
    w = stratum_weights(p, S)
    return (w @ np.asarray(V, np.float64)).sum(axis=0) / S


def stratified_variance_trace(p: np.ndarray, V: np.ndarray, S: int) -> float:
    V = np.asarray(V, np.float64)
    w = stratum_weights(p, S)
    mu_m = w @ V                                   # [S, d]
    second = w @ np.einsum("nd,nd->n", V, V)       # [S]
    tr_m = second - np.einsum("md,md->m", mu_m, mu_m)
    return float(tr_m.sum()) / (S * S)


def stratified_coordinate_variance(p: np.ndarray, V: np.ndarray, S: int) -> np.ndarray:
    V = np.asarray(V, np.float64)
    w = stratum_weights(p, S)
    mu_m = w @ V
    var_m = w @ (V * V) - mu_m * mu_m
    return var_m.sum(axis=0) / (S * S)


def systematic_breakpoints(p: np.ndarray, S: int) -> np.ndarray:
    """Offsets u in [0,1) at which some systematic threshold (j+u)/S crosses a
    CDF edge F(n): u = S F(n) - j.  Between consecutive breakpoints the
    systematic sample is constant."""
    F = cdf(p)
    u = (S * F)[:, None] - np.arange(S)[None, :]
    u = u[(u > 0.0) & (u < 1.0)]
    return np.unique(np.concatenate([[0.0, 1.0], u]))


def expectation_over_offset(estimator, breakpoints: np.ndarray) -> np.ndarray:
    """Exact integral over u in [0,1) of a piecewise-constant estimator(u):
    sum over the pieces of (length * value at the midpoint)."""
    total = None
    for a, b in zip(breakpoints[:-1], breakpoints[1:]):
        if b <= a:
            continue
        val = np.asarray(estimator(0.5 * (a + b)), np.float64) * (b - a)
        total = val if total is None else total + val
    return total


def systematic_estimates(p: np.ndarray, V: np.ndarray, S: int, u: np.ndarray) -> np.ndarray:
    """The systematic estimate (1/S) sum_j V[F^-1((j + u)/S)] for each offset
    in u (shape [M]); F^-1(t) is the first key n with F(n) > t (App. A.4)."""
    F = cdf(p)
    V = np.asarray(V, np.float64)
    t = (np.arange(S, dtype=np.float64)[None, :] + np.asarray(u, np.float64)[:, None]) / S
    keys = np.minimum(np.searchsorted(F, t, side="right"), len(F) - 1)
    return V[keys].mean(axis=1)


def systematic_coordinate_variance(p: np.ndarray, V: np.ndarray, S: int) -> np.ndarray:
    """Per output coordinate, the exact variance of the systematic estimate
    over u ~ U[0, 1): the integral of (estimate(u) - mu)^2.

    As u grows each CDF edge F(n) < 1 is passed by exactly one threshold
    (j + u)/S, at u = S F(n) - floor(S F(n)), and that threshold's key moves
    from n to n + 1, changing the estimate by (V[n+1] - V[n]) / S.  So the
    estimate is the u = 0 estimate plus a running sum of these steps in the
    order of their offsets, constant in between: O(nk d) in all."""
    V = np.asarray(V, np.float64)
    F = cdf(p)
    mu = exact_mean(p, V)
    x = S * F[:-1]
    jn = np.floor(x)
    ue = x - jn
    ev = np.nonzero((ue > 0.0) & (jn < S))[0]          # edges passed for some u in (0, 1)
    order = np.argsort(ue[ev], kind="stable")
    ev = ev[order]
    steps = (V[ev + 1] - V[ev]) / S
    states = np.concatenate([systematic_estimates(p, V, S, np.zeros(1)),
                             systematic_estimates(p, V, S, np.zeros(1)) + np.cumsum(steps, axis=0)])
    cuts = np.concatenate([[0.0], ue[ev], [1.0]])
    dev = states - mu
    return np.diff(cuts) @ (dev * dev)


def expected_unique_keys_systematic(p: np.ndarray, S: int) -> float:
    """E|U| for systematic sampling: key n is drawn as often as the lattice
    {(j + u)/S} meets [F(n-1), F(n)), an interval of length p_n, so at least
    once with probability min(1, S p_n)."""
    return float(np.minimum(1.0, S * np.asarray(p, np.float64)).sum())


def expected_unique_keys_stratified(p: np.ndarray, S: int) -> float:
    """E|U| for independent stratified sampling: stratum m draws key n with
    probability w[m, n] (stratum_weights), independently of the other
    strata, so key n is missed with probability prod_m (1 - w[m, n])."""
    w = stratum_weights(p, S)
    return float((1.0 - np.prod(1.0 - w, axis=0)).sum())


def replicate_variance_trace(estimates: np.ndarray) -> float:
    """App. M replicate estimator: (1/(R-1)) sum_r |est_r - mean|^2."""
    E = np.asarray(estimates, np.float64)
    R = E.shape[0]
    c = E - E.mean(axis=0, keepdims=True)
    return float(np.einsum("rd,rd->", c, c)) / (R - 1)


def bernstein_radius(v: float, vmax: float, S: int, delta: float) -> float:
    """App. B: with probability >= 1 - delta the i.i.d. error norm is below
    sqrt(2 v log(2/delta) / S) + 2 vmax log(2/delta) / (3 S)."""
    L = math.log(2.0 / delta)
    return math.sqrt(2.0 * v * L / S) + 2.0 * vmax * L / (3.0 * S)


def systematic_count_bounds(p: np.ndarray, S: int):
    """Each key's systematic count lies in {floor(S p_n), ceil(S p_n)}
    (lattice points of spacing 1/S in an interval of length p_n)."""
    Sp = S * np.asarray(p, np.float64)
    return np.floor(Sp), np.ceil(Sp)


def expected_unique_keys_iid(p: np.ndarray, S: int) -> float:
    """App. M.1 (1): E|{J_1..J_S}| for S i.i.d. draws from p, sum_n 1 - (1 - p_n)^S."""
    p = np.asarray(p, np.float64)
    with np.errstate(divide="ignore"):   # p_n = 1 gives log(0) = -inf: the key is always drawn
        return float(np.sum(-np.expm1(S * np.log1p(-p))))


def causal_softmax(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """Rows i of softmax(q k^T scale) over keys 0..i (a causal prefill pass), float64."""
    s = (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T) * scale
    n = s.shape[0]
    s[np.triu_indices(n, 1)] = -np.inf
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return p / p.sum(axis=1, keepdims=True)


def prefill_coverage_iid(P: np.ndarray, S: int) -> float:
    """App. F, Table 9: the expected share of the nk V rows drawn by at least
    one query of a causal prefill pass when every query i draws S i.i.d.
    keys from its row P[i]: mean over keys j of 1 - prod_{i >= j} (1 - P_ij)^S."""
    P = np.asarray(P, np.float64)
    with np.errstate(divide="ignore"):   # query 0 draws key 0 with probability 1
        log_none = S * np.log1p(-P).sum(axis=0)
    return float(np.mean(-np.expm1(log_none)))
