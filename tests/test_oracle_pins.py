"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources ("Stochastic Sparse Attention for Memory-Bound Inference"):
worked example Sec. 1 Eq. (2)-(3); SDPA Sec. 2 Eq. (1); estimators Eq. (4)
and Sec. 2.1; inverse CDF App. A.4; unbiasedness Prop. A.2 / A.4; variance
Prop. A.3, Thm. A.6, App. M; Bernstein tail App. B Thm. B.1.  The Philox
stream is pinned against PyTorch's header-only engine (an independent
implementation of Salmon et al., SC'11).
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest
import torch

import synth
from oracle import analysis

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def make_problem(oracle, q, K, V, scale=0.0, dtype="fp32"):
    """Single-sequence fp32 problem from float arrays: q [H,d], K/V [nk,Hkv,d]."""
    q = np.asarray(q, np.float32)
    K = np.asarray(K, np.float32)
    V = np.asarray(V, np.float32)
    if q.ndim == 2:
        q = q[None]
    offs = np.array([0, K.shape[0]], np.int64)
    return oracle.Problem(q, K, V, offs, dtype, K.shape[1], scale)


def problem_from_probs(oracle, p, V):
    """nk keys whose softmax is (numerically) p: q = e0, K_n = log(p_n) e0, scale 1."""
    p = np.asarray(p, np.float64)
    V = np.asarray(V, np.float32)
    nk, d = V.shape
    q = np.zeros((1, max(d, 1)), np.float32)
    q[0, 0] = 1.0
    K = np.zeros((nk, 1, d), np.float32)
    K[:, 0, 0] = np.log(p).astype(np.float32)
    return make_problem(oracle, q, K, V[:, None, :], scale=1.0)


def random_problem(oracle, rng, nk, d, H=1, Hkv=1, spread=2.0):
    q = rng.standard_normal((H, d)).astype(np.float32) * np.float32(spread)
    K = rng.standard_normal((nk, Hkv, d)).astype(np.float32)
    V = rng.standard_normal((nk, Hkv, d)).astype(np.float32)
    return make_problem(oracle, q, K, V)


def values_of(P, b, h):
    """V rows of head (b, h) as float64 [nk, d] (storage is fp32 here)."""
    B, H, Hkv, d = P.shape
    kvh = h // (H // Hkv)
    off = P.kv_offsets
    return synth.storage_to_f64(P.V[off[b]:off[b + 1], kvh], P.dtype)


@pytest.fixture(scope="module")
def torch_philox(tmp_path_factory):
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    out = tmp_path_factory.mktemp("philox") / "libtorch_philox.so"
    subprocess.run(["g++", "-std=c++17", "-O1", "-shared", "-fPIC", "-I", inc,
                    os.path.join(HERE, "philox_torch_shim.cpp"), "-o", str(out)], check=True)
    lib = ctypes.CDLL(str(out))
    lib.torch_philox_block.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                       ctypes.c_void_p]

    def block(seed, subsequence, offset):
        w = np.zeros(4, np.uint32)
        lib.torch_philox_block(seed, subsequence, offset, w.ctypes.data_as(ctypes.c_void_p))
        return w
    return block


# ---------------------------------------------------------------------------
# Philox stream and uniform map
# ---------------------------------------------------------------------------

def test_philox_words_match_torch_engine(oracle_lib, torch_philox):
    """counter (i, h, b, step), key (seed_lo, seed_hi) == torch engine with
    subsequence = step<<32 | b and offset = h<<32 | i."""
    rng = np.random.default_rng(1)
    cases = [(0, 0, 0, 0, 0), (0xFFFFFFFFFFFFFFFF, 7, 31, 5, 3), (123456789, 63, 27, 1 << 20, 1023)]
    for _ in range(200):
        cases.append((int(rng.integers(0, 2**63)), int(rng.integers(0, 64)), int(rng.integers(0, 64)),
                      int(rng.integers(0, 2**32)), int(rng.integers(0, 4096))))
    for seed, b, h, step, i in cases:
        ours = oracle_lib.philox4x32_10([i, h, b, step], [seed & 0xFFFFFFFF, seed >> 32])
        ref = torch_philox(seed, (step << 32) | b, (h << 32) | i)
        np.testing.assert_array_equal(ours, ref)


def test_uniform_map_and_threshold_layout(oracle_lib, torch_philox):
    seed, b, h, step, S = 99, 3, 5, 7, 37
    words = np.concatenate([torch_philox(seed, (step << 32) | b, (h << 32) | i) for i in range((S + 3) // 4)])
    u_ref = (words >> 8).astype(np.float64) / 2.0**24
    u = np.array([oracle_lib.uniform(seed, b, h, step, r) for r in range(S)])
    np.testing.assert_array_equal(u, u_ref[:S])
    assert u.min() >= 0.0 and u.max() <= 1.0 - 2.0**-24
    # Sec. 2.1 threshold rules on that stream
    np.testing.assert_array_equal(oracle_lib.thresholds("systematic", S, seed, b, h, step),
                                  (np.arange(S) + u_ref[0]) / S)
    np.testing.assert_array_equal(oracle_lib.thresholds("stratified", S, seed, b, h, step),
                                  (np.arange(S) + u_ref[:S]) / S)
    np.testing.assert_array_equal(oracle_lib.thresholds("iid", S, seed, b, h, step), np.sort(u_ref[:S]))


# ---------------------------------------------------------------------------
# worked example and the score / softmax stage
# ---------------------------------------------------------------------------

def test_worked_example_nk3(oracle_lib):
    g = json.load(open(os.path.join(HERE, "golden", "worked_example_nk3.json")))
    V = np.array(g["V"], np.float64)
    P = problem_from_probs(oracle_lib, g["p"], V)
    est, J, delta = oracle_lib.sample_head(P, 0, 0, np.array(g["thresholds"]))
    assert list(J + 1) == g["sampled_keys_one_based"]
    counts = np.bincount(J, minlength=g["nk"])
    assert {str(k + 1): int(c) for k, c in enumerate(counts)} == g["counts_one_based"]
    np.testing.assert_allclose(est, (V[0] + V[0] + V[2]) / 3.0, rtol=1e-15, atol=1e-15)
    assert delta.min() > 0.05
    # the same estimate from the index multiset alone (Eq. 2-3 by distributivity)
    idx = np.array(g["sampled_keys_one_based"]) - 1
    np.testing.assert_allclose(oracle_lib.gather(P, 0, 0, idx), (V[0] + V[0] + V[2]) / 3.0, rtol=1e-15,
                               atol=1e-15)


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_dense_matches_torch_sdpa(oracle_lib, dtype):
    """Dense oracle == torch scaled_dot_product_attention in float64 (Eq. 1)."""
    wl = synth.Workload("t", 2, 8, 2, 64, 300, dtype, 8, "systematic")
    inp = synth.generate(wl, 3)
    P = oracle_lib.Problem.from_inputs(inp)
    out = oracle_lib.dense(P)
    q = torch.from_numpy(synth.storage_to_f64(inp.q, dtype))
    K = torch.from_numpy(synth.storage_to_f64(inp.K, dtype))
    V = torch.from_numpy(synth.storage_to_f64(inp.V, dtype))
    G = wl.group
    for b in range(wl.batch):
        sl = slice(int(inp.kv_offsets[b]), int(inp.kv_offsets[b + 1]))
        for h in range(wl.n_q_heads):
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[b, h][None, None, None], K[sl, h // G][None, None], V[sl, h // G][None, None])
            np.testing.assert_allclose(out[b, h], ref.reshape(-1).numpy(), rtol=1e-12, atol=1e-13)
            s, p = oracle_lib.scores(P, b, h)
            ref_p = torch.softmax(q[b, h] @ K[sl, h // G].T / np.sqrt(wl.head_dim), dim=0).numpy()
            np.testing.assert_allclose(p, ref_p, rtol=1e-12, atol=1e-300)


def test_tile_stats_match_logsumexp(oracle_lib):
    from scipy.special import logsumexp
    rng = np.random.default_rng(5)
    P = random_problem(oracle_lib, rng, 1000, 32, H=2, Hkv=1)
    for h in range(2):
        s, _ = oracle_lib.scores(P, 0, h)
        m, l = oracle_lib.tile_stats(P, 0, h, 96)
        assert m.shape[0] == 11
        for t in range(11):
            seg = s[96 * t: 96 * (t + 1)]
            assert m[t] == seg.max()
            np.testing.assert_allclose(m[t] + np.log(l[t]), logsumexp(seg), rtol=1e-14)


# ---------------------------------------------------------------------------
# inverse CDF convention and special cases
# ---------------------------------------------------------------------------

def test_inverse_cdf_left_closed_boundary(oracle_lib):
    """App. A.4: J = j with F(j-1) <= t < F(j).  With K = 0 and nk = 4 the CDF
    is exactly (0.25, 0.5, 0.75, 1); a threshold on an edge picks the next key."""
    V = np.arange(12, dtype=np.float32).reshape(4, 1, 3)
    P = make_problem(oracle_lib, np.ones((1, 3)), np.zeros((4, 1, 3)), V)
    _, J, delta = oracle_lib.sample_head(P, 0, 0, np.array([0.0, 0.25, 0.5, 0.75, 0.2499999, 0.9999, 0.3]))
    assert list(J) == [0, 1, 2, 3, 0, 3, 1]
    # delta: distance to the nearer end of the drawn key's interval [F(J-1), F(J))
    np.testing.assert_allclose(delta, [0.0, 0.0, 0.0, 0.0, 1e-7, 1e-4, 0.05], rtol=1e-6, atol=1e-15)


def test_threshold_at_the_total_mass_goes_to_the_last_key_with_mass(oracle_lib):
    """Reading of the clamp: a threshold at or past the rounded total mass goes
    to the last key with nonzero mass.  Keys whose mass underflows to zero in
    float64 (score 1000 below the others) are never drawn, because
    F(n-1) <= t < F(n) holds for no such key (App. A.4)."""
    d = 4
    q = np.zeros((1, d), np.float32)
    q[0, 0] = 1.0
    K = np.zeros((6, 1, d), np.float32)
    K[:, 0, 0] = [0.5, -0.2, 0.1, -1000.0, -1000.0, -1000.0]
    V = np.arange(6 * d, dtype=np.float32).reshape(6, 1, d)
    P = make_problem(oracle_lib, q, K, V, scale=1.0)
    _, p = oracle_lib.scores(P, 0, 0)
    assert p[3:].max() == 0.0 and p[:3].min() > 0.1
    _, J, _ = oracle_lib.sample_head(P, 0, 0, np.array([1.0, np.nextafter(1.0, 0.0), 0.0]))
    assert list(J) == [2, 2, 0]


def test_estimate_reads_the_rows_of_its_own_sequence(oracle_lib):
    """Eq. 4 in a packed ragged batch: the estimate of head (b, h) is
    (1/S) sum_j V[kv_offsets[b] + J_j, h // G], here by numpy indexing from
    the drawn keys."""
    rng = np.random.default_rng(21)
    lens = [37, 50, 23]
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    H, Hkv, d, S = 4, 2, 16, 16
    q = rng.standard_normal((3, H, d)).astype(np.float32)
    K = rng.standard_normal((offs[-1], Hkv, d)).astype(np.float32)
    V = rng.standard_normal((offs[-1], Hkv, d)).astype(np.float32)
    P = oracle_lib.Problem(q, K, V, offs, "fp32", Hkv)
    for b in range(3):
        for h in range(H):
            t = oracle_lib.thresholds("stratified", S, 5, b, h)
            est, J, _ = oracle_lib.sample_head(P, b, h, t)
            assert J.min() >= 0 and J.max() < lens[b]
            want = V[offs[b] + J, h // (H // Hkv)].astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(est, want, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(oracle_lib.gather(P, b, h, J), want, rtol=1e-12, atol=1e-12)


def test_all_rows_equal_gives_that_row(oracle_lib):
    rng = np.random.default_rng(2)
    row = rng.standard_normal(16).astype(np.float32)
    V = np.tile(row, (50, 1, 1))
    P = make_problem(oracle_lib, rng.standard_normal((1, 16)), rng.standard_normal((50, 1, 16)), V)
    for variant in ("iid", "stratified", "systematic"):
        est, _, _ = oracle_lib.decode(P, variant, 7, seed=11)
        np.testing.assert_array_equal(est[0, 0], row.astype(np.float64))


@pytest.mark.parametrize("variant", ["stratified", "systematic"])
def test_uniform_attention_with_S_equal_nk_visits_every_key_once(oracle_lib, variant):
    rng = np.random.default_rng(3)
    nk, d = 64, 8
    V = rng.standard_normal((nk, 1, d)).astype(np.float32)
    P = make_problem(oracle_lib, rng.standard_normal((1, d)), np.zeros((nk, 1, d)), V)
    for seed in range(5):
        est, J, _ = oracle_lib.decode(P, variant, nk, seed=seed)
        assert list(J[0, 0]) == list(range(nk))
        np.testing.assert_allclose(est[0, 0], V[:, 0].astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(est[0, 0], oracle_lib.dense(P)[0, 0], rtol=1e-12, atol=1e-13)


def test_dominant_key_is_always_drawn(oracle_lib):
    rng = np.random.default_rng(4)
    nk, d = 40, 8
    K = rng.standard_normal((nk, 1, d)).astype(np.float32)
    q = rng.standard_normal((1, d)).astype(np.float32)
    K[17, 0] = 40.0 * q[0] / np.linalg.norm(q[0])       # softmax mass of key 17 ~ 1 - 1e-30
    V = rng.standard_normal((nk, 1, d)).astype(np.float32)
    P = make_problem(oracle_lib, q, K, V, scale=1.0)
    for variant in ("iid", "stratified", "systematic"):
        est, J, _ = oracle_lib.decode(P, variant, 32, seed=1)
        assert set(J[0, 0].tolist()) == {17}
        np.testing.assert_array_equal(est[0, 0], V[17, 0].astype(np.float64))


# ---------------------------------------------------------------------------
# unbiasedness (Prop. A.2, A.4) as exact integrals over the randomness
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 2, 3, 5, 8])
def test_systematic_sampler_exact_expectation_is_attention(oracle_lib, S):
    rng = np.random.default_rng(10 + S)
    P = random_problem(oracle_lib, rng, 9, 6, spread=1.5)
    _, p = oracle_lib.scores(P, 0, 0)
    mu = oracle_lib.dense(P)[0, 0]

    def est_at(u):
        t = (np.arange(S) + u) / S
        return oracle_lib.sample_head(P, 0, 0, t)[0]

    E = analysis.expectation_over_offset(est_at, analysis.systematic_breakpoints(p, S))
    np.testing.assert_allclose(E, mu, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("S", [1, 3, 4, 7])
def test_stratified_per_stratum_expectation(oracle_lib, S):
    """E over each stratum from the oracle's inverse CDF (one threshold swept
    over I_m) == the interval-overlap weights of the closed form; their mean
    over strata == AV."""
    rng = np.random.default_rng(20 + S)
    P = random_problem(oracle_lib, rng, 11, 5, spread=1.5)
    _, p = oracle_lib.scores(P, 0, 0)
    V = values_of(P, 0, 0)
    mu = oracle_lib.dense(P)[0, 0]
    F = np.cumsum(p)
    w = analysis.stratum_weights(p, S)
    total = np.zeros(V.shape[1])
    for m in range(S):
        lo, hi = m / S, (m + 1) / S
        cuts = np.unique(np.concatenate([[lo, hi], F[(F > lo) & (F < hi)]]))
        Em = np.zeros(V.shape[1])
        for a, b in zip(cuts[:-1], cuts[1:]):
            Em += oracle_lib.sample_head(P, 0, 0, np.array([0.5 * (a + b)]))[0] * (b - a) * S
        np.testing.assert_allclose(Em, w[m] @ V, rtol=1e-11, atol=1e-12)
        total += Em
    np.testing.assert_allclose(total / S, mu, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(analysis.stratified_mean(p, V, S), mu, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# statistics over the Philox stream: mean, variance, dominance, tail
# ---------------------------------------------------------------------------

def _seed_estimates(oracle_lib, P, variant, S, n_seeds):
    return np.stack([oracle_lib.decode(P, variant, S, seed=s)[0][0, 0] for s in range(n_seeds)])


@pytest.mark.parametrize("variant", ["iid", "stratified", "systematic"])
def test_mean_over_seeds_within_4_sigma(oracle_lib, variant):
    rng = np.random.default_rng(30)
    P = random_problem(oracle_lib, rng, 200, 8, spread=1.0)
    _, p = oracle_lib.scores(P, 0, 0)
    V = values_of(P, 0, 0)
    S, R = 16, 3000
    E = _seed_estimates(oracle_lib, P, variant, S, R)
    mu = oracle_lib.dense(P)[0, 0]
    if variant == "iid":
        var = analysis.iid_coordinate_variance(p, V, S)
    elif variant == "stratified":
        var = analysis.stratified_coordinate_variance(p, V, S)
    else:
        var = analysis.systematic_coordinate_variance(p, V, S)
        # the exact integral agrees with the replicate estimate (App. M)
        np.testing.assert_allclose(E.var(axis=0, ddof=1), var, rtol=0.15)
    sigma = np.sqrt(np.maximum(var, 1e-14) / R)
    assert np.all(np.abs(E.mean(axis=0) - mu) <= 4.0 * sigma)


@pytest.mark.parametrize("S", [1, 2, 5, 16])
def test_systematic_variance_is_the_integral_over_the_oracle_sampler(oracle_lib, S):
    """The exact systematic variance (float CDF, vectorised) equals the
    integral over u of the squared deviation of the oracle's own sampler
    (fixed-point thresholds, Sec. 2.1 / App. A.4), piece by piece."""
    rng = np.random.default_rng(60 + S)
    P = random_problem(oracle_lib, rng, 23, 5, spread=1.5)
    _, p = oracle_lib.scores(P, 0, 0)
    V = values_of(P, 0, 0)
    mu = oracle_lib.dense(P)[0, 0]

    def sq_dev(u):
        est = oracle_lib.sample_head(P, 0, 0, (np.arange(S) + u) / S)[0]
        return (est - mu) ** 2

    want = analysis.expectation_over_offset(sq_dev, analysis.systematic_breakpoints(p, S))
    np.testing.assert_allclose(analysis.systematic_coordinate_variance(p, V, S), want, rtol=1e-8, atol=1e-14)


def test_systematic_variance_special_cases():
    """S = 1 is one inverse-CDF draw from a uniform: the single-draw variance
    sum_n p_n V_n^2 - mu^2.  When every S p_n is an integer each key is drawn
    exactly S p_n times whatever u: variance zero.  Equal V rows: zero."""
    rng = np.random.default_rng(61)
    p = rng.dirichlet(np.ones(40))
    V = rng.standard_normal((40, 7)) * 2.0 + 1.0
    np.testing.assert_allclose(analysis.systematic_coordinate_variance(p, V, 1),
                               analysis.iid_coordinate_variance(p, V, 1), rtol=1e-10)
    q = np.array([2, 1, 0, 5, 3, 5], np.float64) / 16.0
    Vq = rng.standard_normal((6, 4))
    assert np.abs(analysis.systematic_coordinate_variance(q, Vq, 16)).max() < 1e-20
    assert np.abs(analysis.systematic_coordinate_variance(p, np.tile(V[3], (40, 1)), 9)).max() < 1e-20
    # an average of S draws whose thresholds are uniform on the strata: by
    # Cauchy-Schwarz and the law of total variance it varies no more than a
    # single draw (and, for generic p, more than not at all)
    v_sys = analysis.systematic_coordinate_variance(p, V, 8)
    assert np.all(v_sys > 0) and np.all(v_sys <= analysis.iid_coordinate_variance(p, V, 1))


def test_closed_form_variances_special_cases():
    """Identities the closed forms must meet whatever the data: with all V
    rows equal every estimate is that row, so every variance is zero (App. A:
    the estimators average rows of V); a trace is the sum of the per-coordinate
    variances; the App. M replicate estimator is numpy's unbiased variance
    (ddof = 1) summed over coordinates."""
    rng = np.random.default_rng(40)
    p = rng.dirichlet(np.ones(30))
    row = rng.standard_normal(6) * 5.0 + 10.0
    V_eq = np.tile(row, (30, 1))
    V = rng.standard_normal((30, 6)) + 3.0
    for S in (1, 7, 32):
        assert abs(analysis.iid_variance_trace(p, V_eq, S)) < 1e-10
        assert np.abs(analysis.iid_coordinate_variance(p, V_eq, S)).max() < 1e-10
        assert abs(analysis.stratified_variance_trace(p, V_eq, S)) < 1e-10
        assert np.abs(analysis.stratified_coordinate_variance(p, V_eq, S)).max() < 1e-10
        np.testing.assert_allclose(analysis.iid_coordinate_variance(p, V, S).sum(),
                                   analysis.iid_variance_trace(p, V, S), rtol=1e-12)
        np.testing.assert_allclose(analysis.stratified_coordinate_variance(p, V, S).sum(),
                                   analysis.stratified_variance_trace(p, V, S), rtol=1e-12)
    E = rng.standard_normal((9, 6))
    np.testing.assert_allclose(analysis.replicate_variance_trace(E), np.var(E, axis=0, ddof=1).sum(), rtol=1e-13)


@pytest.mark.parametrize("variant", ["iid", "stratified"])
def test_empirical_variance_matches_closed_form(oracle_lib, variant):
    rng = np.random.default_rng(31)
    P = random_problem(oracle_lib, rng, 150, 6, spread=1.2)
    _, p = oracle_lib.scores(P, 0, 0)
    V = values_of(P, 0, 0)
    S, R = 8, 4000
    E = _seed_estimates(oracle_lib, P, variant, S, R)
    emp = analysis.replicate_variance_trace(E)
    closed = (analysis.iid_variance_trace(p, V, S) if variant == "iid"
              else analysis.stratified_variance_trace(p, V, S))
    # the trace estimate over R replicates has relative s.d. below ~sqrt(2/R)*few
    assert abs(emp / closed - 1.0) < 6.0 * np.sqrt(2.0 / R)


def test_stratified_variance_never_exceeds_iid(oracle_lib):
    """Thm. A.6 / Cor. A.7 on the closed forms, and the ordering seen empirically."""
    rng = np.random.default_rng(32)
    for trial in range(20):
        P = random_problem(oracle_lib, rng, int(rng.integers(5, 300)), 4, spread=float(rng.uniform(0.1, 3)))
        _, p = oracle_lib.scores(P, 0, 0)
        V = values_of(P, 0, 0)
        for S in (1, 2, 5, 16, 64):
            assert (analysis.stratified_variance_trace(p, V, S)
                    <= analysis.iid_variance_trace(p, V, S) * (1 + 1e-12) + 1e-15)
    P = random_problem(oracle_lib, rng, 120, 6, spread=1.0)
    S, R = 8, 1500
    v = {var: analysis.replicate_variance_trace(_seed_estimates(oracle_lib, P, var, S, R))
         for var in ("iid", "stratified", "systematic")}
    assert v["stratified"] < v["iid"] and v["systematic"] < v["iid"]


def test_sampling_count_invariants(oracle_lib):
    """Systematic counts are floor/ceil(S p_n); stratified within +-1 of them;
    all counts sum to S; zero-mass keys never drawn."""
    rng = np.random.default_rng(33)
    P = random_problem(oracle_lib, rng, 300, 8, spread=2.5)
    _, p = oracle_lib.scores(P, 0, 0)
    S = 64
    lo, hi = analysis.systematic_count_bounds(p, S)
    for seed in range(200):
        _, Js, _ = oracle_lib.decode(P, "systematic", S, seed=seed)
        c = np.bincount(Js[0, 0], minlength=300)
        assert c.sum() == S
        assert np.all(c >= lo - 1e-9) and np.all(c <= hi + 1e-9)
        _, Jt, _ = oracle_lib.decode(P, "stratified", S, seed=seed)
        c = np.bincount(Jt[0, 0], minlength=300)
        assert c.sum() == S
        assert np.all(c >= np.maximum(0, lo - 1)) and np.all(c <= hi + 1)
        assert np.all(np.diff(Js[0, 0]) >= 0) and np.all(np.diff(Jt[0, 0]) >= 0)


def test_iid_bernstein_tail(oracle_lib):
    """App. B, Thm. B.1: the error norm exceeds the delta-radius at most a
    delta fraction of the time (checked with a binomial margin)."""
    rng = np.random.default_rng(34)
    P = random_problem(oracle_lib, rng, 100, 8, spread=1.0)
    _, p = oracle_lib.scores(P, 0, 0)
    V = values_of(P, 0, 0)
    mu = oracle_lib.dense(P)[0, 0]
    v = analysis.iid_variance_trace(p, V, 1)
    vmax = float(np.max(np.linalg.norm(V - mu, axis=1)))
    S, R, delta = 16, 2000, 0.05
    r = analysis.bernstein_radius(v, vmax, S, delta)
    E = _seed_estimates(oracle_lib, P, "iid", S, R)
    frac = np.mean(np.linalg.norm(E - mu, axis=1) >= r)
    assert frac <= delta + 3 * np.sqrt(delta * (1 - delta) / R)


def test_decode_layout_ragged_and_padding(oracle_lib):
    """Per-sequence budgets: rows beyond S_b are -1; each head equals a
    single-head call."""
    wl = synth.Workload("r", 3, 4, 2, 32, 200, "bf16", 24, "stratified", ragged=(50, 200))
    inp = synth.generate(wl, 9)
    Sp = np.array([24, 5, 13], np.int32)
    P = oracle_lib.Problem.from_inputs(inp)
    est, J, delta = oracle_lib.decode(P, "stratified", 24, seed=4, S_per_seq=Sp)
    for b in range(3):
        for h in range(4):
            e1, J1, d1 = oracle_lib.decode_head(P, "stratified", int(Sp[b]), 4, b, h)
            np.testing.assert_array_equal(J[b, h, :Sp[b]], J1)
            np.testing.assert_array_equal(est[b, h], e1)
            assert np.all(J[b, h, Sp[b]:] == -1)
            assert J1.max() < inp.nk_per_seq[b]


# ---------------------------------------------------------------------------
# tile samplers: S2ANTA-prop (App. O, Alg. 2-5) and S2ANTA-flash (App. P,
# Alg. 6-8)
# ---------------------------------------------------------------------------

def test_prop_budgets_worked_examples(oracle_lib):
    """Largest remainder (App. O, Alg. 4), cases worked by hand."""
    g = json.load(open(os.path.join(HERE, "golden", "prop_budgets.json")))
    for case in g["cases"]:
        got = oracle_lib.prop_budgets(np.array(case["W"], np.float64), case["S"])
        assert got.tolist() == case["budgets"], case


@pytest.mark.parametrize("seed", range(6))
def test_prop_budgets_brute_force(oracle_lib, seed):
    """Among all vectors with S_t in {floor q_t, floor q_t + 1} summing to S,
    the allocation puts the extra samples on the largest fractional parts:
    it maximises the sum of the chosen fractional parts (searched over every
    subset), and |S_t - q_t| < 1, sum S_t = S."""
    import itertools
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(2, 7))
    S = int(rng.integers(1, 13))
    W = rng.exponential(size=T) * (rng.random(T) > 0.2)
    W[0] += 0.1
    q = S * W / W.sum()
    fl = np.floor(q).astype(int)
    R = S - fl.sum()
    fr = q - fl
    best = max(itertools.combinations(range(T), R), key=lambda c: (sum(fr[list(c)]), [-i for i in c]))
    want = fl.copy()
    want[list(best)] += 1
    got = oracle_lib.prop_budgets(W, S)
    assert got.sum() == S and np.all(np.abs(got - q) < 1.0)
    assert got.tolist() == want.tolist()


def _tile_x_prefixes(P, b, h, tile_len, budgets):
    """Per tile, the running sums of x_n = budget_t exp(s_n - m_t) / l_t (the
    quantities of App. O, Alg. 5), from the pinned scores."""
    s, _ = oracle_lib_scores(P, b, h)
    out = []
    for t in range(-(-len(s) // tile_len)):
        st = s[t * tile_len:(t + 1) * tile_len]
        u = np.exp(st - st.max())
        x = budgets[t] * u / u.sum()
        out.append(np.concatenate([[0.0], np.cumsum(x)]))
    return out


def oracle_lib_scores(P, b, h):
    import oracle
    return oracle.scores(P, b, h)


def _offset_breakpoints(prefixes):
    """Common offsets a0 in [0, 1) at which a0 + (a running sum) is an integer:
    between them every tile's systematic counts are constant."""
    pts = [np.mod(-pr, 1.0) for pr in prefixes]
    return np.unique(np.concatenate([[0.0, 1.0]] + pts))


@pytest.mark.parametrize("nk,tile_len,S", [(40, 16, 6), (37, 8, 11), (64, 64, 5)])
def test_flash_exact_expectation_is_attention(oracle_lib, nk, tile_len, S):
    """App. P, Alg. 8: with W_t / Z weights and E[c_n] = S_tile u_n / l_t, the
    merged estimate's expectation over the tile offsets is softmax . V
    exactly.  Integrated piece by piece over a common offset a0."""
    rng = np.random.default_rng(nk + S)
    P = random_problem(oracle_lib, rng, nk, 6, spread=1.0)
    T = -(-nk // tile_len)
    _, _, _, St = oracle_lib.tiled_head(P, 0, 0, "flash", S, tile_len, seed=0)
    assert np.all(St == max(1, int(np.floor(S / T + 0.5))))
    bps = _offset_breakpoints(_tile_x_prefixes(P, 0, 0, tile_len, St))
    E = analysis.expectation_over_offset(
        lambda a: oracle_lib.tiled_head(P, 0, 0, "flash", S, tile_len, seed=0, a0=np.full(T, a))[0], bps)
    np.testing.assert_allclose(E, oracle_lib.dense(P)[0, 0], rtol=1e-10, atol=1e-11)


@pytest.mark.parametrize("nk,tile_len,S", [(40, 16, 6), (37, 8, 11), (50, 10, 3)])
def test_prop_exact_expectation_is_budget_mixture(oracle_lib, nk, tile_len, S):
    """App. O, Alg. 2: E[c_n] = S_t u_n / l_t inside tile t, so the estimate's
    expectation is sum_t (S_t / S) sum_n (u_n / l_t) V_n, the tile
    distributions mixed by the integer budgets."""
    rng = np.random.default_rng(7 * nk + S)
    P = random_problem(oracle_lib, rng, nk, 5, spread=1.0)
    T = -(-nk // tile_len)
    _, _, _, St = oracle_lib.tiled_head(P, 0, 0, "prop", S, tile_len, seed=0)
    s, _ = oracle_lib.scores(P, 0, 0)
    V = values_of(P, 0, 0)
    want = np.zeros(V.shape[1])
    for t in range(T):
        st = s[t * tile_len:(t + 1) * tile_len]
        u = np.exp(st - st.max())
        want += St[t] / S * (u / u.sum()) @ V[t * tile_len:(t + 1) * tile_len]
    bps = _offset_breakpoints(_tile_x_prefixes(P, 0, 0, tile_len, St))
    E = analysis.expectation_over_offset(
        lambda a: oracle_lib.tiled_head(P, 0, 0, "prop", S, tile_len, seed=0, a0=np.full(T, a))[0], bps)
    np.testing.assert_allclose(E, want, rtol=1e-10, atol=1e-11)


def test_prop_proportional_budgets_are_unbiased_and_uniform_visits_every_key(oracle_lib):
    """Equal tiles under uniform attention: S_t = S / T exactly, so prop is
    unbiased; with S = nk every key is drawn exactly once whatever a0, giving
    mean(V) = softmax . V."""
    rng = np.random.default_rng(3)
    nk, d, L = 64, 8, 16
    V = rng.standard_normal((nk, 1, d)).astype(np.float32)
    P = make_problem(oracle_lib, rng.standard_normal((1, d)), np.zeros((nk, 1, d)), V)
    dense = oracle_lib.dense(P)[0, 0]
    for a in (0.0, 0.3, 0.999):
        est, counts, _, St = oracle_lib.tiled_head(P, 0, 0, "prop", nk, L, seed=0, a0=np.full(4, a))
        assert St.tolist() == [16] * 4 and np.all(counts == 1)
        np.testing.assert_allclose(est, dense, rtol=1e-12, atol=1e-13)
    _, _, _, St = oracle_lib.tiled_head(P, 0, 0, "prop", 8, L, seed=0)
    assert St.tolist() == [2] * 4


@pytest.mark.parametrize("sampler", ["prop", "flash"])
def test_tile_counts_sum_to_budgets(oracle_lib, sampler):
    """Alg. 5 / Alg. 7: the counts of tile t add up to its budget (the x of
    a tile sum to it), zero-budget tiles draw nothing."""
    rng = np.random.default_rng(5)
    nk, L, S = 300, 32, 17
    P = random_problem(oracle_lib, rng, nk, 8, spread=2.5)
    for seed in range(5):
        _, counts, _, St = oracle_lib.tiled_head(P, 0, 0, sampler, S, L, seed=seed)
        per_tile = np.add.reduceat(counts, np.arange(0, nk, L))
        assert per_tile.tolist() == St.tolist()
        if sampler == "prop":
            assert St.sum() == S


@pytest.mark.parametrize("sampler", ["prop", "flash"])
def test_tile_count_rule_on_exact_interval_ends(oracle_lib, sampler):
    """Alg. 5 / Alg. 7 by hand: c_n = floor(a0 + p + x) - floor(a0 + p) gives
    key n the integers in (a0 + p, a0 + p + x], open on the left.  One tile of
    four keys with equal scores (u_n = 1, l = 4) and budget 2 has x = 1/2,
    so every interval end is a multiple of 1/2: a0 = 0 draws keys 1 and 3,
    a0 = 1/2 keys 0 and 2."""
    V = np.arange(8, dtype=np.float32).reshape(4, 1, 2)
    P = make_problem(oracle_lib, np.ones((1, 2)), np.zeros((4, 1, 2)), V)
    for a, want in ((0.0, [0, 1, 0, 1]), (0.5, [1, 0, 1, 0])):
        est, counts, _, St = oracle_lib.tiled_head(P, 0, 0, sampler, 2, 4, seed=0, a0=np.array([a]))
        assert St.tolist() == [2] and counts.tolist() == want, (a, counts)
        np.testing.assert_allclose(est, V[np.nonzero(want)[0], 0].astype(np.float64).mean(axis=0), rtol=1e-15)


def test_tile_boundary_distances_by_hand(oracle_lib):
    """The tile samplers' boundary distance: for a key that draws, the
    distance from its interval ends (a0 + p, a0 + p + x] to the nearest
    integer inside, in probability units (x units times W_t / (Z S_t)).
    Two tiles of four equal-score keys, the second tile's scores ln 3 higher
    (W = 4, 12: W/Z = 1/4, 3/4), flash with S = 4 (S_tile = 2, x = 1/2) and
    a0 = 0.1: keys 1 and 3 of each tile draw once, 0.1 x-units from an end."""
    q = np.ones((1, 1), np.float32)
    K = np.zeros((8, 1, 1), np.float32)
    K[4:, 0, 0] = np.float32(np.log(3.0))
    V = np.arange(8, dtype=np.float32).reshape(8, 1, 1)
    P = make_problem(oracle_lib, q, K, V, scale=1.0)
    _, counts, delta, St = oracle_lib.tiled_head(P, 0, 0, "flash", 4, 4, seed=0, a0=np.array([0.1, 0.1]))
    assert St.tolist() == [2, 2] and counts.tolist() == [0, 1, 0, 1, 0, 1, 0, 1]
    np.testing.assert_allclose(delta, [-1, 0.0125, -1, 0.0125, -1, 0.0375, -1, 0.0375], rtol=1e-5)


def test_tile_offsets_come_from_the_heads_philox_stream(oracle_lib, torch_philox):
    """a0 of tile t is uniform number t of head (b, h) (the Philox layout of
    the global samplers; the pages draw a0 ~ U[0, 1) per tile and name no
    generator): drawing with a0 = None equals passing those uniforms, taken
    here from PyTorch's Philox engine."""
    rng = np.random.default_rng(30)
    P = random_problem(oracle_lib, rng, 100, 8)
    seed, step, T = 11, 2, 7
    words = np.concatenate([torch_philox(seed, (step << 32) | 0, (0 << 32) | i) for i in range(2)])
    a0 = (words[:T] >> 8).astype(np.float64) / 2.0 ** 24
    for sampler in ("prop", "flash"):
        e1, c1, _, _ = oracle_lib.tiled_head(P, 0, 0, sampler, 24, 16, seed=seed, step=step)
        e2, c2, _, _ = oracle_lib.tiled_head(P, 0, 0, sampler, 24, 16, seed=seed, step=step, a0=a0)
        np.testing.assert_array_equal(c1, c2)
        np.testing.assert_array_equal(e1, e2)


def test_flash_tile_budget_rounds_to_nearest(oracle_lib):
    """Alg. 6 gives every tile about S / T samples: the reading taken is
    S_tile = max(1, floor(S / T + 1/2)); three tiles of 16 keys."""
    rng = np.random.default_rng(8)
    P = random_problem(oracle_lib, rng, 48, 4)
    for S, want in ((1, 1), (4, 1), (5, 2), (7, 2), (8, 3)):
        _, counts, _, St = oracle_lib.tiled_head(P, 0, 0, "flash", S, 16, seed=1)
        assert St.tolist() == [want] * 3, (S, St)
        assert counts.sum() == 3 * want


@pytest.mark.parametrize("S,a", [(5, 0.37), (16, 0.0), (9, 0.9)])
def test_flash_single_tile_is_the_systematic_sampler(oracle_lib, S, a):
    """One tile covering all keys: the count rule of Alg. 7 is systematic
    sampling with thresholds (j + 1 - a0) / S, j = 0..S-1, read with intervals
    open on the left; away from interval ends it draws what the pinned
    inverse-CDF sampler draws, and the merge leaves (1/S) sum c_n V_n."""
    rng = np.random.default_rng(S)
    nk = 30
    P = random_problem(oracle_lib, rng, nk, 4, spread=1.5)
    est, counts, delta, St = oracle_lib.tiled_head(P, 0, 0, "flash", S, nk, seed=0, a0=np.array([a]))
    assert St.tolist() == [S]
    t = (np.arange(S) + 1.0 - a) / S
    _, J, dl = oracle_lib.sample_head(P, 0, 0, t[t < 1.0])
    ref = np.bincount(J, minlength=nk)
    if a == 0.0:   # the last threshold is 1: it falls on the last key
        ref[nk - 1] += 1
    assert np.all(counts == ref) or np.all((counts == ref) | (delta < 1e-9) | (np.roll(delta, 1) < 1e-9)
                                          | (np.roll(delta, -1) < 1e-9))
    np.testing.assert_allclose(est, counts @ values_of(P, 0, 0) / S, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# synthetic measurement pins: distinct keys and prefill coverage (App. F,
# Table 9; App. L, Table 17; App. D, Fig. 7; App. M)
# ---------------------------------------------------------------------------

def _gaussian_fp16(rng, n, d):
    return rng.standard_normal((n, d)).astype(np.float16).astype(np.float64)


def test_causal_softmax_rows_match_scipy():
    """The causal prefill attention of App. F: query i attends to keys 0..i
    only; each row equals scipy's softmax over those keys, zero beyond."""
    from scipy.special import softmax
    rng = np.random.default_rng(41)
    q, k = rng.standard_normal((12, 8)), rng.standard_normal((12, 8))
    P = analysis.causal_softmax(q, k, 0.5)
    s = q @ k.T * 0.5
    for i in range(12):
        np.testing.assert_allclose(P[i, :i + 1], softmax(s[i, :i + 1]), rtol=1e-13, atol=1e-15)
        assert np.all(P[i, i + 1:] == 0.0)


def test_prefill_coverage_reproduces_table9(oracle_lib):
    """App. F, Table 9: share of V rows a causal prefill pass of i.i.d. SANTA
    reads, Gaussian fp16 Q, K, d = 128, from the exact causal softmax; within
    0.3 percentage points of the printed means."""
    g = json.load(open(os.path.join(HERE, "golden", "table9_prefill_coverage.json")))
    rng = np.random.default_rng(9)
    for col, nk in enumerate(g["nk"][:2]):
        Ps = [analysis.causal_softmax(_gaussian_fp16(rng, nk, 128), _gaussian_fp16(rng, nk, 128), 128 ** -0.5)
              for _ in range(3)]
        for S in g["S"]:
            got = 100.0 * np.mean([analysis.prefill_coverage_iid(P, S) for P in Ps])
            want = g["percent"][str(S)][col]
            assert abs(got - want) < 0.3, (nk, S, got, want)


def test_prefill_coverage_closed_form_matches_the_sampler(oracle_lib):
    """The closed form against the oracle's own i.i.d. sampler (Philox
    uniforms, inverse CDF): union of the draws of every query of a causal pass."""
    rng = np.random.default_rng(4)
    nk, d, S = 192, 16, 4
    q = rng.standard_normal((nk, d)).astype(np.float32)
    k = rng.standard_normal((nk, d)).astype(np.float32)
    V = rng.standard_normal((nk, 1, d)).astype(np.float32)
    want = analysis.prefill_coverage_iid(analysis.causal_softmax(q, k, d ** -0.5), S)
    shares = []
    for seed in range(12):
        seen = np.zeros(nk, bool)
        for i in range(nk):
            P = make_problem(oracle_lib, q[i:i + 1], k[:i + 1, None, :], V[:i + 1])
            _, J, _ = oracle_lib.sample_head(P, 0, 0, oracle_lib.thresholds("iid", S, seed, 0, i))
            seen[J] = True
        shares.append(seen.mean())
    assert abs(np.mean(shares) - want) < 4 * np.std(shares) / np.sqrt(len(shares)) + 0.01


def test_unique_keys_iid_closed_form_matches_the_sampler(oracle_lib):
    """App. M.1 (1): E|U| = sum_n 1 - (1 - p_n)^S for i.i.d. draws."""
    rng = np.random.default_rng(6)
    P = random_problem(oracle_lib, rng, 400, 16, spread=2.0)
    _, p = oracle_lib.scores(P, 0, 0)
    for S in (8, 64):
        want = analysis.expected_unique_keys_iid(p, S)
        got = [np.unique(oracle_lib.decode(P, "iid", S, seed=s)[1][0, 0]).size for s in range(200)]
        assert abs(np.mean(got) - want) < 4 * np.std(got) / np.sqrt(len(got)) + 1e-9, (S, np.mean(got), want)


@pytest.mark.parametrize("variant", ["stratified", "systematic"])
def test_unique_keys_closed_forms_match_the_sampler(oracle_lib, variant):
    """E|U| for the stratified sampler, sum_n 1 - prod_m (1 - w[m, n]), and
    for the systematic one, sum_n min(1, S p_n), against the oracle's own
    sampler averaged over Philox seeds."""
    rng = np.random.default_rng(7)
    P = random_problem(oracle_lib, rng, 300, 16, spread=2.0)
    _, p = oracle_lib.scores(P, 0, 0)
    f = analysis.expected_unique_keys_stratified if variant == "stratified" else analysis.expected_unique_keys_systematic
    for S in (8, 64):
        want = f(p, S)
        got = [np.unique(oracle_lib.decode(P, variant, S, seed=s)[1][0, 0]).size for s in range(300)]
        assert abs(np.mean(got) - want) < 4 * np.std(got) / np.sqrt(len(got)) + 0.02, (S, np.mean(got), want)


def test_unique_keys_closed_forms_special_cases():
    """S = 1: one key, whatever the sampler.  S p_n integers: the stratified
    and systematic samplers draw every key of positive mass (S p_n times).
    Uniform p over nk = S keys: every key exactly once for both, while S
    i.i.d. draws miss a share (1 - 1/S)^S of them."""
    rng = np.random.default_rng(8)
    p = rng.dirichlet(np.ones(50))
    for f in (analysis.expected_unique_keys_iid, analysis.expected_unique_keys_stratified,
              analysis.expected_unique_keys_systematic):
        assert abs(f(p, 1) - 1.0) < 1e-12
    q = np.array([2, 1, 0, 5, 3, 5], np.float64) / 16.0
    assert abs(analysis.expected_unique_keys_systematic(q, 16) - 5.0) < 1e-12
    assert abs(analysis.expected_unique_keys_stratified(q, 16) - 5.0) < 1e-12
    u = np.full(32, 1.0 / 32)
    assert abs(analysis.expected_unique_keys_systematic(u, 32) - 32.0) < 1e-9
    assert abs(analysis.expected_unique_keys_stratified(u, 32) - 32.0) < 1e-9
    assert abs(analysis.expected_unique_keys_iid(u, 32) - 32.0 * (1.0 - (31.0 / 32.0) ** 32)) < 1e-9


def _decode_head_8k():
    """One synthetic decode head of the Llama shape at 8K keys (planted keys as
    in the benchmark inputs), as an oracle problem."""
    import oracle
    inp = synth.generate(synth.llama32k(8192, 256, "systematic"), 0)
    return oracle.Problem.from_inputs(inp)


def test_stratified_variants_draw_more_distinct_keys(oracle_lib):
    """App. L, Table 17 (model attention there; a synthetic 8K decode head
    here): for each S the stratified and systematic samplers touch more
    distinct keys than i.i.d. SANTA, and fewer than S."""
    P = _decode_head_8k()
    rows = []
    for S in (32, 64, 128, 256):
        U = {}
        for variant in ("iid", "stratified", "systematic"):
            _, J, _ = oracle_lib.decode(P, variant, S, seed=1)
            U[variant] = np.mean([np.unique(J[0, h]).size for h in range(J.shape[1])])
        rows.append((S, U["iid"], U["stratified"], U["systematic"]))
        assert U["iid"] < U["stratified"] <= S and U["iid"] < U["systematic"] <= S, (S, U)
    print("\nS, mean distinct keys per head: i.i.d., stratified, systematic")
    for r in rows:
        print("  %4d  %7.1f  %7.1f  %7.1f" % r)


def test_variance_falls_with_S_and_stratification_helps(oracle_lib):
    """App. D, Fig. 7 (model attention there; a synthetic 8K decode head here):
    variance traces against S -- i.i.d. closed form (slope -1 on log-log),
    stratified closed form, systematic by replicates (App. M) -- with
    stratified and systematic below i.i.d. at every S (Thm. A.6 for
    stratified; empirical for systematic)."""
    P = _decode_head_8k()
    _, p = oracle_lib.scores(P, 0, 0)
    V = values_of(P, 0, 0)
    mu = p @ V
    Ss = np.array([32, 64, 128, 256])
    vi, vs, vy = [], [], []
    rng = np.random.default_rng(2)
    for S in Ss:
        vi.append(analysis.iid_variance_trace(p, V, int(S)))
        vs.append(analysis.stratified_variance_trace(p, V, int(S)))
        reps = [oracle_lib.sample_head(P, 0, 0, (np.arange(S) + u) / S)[0] for u in rng.random(48)]
        vy.append(analysis.replicate_variance_trace(np.array(reps)))
    slope = lambda v: float(np.polyfit(np.log(Ss), np.log(v), 1)[0])
    assert abs(slope(vi) + 1.0) < 1e-9
    assert np.all(np.array(vs) < np.array(vi)) and np.all(np.array(vy) < np.array(vi))
    print("\nslopes of log variance trace against log S: i.i.d. %.2f, stratified %.2f, systematic %.2f"
          % (slope(vi), slope(vs), slope(vy)))


# ---------------------------------------------------------------------------
# Bernoulli qK^T, mean group query (App. C, Eq. 8-13; Fig. 6)
# ---------------------------------------------------------------------------

def test_storage_rounding_matches_numpy(oracle_lib):
    """fp32 -> fp16 / bf16 round to nearest even, against numpy's float16 cast
    and a bf16 rounding written from the bit layout in synth."""
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-9, 5, 2000),
                         [0.0, -0.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 1e-30]])
    xs = xs.astype(np.float32)
    with np.errstate(over="ignore"):
        want16 = xs.astype(np.float16).view(np.uint16)
    got16 = np.array([oracle_lib.store_elem("fp16", float(x)) for x in xs], np.uint16)
    np.testing.assert_array_equal(got16, want16)
    gotb = np.array([oracle_lib.store_elem("bf16", float(x)) for x in xs], np.uint16)
    np.testing.assert_array_equal(gotb, synth.f32_to_bf16_bits(xs))
    # exact halfway cases (bf16 keeps 8 significant bits, fp16 11), against
    # PyTorch's conversions, which round to nearest even
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3 + 2.0 ** -7, 1 + 2.0 ** -11,
                     1 + 3 * 2.0 ** -11, 2.0 ** -24 * 1.5, 2.0 ** -24 * 2.5], np.float32)
    tb = torch.from_numpy(ties).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    th = torch.from_numpy(ties).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal([oracle_lib.store_elem("bf16", float(x)) for x in ties], tb)
    np.testing.assert_array_equal([oracle_lib.store_elem("fp16", float(x)) for x in ties], th)


def _bern_problem(oracle_lib, rng, G=4, d=128, nk=64, dtype="fp32"):
    q = rng.standard_normal((1, G, d)).astype(np.float32)
    K = rng.standard_normal((nk, 1, d)).astype(np.float32)
    V = rng.standard_normal((nk, 1, d)).astype(np.float32)
    return oracle_lib.Problem(q, K, V, np.array([0, nk], np.int64), dtype, 1)


@pytest.mark.parametrize("stratified", [False, True])
def test_bernoulli_counts_law(oracle_lib, stratified):
    """Eq. (11)-(12): the ones per feature over B samples have mean B p_i with
    p_i = m_i / max m (so m^ is unbiased, Eq. 12, and q~ is unbiased for q,
    Eq. 13); plain sampling is Binomial(B, p_i), stratified sampling takes only
    floor(B p_i) or floor(B p_i) + 1."""
    rng = np.random.default_rng(11)
    P = _bern_problem(oracle_lib, rng)
    m = np.abs(P.q[0].astype(np.float64)).mean(axis=0)
    p = m / m.max()
    Bs = 4
    C = np.array([oracle_lib.bernoulli_group(P, 0, 0, Bs, stratified, seed)[1] for seed in range(600)])
    mean, var = C.mean(axis=0), C.var(axis=0)
    f = Bs * p - np.floor(Bs * p)
    law_var = f * (1 - f) if stratified else Bs * p * (1 - p)   # variance of the count under the stated law
    se = np.sqrt(law_var / C.shape[0])
    assert np.all(np.abs(mean - Bs * p) < 5 * se + 0.01)
    if stratified:
        fl = np.floor(Bs * p)
        assert np.all((C == fl) | (C == fl + 1))
    else:
        assert np.all(np.abs(var - Bs * p * (1 - p)) < 0.25 + 0.35 * Bs * p * (1 - p))
    assert np.all(C[:, np.argmax(m)] == Bs)   # the largest feature has p = 1


@pytest.mark.parametrize("stratified", [False, True])
def test_bernoulli_draws_use_their_own_philox_stream_and_a_strict_test(oracle_lib, torch_philox, stratified):
    """Eq. 11 draws b ~ Bernoulli(p) as a24 < p 2^24 with a24 the top 24 bits
    of a Philox word: for p 2^24 an integer that is probability p exactly
    (a non-strict test would add 2^-24).  Sample n of feature i in group
    (b, kvh) takes word r % 4, r = n d + i, of the block at counter
    (r / 4, H + kvh, b, step), here from PyTorch's Philox engine.  With
    G = 1, fp32 queries and one feature at |q| = 1 (so norm = 1), feature i
    is given p_i = a24_i / 2^24 (no draw) or (a24_i + 1) / 2^24 (one draw).
    With one sample the stratified rule (n + u)/B < p (App. C.1) is the same
    test."""
    seed, step, b, kvh, H, d = 77, 3, 1, 1, 2, 64
    words = np.concatenate([torch_philox(seed, (step << 32) | b, ((H + kvh) << 32) | i) for i in range(d // 4)])
    a24 = (words >> 8).astype(np.int64)
    rng = np.random.default_rng(4)
    hit = rng.integers(0, 2, d).astype(bool)
    hit[0] = True
    num = np.where(hit, a24 + 1, a24)
    num[0] = 1 << 24
    num = np.where(num == 0, 1, num)              # p = 0 would skip the feature
    hit = np.where((a24 == 0) & ~hit, True, hit)  # ...and a24 = 0 < 1 draws
    q = np.zeros((2, H, d), np.float32)
    q[b, kvh] = (num / 2.0 ** 24).astype(np.float32) * np.where(rng.integers(0, 2, d) == 1, 1, -1)
    q[b, 0] = rng.standard_normal(d).astype(np.float32)
    K = rng.standard_normal((8, H, d)).astype(np.float32)
    P = oracle_lib.Problem(q, K, K, np.array([0, 4, 8], np.int64), "fp32", H)
    _, counts = oracle_lib.bernoulli_group(P, b, kvh, 1, stratified, seed, step)
    np.testing.assert_array_equal(counts, hit.astype(np.int32))


def test_bernoulli_effective_query_is_unbiased(oracle_lib):
    """Eq. (13): E[q~] = q (averaged over seeds, fp32 storage)."""
    rng = np.random.default_rng(12)
    P = _bern_problem(oracle_lib, rng, G=2, d=64)
    Bs, N = 8, 400
    qs = np.array([oracle_lib.bernoulli_group(P, 0, 0, Bs, True, seed)[0] for seed in range(N)], np.float64)
    q = P.q[0].astype(np.float64)
    m = np.abs(q).mean(axis=0)
    f = np.mod(Bs * m / m.max(), 1.0)
    se = np.abs(q) * m.max() / (m * Bs) * np.sqrt(f * (1 - f) / N)   # q~ = (max m) (c / B) q / m
    assert np.all(np.abs(qs.mean(axis=0) - q) < 5 * se + 1e-6 * np.abs(q) + 1e-9)


def test_bernoulli_score_error_reproduces_fig6(oracle_lib):
    """App. C.1, Fig. 6: relative L2 error of the Bernoulli scores for one query
    (d = 128, nk = 1024, q ~ N(0, 1), K ~ N(0, 1)/sqrt(d)), about 60% at B = 4
    for plain sampling and about 30% for stratified; plain falls like
    B^-1/2 and stratified like B^-1."""
    rng = np.random.default_rng(13)
    d, nk, n_inst = 128, 1024, 40
    err = {False: {}, True: {}}
    for B in (4, 16, 64):
        for strat in (False, True):
            e = []
            for inst in range(n_inst):
                q = rng.standard_normal((1, 1, d)).astype(np.float32)
                K = (rng.standard_normal((nk, 1, d)) / np.sqrt(d)).astype(np.float32)
                P = oracle_lib.Problem(q, K, K, np.array([0, nk], np.int64), "fp32", 1)
                qt, _ = oracle_lib.bernoulli_group(P, 0, 0, B, strat, seed=inst)
                s = K[:, 0].astype(np.float64) @ q[0, 0].astype(np.float64)
                sh = K[:, 0].astype(np.float64) @ qt[0].astype(np.float64)
                e.append(np.linalg.norm(sh - s) / np.linalg.norm(s))
            err[strat][B] = float(np.mean(e))
    assert 0.5 < err[False][4] < 0.7 and 0.2 < err[True][4] < 0.4, err
    slope = lambda d_: np.polyfit(np.log([4, 16, 64]), np.log([d_[4], d_[16], d_[64]]), 1)[0]
    assert abs(slope(err[False]) + 0.5) < 0.1 and abs(slope(err[True]) + 1.0) < 0.15, err
    print("\nBernoulli score error (B = 4, 16, 64): plain %s, stratified %s"
          % ([round(err[False][b], 3) for b in (4, 16, 64)], [round(err[True][b], 3) for b in (4, 16, 64)]))


def test_empty_sequence_is_rejected(oracle_lib):
    """A sequence with no keys has no softmax (Eq. 1 normalises over an empty
    set): the oracle refuses it rather than invent an output, for the
    whole-step decode and for a single head, and still serves the others."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 2, 64)).astype(np.float32)
    K = rng.standard_normal((40, 1, 64)).astype(np.float32)
    P = oracle_lib.Problem(q, K, K, np.array([0, 40, 40], np.int64), "fp32", 1)
    with pytest.raises(ValueError):
        oracle_lib.decode_head(P, "systematic", 4, 0, 1, 0)
    with pytest.raises(ValueError):
        oracle_lib.decode(P, "systematic", 4, 0)
    est, J, _ = oracle_lib.decode_head(P, "systematic", 4, 0, 0, 1)
    assert np.all((J >= 0) & (J < 40)) and np.all(np.isfinite(est))
