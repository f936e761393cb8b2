"""Pins of outlier selection: SPECTRA Proposition 1 (kurtosis bound, the r bounds
printed for K = 1536 / 3072 / 8192 / 65536, the 3 % cap point), the top-n selection
rule by exhaustive comparison, and the otf-llm impact score on constructed inputs."""
import math

import numpy as np

from oracle import lbq_oracle as O


def test_prop1_kurtosis_bounded_by_width():
    rng = np.random.default_rng(0)
    for K in (8, 64, 1536):
        for _ in range(20):
            S = np.abs(rng.standard_cauchy(K))
            assert O.population_kurtosis(S) <= K


def test_prop1_extremal_vector_closed_form():
    # one spike among K-1 equal values: kappa = (K^2 - 3K + 3)/(K - 1) < K
    for K in (4, 100, 1536, 8192):
        S = np.ones(K)
        S[K // 3] = 7.0
        kappa = O.population_kurtosis(S)
        closed = (K * K - 3 * K + 3) / (K - 1)
        assert abs(kappa - closed) <= 1e-9 * closed
        assert kappa < K


def test_prop1_printed_ratio_bounds():
    """r <= 0.01 (1 + 0.15 ln(K - 2)) = 2.10 / 2.20 / 2.35 / 2.66 % (printed)."""
    for K, pct in ((1536, 2.10), (3072, 2.20), (8192, 2.35), (65536, 2.66)):
        assert round(O.outlier_ratio(K) * 100, 2) == pct
    assert O.outlier_ratio(0.0) == 0.01           # mesokurtic: r_base
    assert O.outlier_ratio(3.0) == 0.01
    # 3 % cap reached only once kappa exceeds ~6.2e5
    assert O.outlier_ratio(6.0e5) < 0.03
    assert O.outlier_ratio(6.4e5) == 0.03
    assert O.outlier_ratio(1e9) == 0.03


def test_top_indices_exhaustive():
    rng = np.random.default_rng(1)
    for _ in range(30):
        s = rng.integers(0, 6, size=40).astype(float)   # many ties
        n = int(rng.integers(0, 41))
        sel = O.top_indices(s, n)
        assert len(sel) == n and list(sel) == sorted(sel)
        chosen = set(sel.tolist())
        for j in chosen:
            for i in set(range(40)) - chosen:
                assert s[j] > s[i] or (s[j] == s[i] and j < i)


def test_select_outliers_w4_count_and_members():
    rng = np.random.default_rng(2)
    N, K = 64, 1536
    W = rng.standard_normal((N, K)).astype(np.float32)
    heavy = rng.choice(K, size=15, replace=False)
    W[:, heavy] *= 20
    S = np.sqrt((W.astype(np.float64) ** 2).sum(0))
    mu, sd = S.mean(), S.std()
    kappa = float((((S - mu) / sd) ** 4).mean())
    r = min(max(0.01 * (1 + 0.15 * math.log(1 + max(0.0, kappa - 3))), 0.005), 0.03)
    idx = O.select_outliers_w4(W)
    assert len(idx) == int(r * K)
    assert set(heavy.tolist()) <= set(idx.tolist())


def test_impact_score_constructed():
    # column c has norm (c+1) and mean |x| of 1/(c+1) except three boosted columns
    K, P = 64, 8
    W = np.zeros((4, K), np.float32)
    W[0] = np.arange(1, K + 1)
    X = np.tile((1.0 / np.arange(1, K + 1)).astype(np.float16), (P, 1))
    X[:, [5, 17, 40]] = np.float16(2.0)
    I = O.impact_scores(W, X)
    base = np.arange(1, K + 1) * (1.0 / np.arange(1, K + 1)).astype(np.float16).astype(np.float64)
    expect = base.copy()
    expect[[5, 17, 40]] = np.array([6, 18, 41]) * 2.0
    assert np.allclose(I, expect, rtol=1e-15, atol=0)
    sel = O.select_outliers_impact(W, X, frac=3 / 64 + 1e-9)
    assert sel.tolist() == [5, 17, 40]


def test_w2_outlier_count_reading():
    assert int(math.floor(O.W2_OUTLIER_FRAC * 4096)) == 143
    assert int(math.floor(O.W2_OUTLIER_FRAC * 14336)) == 501
