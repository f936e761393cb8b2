"""Pins of the oracle's selective refinement (StrataFlux paper, section 3
"Weight Refinement", Eq. 2 and "Channel selection"): hand-worked column records
and selections, selection against a rank-counting brute force, the zero
residual identity, and the closed-form error bound of a fully refined product."""
import numpy as np
import pytest

from oracle import lbq_oracle as O


def _bytes(tokens):
    return np.array([int(t, 16) for t in tokens], dtype=np.uint8)


def test_hand_worked_column_records(golden):
    g = golden("refine_column_example.txt")
    q0 = np.array([int(t) for t in g["col0_q_group0"]])
    R = np.zeros((64, 2), np.float32)
    R[:32, 0] = (q0 - 3) / 1024.0
    R[:, 1] = 0.5
    blob = O.pack_refine(R)
    cb = int(g["column_bytes"][0])
    assert O.refine_column_bytes(64) == cb and blob.size == int(g["total_bytes"][0])
    assert np.array_equal(blob[:64], _bytes(g["header"]))
    assert np.array_equal(blob[64:64 + cb], _bytes(g["col0_record"]))
    assert np.array_equal(blob[64 + cb:64 + 2 * cb], _bytes(g["col1_record"]))
    C = O.unpack_refine(blob)
    assert np.array_equal(C[:, 0], R[:, 0].astype(np.float64))     # exactly representable column
    assert np.array_equal(C[:, 1], np.zeros(64))                   # constant group -> 0


def test_hand_worked_selection(golden):
    g = golden("refine_column_example.txt")
    x = np.zeros(64, np.float16)
    for tok in g["select_x_nonzero"]:
        i, v = tok.split(":")
        x[int(i)] = float(v)
    for k in (2, 3, 4):
        want = [int(t) for t in g["select_k%d" % k]]
        assert O.select_refine(x, k).tolist() == want
    assert O.select_refine(x, 100).tolist() == list(range(64))


def _rank_select(x, k):
    """i is kept iff fewer than k channels of its chunk beat it (larger |x|, or equal
    |x| and a lower index): a definition by counting, independent of sorting."""
    a = np.abs(x.astype(np.float64))
    keep = []
    for c0 in range(0, a.size, 1024):
        c1 = min(a.size, c0 + 1024)
        for i in range(c0, c1):
            beat = sum(1 for j in range(c0, c1) if a[j] > a[i] or (a[j] == a[i] and j < i))
            if beat < k:
                keep.append(i)
    return keep


@pytest.mark.parametrize("K,k", [(64, 1), (1088, 5), (2048, 33), (1100, 80)])
def test_selection_matches_rank_counting(K, k):
    rng = np.random.default_rng(K + k)
    x = (rng.integers(-6, 7, size=K) * 0.5).astype(np.float16)   # many ties
    x[rng.choice(K, size=K // 3, replace=False)] = 0
    assert O.select_refine(x, k).tolist() == _rank_select(x, k)


def test_selection_ranks_non_finite_values_above_finite():
    """NaN above infinity above every finite |x| (the FP16 magnitude field's order);
    +inf and -inf tie, the lower channel first; finite values keep the |x| order."""
    x = np.zeros(2048, np.float16)
    x[10] = np.float16(60000.0)            # the largest finite magnitude present
    x[700] = np.float16(np.inf)
    x[33] = np.float16(-np.inf)
    x[900] = np.float16(np.nan)
    x[1500] = np.float16(-np.nan)
    x[1024 + 5] = np.float16(-3.0)
    x[1024 + 6] = np.float16(2.0)
    assert O.select_refine(x, 1).tolist() == [900, 1500]
    assert O.select_refine(x, 2).tolist() == [33, 900, 1029, 1500]
    assert O.select_refine(x, 3).tolist() == [33, 700, 900, 1029, 1030, 1500]
    assert O.select_refine(x, 4).tolist() == [10, 33, 700, 900, 1024, 1029, 1030, 1500]


def test_zero_residual_gives_zero_refinement():
    R = np.zeros((128, 5), np.float32)
    C = O.unpack_refine(O.pack_refine(R))
    assert np.array_equal(C, np.zeros((128, 5)))


def test_full_refinement_error_bound():
    """With every channel selected, y' - W x = (C - R) x, and per 32-row group of a
    column |C - R| <= s16 / 2 + 15 |s16 - s| (Proposition 2 with the stored FP16
    scale); the bound is computed from R directly, not from the packed bytes."""
    rng = np.random.default_rng(3)
    N, K = 128, 1088
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    base = O.pack_w4(W)
    R = (W - O.dequant_eff(base).astype(np.float32)).astype(np.float32)
    x = rng.standard_normal(K).astype(np.float16)
    ref_blob = O.pack_refine(R)
    idx = O.select_refine(x, 1024)
    assert idx.size == K
    y0 = O.gemv(base, x)
    y1 = O.refine_apply(ref_blob, x, idx, y0)
    xv = x.astype(np.float64)
    exact = (W.astype(np.float64) - O.dequant_eff(base) + O.dequant_eff(base)) @ xv
    Rg = R.astype(np.float64).T.reshape(K, N // 32, 32)
    s = np.maximum((Rg.max(2) - Rg.min(2)) / 15.0, 1e-8)
    s16 = O.fp16_round(s).astype(np.float64)
    err_col = (s16 / 2 + 15 * np.abs(s16 - s))                         # (K, N/32)
    bound = (np.abs(xv)[:, None, None] * np.repeat(err_col[:, :, None], 32, axis=2)).reshape(K, N).sum(0)
    assert np.all(np.abs(y1 - exact) <= bound * (1 + 1e-9) + 1e-12)
    # and the refined product is closer to W x than the base one
    assert np.linalg.norm(y1 - exact) < 0.5 * np.linalg.norm(y0 - exact)


def test_apply_is_the_selected_column_product():
    rng = np.random.default_rng(4)
    N, K = 64, 2048
    R = (rng.standard_normal((N, K)) * 1e-3).astype(np.float32)
    blob = O.pack_refine(R)
    x = rng.standard_normal(K).astype(np.float16)
    idx = O.select_refine(x, 7)
    assert idx.size == 14
    C = O.unpack_refine(blob)
    y = rng.standard_normal(N)
    ref = y + C[:, idx] @ x[idx].astype(np.float64)
    assert np.allclose(O.refine_apply(blob, x, idx, y), ref, rtol=0, atol=1e-12)
