"""Pins of the oracle's 2-bit Lloyd-Max codebook quantiser (otf-llm 4.0.0, sections
2, 3 and 5): FP16 codebook bits, the hand-worked group, OLS against a least-squares
solve, nearest-centroid assignment by enumeration, crumb order, affine special case."""
import numpy as np

from oracle import lbq_oracle as O


def test_codebook_f16_bits_and_symmetry(golden):
    g = golden("w2_worked_example.txt")
    bits = O.CODEBOOK_F16.view("<u2").tolist()
    assert bits == [int(v, 16) for v in g["codebook_f16_bits"]]
    C = O.C16
    assert C[0] + C[3] == 0.0 and C[1] + C[2] == 0.0
    assert C.tolist() == [-1.51953125, -0.449951171875, 0.449951171875, 1.51953125]


def test_worked_group(golden):
    g = golden("w2_worked_example.txt")
    codes0 = [int(v) for v in g["codes_group0"]]
    w = np.empty((1, 64), np.float32)
    w[0, :32] = [O.C16[c] / 16 + 0.125 for c in codes0]
    w[0, 32:] = 0.25
    q, S, Z = O.quantise_w2(w)
    assert q[0, :32].tolist() == codes0
    assert q[0, 32:].tolist() == [int(v) for v in g["codes_group1"]]
    blob = O.pack_w2cb(w)
    rec = O.read_header(blob)["area"]            # row block 0, record 0, row 0
    assert blob[rec:rec + 16].tolist() == [int(v, 16) for v in g["code_bytes"]]
    assert blob[rec + 1024:rec + 1028].view("<u2").tolist() == [int(v, 16) for v in g["S_f16_bits"]]
    assert blob[rec + 1280:rec + 1284].view("<u2").tolist() == [int(v, 16) for v in g["Z_f16_bits"]]


def test_ols_matches_least_squares():
    rng = np.random.default_rng(5)
    Wg = rng.standard_normal((200, 32)) * 0.05 + rng.standard_normal((200, 1)) * 0.01
    q = rng.integers(0, 4, size=(200, 32)).astype(np.uint8)
    q[:, :4] = [0, 1, 2, 3]                       # every group uses several codes
    S, Z = O.ols_fit(Wg, q)
    for i in range(200):
        A = np.stack([O.C16[q[i]], np.ones(32)], axis=1)
        sol, *_ = np.linalg.lstsq(A, Wg[i], rcond=None)
        D = float(((O.C16[q[i]] - O.C16[q[i]].mean()) ** 2).sum())
        assert abs(S[i] - sol[0]) <= abs(sol[0]) * (2e-8 / D) + 1e-14
        assert abs(Z[i] - sol[1]) <= 1e-9 * (abs(sol[1]) + abs(sol[0]))


def test_ols_constant_group():
    Wg = np.full((1, 32), 0.375)
    q = O.assign_codes(Wg)
    S, Z = O.ols_fit(Wg, q)
    assert S[0] == 0.0 and Z[0] == 0.375


def test_assignment_is_nearest_centroid():
    rng = np.random.default_rng(9)
    Wg = rng.standard_normal((300, 32)) * rng.uniform(0.01, 2.0, size=(300, 1)) + rng.standard_normal((300, 1))
    q = O.assign_codes(Wg)
    for i in range(300):
        mu = sum(Wg[i]) / 32
        sd = (sum((w - mu) ** 2 for w in Wg[i]) / 32) ** 0.5
        for k in range(32):
            u = (Wg[i, k] - mu) / sd
            d = [abs(u - c) for c in O.C16]
            best = min(d)
            assert abs(d[q[i, k]] - best) <= 1e-12
            assert q[i, k] == min(c for c in range(4) if d[c] - best <= 1e-12)


def test_affine_image_of_codebook_is_recovered():
    """w = a C[c] + b with balanced codes: assignment returns c and OLS returns (a, b)."""
    rng = np.random.default_rng(4)
    for _ in range(50):
        c = rng.permutation(np.repeat(np.arange(4), 8)).astype(np.uint8)
        a = rng.uniform(0.001, 0.1)
        b = rng.uniform(-0.05, 0.05)
        Wg = (a * O.C16[c] + b)[None, :]
        q = O.assign_codes(Wg)
        assert q[0].tolist() == c.tolist()
        S, Z = O.ols_fit(Wg, q)
        assert abs(S[0] - a) <= a * 1e-8 and abs(Z[0] - b) <= 1e-12


def test_crumb_order():
    rng = np.random.default_rng(2)
    q = rng.integers(0, 4, size=(3, 128), dtype=np.uint8)
    b = O.pack_crumbs(q)
    for n in range(3):
        for i in range(32):
            v = int(b[n, i])
            assert [(v >> (2 * j)) & 3 for j in range(4)] == q[n, 4 * i:4 * i + 4].tolist()


def test_w2_pack_unpack_and_dequant():
    rng = np.random.default_rng(6)
    W = (rng.standard_normal((5, 128)) * 0.02).astype(np.float32)
    blob = O.pack_w2cb(W, np.array([1, 64], np.int32))
    q, S16, Z16, idx, vals = O.unpack_w2(blob)
    q2, S, Z = O.quantise_w2(np.where(np.isin(np.arange(128), [1, 64]), 0.0, W).astype(np.float32))
    assert np.array_equal(q, q2)
    assert np.array_equal(S16, O.fp16_round(S).astype(np.float64))
    assert np.array_equal(Z16, O.fp16_round(Z).astype(np.float64))
    Wh = O.dequant_w2(blob)
    assert np.array_equal(Wh, (S16[..., None] * O.C16[q].reshape(5, 4, 32) + Z16[..., None]).reshape(5, 128))
