"""Pins of the oracle's 4-bit Group-32 quantiser and layout against what the SPECTRA
article fixes: the hand-worked group, Proposition 2's bound, Proposition 3 and the
printed Experiment A statistics, the bit layout and the 4.625 bits/weight budget."""
import math

import numpy as np
import pytest

from oracle import lbq_oracle as O


def test_worked_group_codes_and_bytes(golden):
    g = golden("w4_worked_example.txt")
    w = np.array([float(v) for v in g["w_group0"] + g["w_group1"]], dtype=np.float32)[None, :]
    q, z, s = O.quantise_w4(w)
    assert q[0, 0].tolist() == [int(v) for v in g["q_group0"]]
    assert q[0, 1].tolist() == [int(v) for v in g["q_group1"]]
    assert z[0].tolist() == [int(v) for v in g["z"]]
    assert np.all(s == 1.0)
    blob = O.pack_w4(w)
    h = O.read_header(blob)
    rec = h["area"]                               # row block 0, record 0, row 0
    assert blob[rec:rec + 32].tolist() == [int(v, 16) for v in g["qweight_bytes"]]
    assert blob[rec + 2048:rec + 2052].view("<u2").tolist() == [int(v, 16) for v in g["scale_f16_bits"]]
    assert blob[rec + 2304:rec + 2305].tolist() == [int(v, 16) for v in g["zero_bytes"]]
    # groups 2..31 of the record and rows 1..3 of the row block are zero padding
    assert not blob[rec + 32:rec + 2048].any()
    assert not blob[rec + 2052:rec + 2304].any()
    assert not blob[rec + 2305:rec + 2368].any()


def test_round_half_even_points():
    # s = 1, z = 0 (wmin = 0): w = k + 0.5 sits exactly on a rounding tie
    w = np.zeros((1, 64), np.float32)
    w[0, :32] = [0.0, 15.0] + [0.5, 1.5, 2.5, 3.5, 4.5, 5.5, 6.5, 7.5, 8.5, 9.5, 10.5, 11.5, 12.5, 13.5] + [7.0] * 16
    q, z, s = O.quantise_w4(w)
    assert z[0, 0] == 0 and s[0, 0] == 1.0
    assert q[0, 0, 2:16].tolist() == [0, 2, 2, 4, 4, 6, 6, 8, 8, 10, 10, 12, 12, 14]


def _gaussian(N, K, seed):
    return np.random.default_rng(seed).standard_normal((N, K)).astype(np.float32)


def test_prop2_bound_sign_spanning_groups():
    W = _gaussian(512, 1024, 3)
    q, z, s = O.quantise_w4(W)
    Wg = W.astype(np.float64).reshape(512, 32, 32)
    spans = (Wg.min(2) <= 0) & (Wg.max(2) >= 0)
    assert spans.mean() > 0.999
    err = np.abs(Wg - (q.astype(np.float64) - z[..., None]) * s[..., None])
    assert np.all(err[spans] <= s[..., None].repeat(32, 2)[spans] * (0.5 + 1e-12))
    # with the stored FP16 scale the bound widens by the scale's own rounding
    s16 = O.fp16_round(s).astype(np.float64)
    err16 = np.abs(Wg - (q.astype(np.float64) - z[..., None]) * s16[..., None])
    bound16 = s16 / 2 + 15 * np.abs(s - s16) + 1e-12
    assert np.all(err16[spans] <= bound16[..., None].repeat(32, 2)[spans])


def test_one_sided_and_constant_groups():
    w = np.zeros((1, 64), np.float32)
    w[0, :32] = np.linspace(1.0, 4.0, 32)          # all positive: z clamps to 0
    w[0, 32:] = 0.0                                 # constant zero group: s floor, exact 0
    q, z, s = O.quantise_w4(w)
    assert z[0, 0] == 0 and z[0, 1] == 0
    assert s[0, 1] == O.EPS_SCALE and np.all(q[0, 1] == 0)
    assert O.fp16_round(O.EPS_SCALE) == 0.0        # the 1e-8 floor underflows FP16
    Wh = O.dequant_w4(O.pack_w4(w))
    assert np.all(Wh[0, 32:] == 0.0)


def test_experiment_a_printed_statistics():
    """SPECTRA section 5.7 Experiment A / section 2.3: 2048 x 2048 Gaussian, G32 ->
    8.08 %, 21.85 dB, cosine 0.99676, max |w - w_hat| / s = 0.50000 (printed)."""
    W = _gaussian(2048, 2048, 0)
    q, z, s = O.quantise_w4(W)
    Wg = W.astype(np.float64).reshape(2048, 64, 32)
    Wh = (q.astype(np.float64) - z[..., None]) * s[..., None]
    err = np.linalg.norm(Wg - Wh) / np.linalg.norm(Wg)
    snr = 10 * math.log10(float((Wg ** 2).sum() / ((Wg - Wh) ** 2).sum()))
    cos = float((Wg * Wh).sum() / math.sqrt(float((Wg ** 2).sum() * (Wh ** 2).sum())))
    mx = float((np.abs(Wg - Wh) / s[..., None]).max())
    assert abs(err * 100 - 8.08) <= 0.005
    assert abs(snr - 21.85) <= 0.005
    assert abs(cos - 0.99676) <= 1e-5
    assert round(mx, 5) == 0.5
    # Proposition 3: closed-form 7.97 %, matched "within 0.11 percentage points"
    d = 4.14
    pred = d / (15 * math.sqrt(12))
    assert abs(pred * 100 - 7.97) < 0.005
    assert abs(20 * math.log10(15 * math.sqrt(12) / d) - 21.97) < 0.005
    assert abs(err * 100 - pred * 100) <= 0.12


def test_pack_unpack_round_trip_random_codes():
    rng = np.random.default_rng(7)
    q = rng.integers(0, 16, size=(5, 8, 32), dtype=np.uint8)
    z = rng.integers(0, 16, size=(5, 8), dtype=np.uint8)
    qb = O.pack_nibbles(q)
    zb = O.pack_zero_points(z)
    assert qb.shape == (5, 128) and zb.shape == (5, 4)
    # independent decode of the bit positions
    for n in range(5):
        for g in range(8):
            for k in range(16):
                b = int(qb[n, g * 16 + k])
                assert b & 15 == q[n, g, k] and b >> 4 == q[n, g, k + 16]
        for m in range(4):
            assert int(zb[n, m]) == int(z[n, 2 * m]) | (int(z[n, 2 * m + 1]) << 4)


def test_byte_budget_4_625_bits_per_weight():
    """SPECTRA section 7.2: Group-32 costs 4.625 bits per weight (4 + 16/32 + 4/32)."""
    N, K = 16, 4096
    L = O.layout("w4", N, K, 0)
    assert L["rb_bytes"] * L["n_rb"] * 8 / (N * K) == 4.625
    assert O.layout("w2", N, K, 0)["rb_bytes"] * 4 * 8 / (N * K) == 3.0


def _golden_layout(g, key):
    return {k: int(v) for k, v in (item.split("=") for item in g[key])}


def test_layout_golden(golden):
    g = golden("blob_layout_example.txt")
    for key, kind, N, K, n in (("w4_N3_K64_nout2", "w4", 3, 64, 2), ("w4_N5_K2112_nout0", "w4", 5, 2112, 0),
                               ("w2_N2_K128_nout5", "w2", 2, 128, 5), ("w2_N4_K4096_nout300", "w2", 4, 4096, 300)):
        want = _golden_layout(g, key)
        L = O.layout(kind, N, K, n)
        assert {k: L[k] for k in want} == want, key
        rng = np.random.default_rng(N)
        W = rng.standard_normal((N, K)).astype(np.float32)
        idx = np.arange(n, dtype=np.int32) * 3
        blob = (O.pack_w4 if kind == "w4" else O.pack_w2cb)(W, idx)
        h = O.read_header(blob)
        assert len(blob) == want["total"] and {k: h[k] for k in want if k in h} == \
            {k: want[k] for k in want if k in h}


def test_outlier_columns_are_isolated():
    rng = np.random.default_rng(11)
    W = rng.standard_normal((6, 128)).astype(np.float32)
    idx = np.array([3, 40, 77], np.int32)
    blob = O.pack_w4(W, idx)
    Wh = O.dequant_w4(blob)
    assert np.all(Wh[:, idx] == 0.0)               # zeroed before grouping -> q = z
    i2, vals = O.outliers(blob)
    assert i2.tolist() == idx.tolist()
    assert np.array_equal(vals, W[:, idx].astype(np.float16).astype(np.float64))


def test_embedding_gather_of_the_worked_row(golden):
    """SPECTRA 4.3 row gather: the worked row (s = 1, so w_hat = q - z exactly),
    gathered twice, in FP16 and FP32."""
    g = golden("w4_worked_example.txt")
    w = np.array([float(v) for v in g["w_group0"] + g["w_group1"]], dtype=np.float32)[None, :]
    q = np.array([int(v) for v in g["q_group0"] + g["q_group1"]], dtype=np.float64)
    z = np.repeat([float(v) for v in g["z"]], 32)
    blob = O.pack_w4(np.vstack([w, 2 * w]))
    for dt in (np.float16, np.float32):
        rows = O.embed(blob, [0, 0], out_dtype=dt)
        assert rows.dtype == dt
        assert np.array_equal(rows.astype(np.float64), np.vstack([q - z, q - z]))


def test_kv_cache_record_of_the_worked_row(golden):
    """SPECTRA 4.5 KV cache: the worked row (FP16-exact values) gives the worked
    codes, scales and zero byte in its record, and reads back exactly."""
    g = golden("w4_worked_example.txt")
    w = np.array([float(v) for v in g["w_group0"] + g["w_group1"]], dtype=np.float16)[None, :]
    rec = O.kv_quantize(w)
    assert rec.shape == (1, O.kv_record_bytes(64)) and O.kv_record_bytes(64) == 48
    assert rec[0, :32].tolist() == [int(v, 16) for v in g["qweight_bytes"]]
    assert rec[0, 32:36].tolist() == [0x00, 0x3C, 0x00, 0x3C]          # FP16 1.0, 1.0
    assert rec[0, 36] == int(g["zero_bytes"][0], 16)
    q = np.array([int(v) for v in g["q_group0"] + g["q_group1"]], dtype=np.float64)
    z = np.repeat([float(v) for v in g["z"]], 32)
    assert np.array_equal(O.kv_dequant(rec, 64)[0].astype(np.float64), q - z)


def test_kv_cache_roundtrip_bound():
    """Prop. 2: every read-back value is within s16/2 + 15|s16 - s| of the state
    (plus half an FP16 ulp of the read), for random states with spikes."""
    rng = np.random.default_rng(8)
    X = (rng.standard_normal((33, 1024)) * 3).astype(np.float16)
    X[:, rng.choice(1024, size=6, replace=False)] *= 100
    X[5, :32] = np.float16(0.75)                                       # a constant group reads back 0
    back = O.kv_dequant(O.kv_quantize(X), 1024).astype(np.float64)
    Xg = X.astype(np.float64).reshape(33, 32, 32)
    s = np.maximum((Xg.max(2) - Xg.min(2)) / 15.0, 1e-8)
    s16 = O.fp16_round(s).astype(np.float64)
    bound = np.repeat(s16 / 2 + 15 * np.abs(s16 - s), 32, axis=1) + 0.5 * O.fp16_ulp(back)
    err = np.abs(back - X.astype(np.float64))
    err[5, :32] = 0.0
    assert np.all(err <= bound * (1 + 1e-9))
    assert np.array_equal(back[5, :32], np.zeros(32))
