"""Brute-force pin of the oracle GEMV: exact rational arithmetic over a blob decoded
bit by bit (header parsed independently with struct), on tiny shapes, with and
without outlier columns, M = 1 and M > 1."""
import struct
from fractions import Fraction

import numpy as np
import pytest

from oracle import lbq_oracle as O


def _f16_value(bits: int) -> Fraction:
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 10) & 0x1F
    m = bits & 0x3FF
    assert e != 31
    if e == 0:
        return sign * Fraction(m, 1 << 24)
    return sign * Fraction(1024 + m, 1024) * (Fraction(2) ** (e - 15))


def _decode(blob):
    """Independent reading of the documented blob layout, element by element."""
    b = bytes(blob)
    magic = b[:8]
    N, K = struct.unpack_from("<qq", b, 16)
    n_out = struct.unpack_from("<i", b, 32)[0]
    area, rb_bytes, rec_bytes, recs, out_rec_bytes, out_recs, idx_off = struct.unpack_from("<7Q", b, 48)
    W = [[Fraction(0)] * K for _ in range(N)]
    for n in range(N):
        rb, r = divmod(n, 4)
        for g in range(K // 32):
            blk, gl = divmod(g, 32)
            rec = area + rb * rb_bytes + blk * rec_bytes
            if magic == b"LBQW4G32":
                s = _f16_value(struct.unpack_from("<H", b, rec + 2048 + (r * 32 + gl) * 2)[0])
                zb = b[rec + 2304 + r * 16 + gl // 2]
                z = (zb >> 4) if gl % 2 else (zb & 15)
                for k in range(32):
                    byte = b[rec + (r * 32 + gl) * 16 + (k % 16)]
                    q = (byte >> 4) if k >= 16 else (byte & 15)
                    W[n][g * 32 + k] = (q - z) * s
            else:
                S = _f16_value(struct.unpack_from("<H", b, rec + 1024 + (r * 32 + gl) * 2)[0])
                Z = _f16_value(struct.unpack_from("<H", b, rec + 1280 + (r * 32 + gl) * 2)[0])
                for k in range(32):
                    byte = b[rec + (r * 32 + gl) * 8 + k // 4]
                    q = (byte >> (2 * (k % 4))) & 3
                    C = [-Fraction(389, 256), -Fraction(1843, 4096), Fraction(1843, 4096), Fraction(389, 256)][q]
                    W[n][g * 32 + k] = S * C + Z
    idx = list(struct.unpack_from("<%di" % n_out, b, idx_off)) if n_out else []
    vals = []
    for n in range(N):
        rb, r = divmod(n, 4)
        row = []
        for j in range(n_out):
            o, jj = divmod(j, 256)
            # full records are 256 columns wide; the last one holds the rest rounded up to 8
            width = min(256, -(-n_out // 8) * 8 - 256 * o)
            off = area + rb * rb_bytes + recs * rec_bytes + o * out_rec_bytes + (r * width + jj) * 2
            row.append(_f16_value(struct.unpack_from("<H", b, off)[0]))
        vals.append(row)
    return W, idx, vals


def _exact_gemm(blob, X16):
    W, idx, vals = _decode(blob)
    N = len(W)
    K = len(W[0])
    out = []
    for x in X16:
        xf = [_f16_value(int(v)) for v in x.view("<u2")]
        y = []
        for n in range(N):
            acc = sum(W[n][k] * xf[k] for k in range(K) if k not in idx)
            acc += sum(vals[n][j] * xf[idx[j]] for j in range(len(idx)))
            y.append(acc)
        out.append(y)
    return out


@pytest.mark.parametrize("kind,N,K,idx", [
    ("w4", 8, 64, []),
    ("w4", 3, 128, [0, 33, 127]),
    ("w2", 8, 64, []),
    ("w2", 3, 128, [2, 64, 100, 101]),
])
def test_gemv_exact_rational(kind, N, K, idx):
    rng = np.random.default_rng(N * 1000 + K + len(idx))
    W = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    X = rng.standard_normal((2, K)).astype(np.float16)
    X[:, 5] *= 100
    idx = np.array(idx, np.int32)
    blob = O.pack_w4(W, idx) if kind == "w4" else O.pack_w2cb(W, idx)
    exact = _exact_gemm(blob, X)
    Y = O.gemm(blob, X)
    for m in range(2):
        for n in range(N):
            e = float(exact[m][n])
            assert abs(Y[m, n] - e) <= 1e-13 * (abs(e) + 1e-3)
    y0 = O.gemv(blob, X[0])
    assert np.array_equal(y0, Y[0])
    # row subset agrees with the full product
    assert np.array_equal(O.gemm(blob, X, rows=[1, N - 1]), Y[:, [1, N - 1]])


def test_tolerance_function():
    y = np.array([1.0, -2.0, 100.0, 0.0])
    rms = np.sqrt(np.mean(y * y))
    ok = O.within_tolerance(y + 2e-3 * rms * 0.99, y)
    assert ok.all()
    bad = O.within_tolerance(y + (2e-3 * rms + 1e-3 * np.abs(y)) * 1.01, y)
    assert not bad.any()
    assert O.fp16_ulp(np.array([1.0, 1024.0, 2.0 ** -20]))[0] == 2.0 ** -10
    assert O.fp16_ulp(np.array([1024.0]))[0] == 1.0
    assert O.fp16_ulp(np.array([2.0 ** -20]))[0] == 2.0 ** -24


def test_row_chunks_equal_whole_matrix():
    """The every-row parity tests compute the oracle over row chunks in worker
    processes; rows are independent in the blob format, so the chunks'
    products concatenate to the whole matrix's, bit for bit (both formats,
    with outliers, a ragged last chunk)."""
    import oracle_rows
    rng = np.random.default_rng(5)
    N, K = 70, 1088
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    X = rng.standard_normal((3, K)).astype(np.float16)
    idx = np.sort(rng.choice(K, size=21, replace=False)).astype(np.int32)
    with oracle_rows.pool(2) as ex:
        for kind, pack in (("w4", O.pack_w4), ("w2", O.pack_w2cb)):
            whole = O.gemm(pack(W, idx), X)
            assert np.array_equal(oracle_rows.collect(oracle_rows.submit(ex, kind, W, idx, X, chunk=24)), whole)
