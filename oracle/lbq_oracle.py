"""CPU oracle for the Group-32 low-bit weight-only decode GEMV (FP64, NumPy).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The library itself never calls it; it shares no code, table or
helper with the C++/CUDA path under ``bit_weight_only_lbq_gb300/csrc``.

What it computes, and where the definition comes from
-----------------------------------------------------
* 4-bit asymmetric Group-32 quantiser and its byte layout: SPECTRA article
  ("Compress any LLM 3x in one click", wpnews.pro), section 3.4
  "Microscaled Group-32 Quantization with Marlin-Interleaved Layout" and
  Appendix A, Proposition 2 (the rounding rule q = clamp(round(w/s + z), 0, 15)).
* Kurtosis-adaptive outlier ratio and channel saliency S_j = |gamma_j| ||W[:,j]||_2
  with gamma = 1: same article, sections 3.2-3.3 and Proposition 1.
* 2-bit Lloyd-Max codebook, OLS group fit, 4-codes-per-byte packing and
  profile-guided impact score: otf-llm 4.0.0 (PyPI page), sections 2, 3, 4, 5.
* Fused GEMV with exact FP16 outlier columns: SPECTRA section 4.1 and the
  otf-llm "Architecture & Key Innovations" diagram (FP16 outliers + INT2
  background = exact output).

Readings where the pages are silent (each listed in the design notes):
* all statistics in FP64 from the FP32 input; every sum is sequential in
  index order; round-half-to-even; FP16 rounding once, at storage;
* z and q use the FP64 scale s; dequantisation uses the stored FP16 scale;
* W2 code assignment: standardise each group by its mean and population
  standard deviation, then nearest FP16 centroid (ties to the lower code);
* OLS epsilon = 1e-8;  W2 outlier count floor(0.035 K);  W4 outlier count
  floor(r K);
* outlier columns are zeroed in the dense matrix before grouping and excluded
  from the background product (x with those channels zeroed).

Blob format (version 1), all integers little-endian, written here from the
layout description, independently of the C++ packer:
  [0:8)   magic  b"LBQW4G32" (4-bit) or b"LBQW2C32" (2-bit codebook)
  [8:12)  u32 version = 1        [12:16) u32 header bytes = 128
  [16:24) i64 N                  [24:32) i64 K
  [32:36) i32 n_out              [36:40) u32 group size = 32
  [40:48) u64 total blob bytes
  [48:128) five (u64 offset, u64 row stride) pairs for the sections
     4-bit : qweight, scales, zeros, outlier idx, outlier vals
     2-bit : codes,   S,      Z,     outlier idx, outlier vals
  Every section starts on a 256-byte boundary (the first at 256); every row of
  a 2-D section is padded with zero bytes to a multiple of 16 bytes.
"""
from __future__ import annotations

import math
import struct

import numpy as np

G = 32
EPS_SCALE = 1e-8          # SPECTRA section 3.4: s = max((wmax - wmin)/15, 1e-8)
EPS_OLS = 1e-8            # otf-llm section 3: epsilon of the OLS denominator (value: a reading)
CODEBOOK_DECIMAL = (-1.52, -0.45, 0.45, 1.52)   # otf-llm section 2
W2_OUTLIER_FRAC = 0.035   # otf-llm section 4 / quickstart "32 0.035"
HEADER_BYTES = 128
SECTION_ALIGN = 256
ROW_ALIGN = 16
MAGIC_W4 = b"LBQW4G32"
MAGIC_W2 = b"LBQW2C32"
VERSION = 1

F64 = np.float64


def fp16_round(a) -> np.ndarray:
    """Round FP64 values to the nearest FP16 (ties to even), returned as float16."""
    with np.errstate(over="ignore"):
        return np.asarray(a, dtype=F64).astype(np.float16)


# FP16 codebook: the decimal Lloyd-Max centroids rounded once to FP16
CODEBOOK_F16 = fp16_round(CODEBOOK_DECIMAL)
C16 = CODEBOOK_F16.astype(F64)


def seq_sum_last(a: np.ndarray) -> np.ndarray:
    """Sum along the last axis, strictly left to right, in FP64."""
    a = np.asarray(a, dtype=F64)
    acc = a[..., 0].copy()
    for k in range(1, a.shape[-1]):
        acc = acc + a[..., k]
    return acc


def seq_sum_vector(v: np.ndarray) -> float:
    """Sequential FP64 sum of a 1-D vector (accumulate is inherently ordered)."""
    v = np.asarray(v, dtype=F64)
    if v.size == 0:
        return 0.0
    return float(np.add.accumulate(v)[-1])


# ---------------------------------------------------------------------------
# blob layout
# ---------------------------------------------------------------------------

def _up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def layout(kind: str, N: int, K: int, n_out: int) -> dict:
    """Offsets and row strides of the five sections (see module docstring)."""
    if kind == "w4":
        rows = (K // 2, K // 32 * 2, K // 64)          # qweight, scales, zeros: bytes per row
    elif kind == "w2":
        rows = (K // 4, K // 32 * 2, K // 32 * 2)      # codes, S, Z
    else:
        raise ValueError(kind)
    ld = [_up(r, ROW_ALIGN) for r in rows]
    off = []
    cur = SECTION_ALIGN
    for l in ld:
        off.append(cur)
        cur = _up(cur + N * l, SECTION_ALIGN)
    off_idx = cur
    cur = _up(cur + 4 * n_out, SECTION_ALIGN)
    ld_v = _up(2 * n_out, ROW_ALIGN)
    off_vals = cur
    total = _up(cur + N * ld_v, SECTION_ALIGN)
    return {
        "offsets": off + [off_idx, off_vals],
        "strides": ld + [0, ld_v],
        "total": total,
    }


def _write_blob(kind: str, N: int, K: int, idx: np.ndarray, sec_rows: list, vals16: np.ndarray) -> np.ndarray:
    n_out = int(idx.size)
    L = layout(kind, N, K, n_out)
    blob = np.zeros(L["total"], dtype=np.uint8)
    hdr = bytearray(HEADER_BYTES)
    hdr[0:8] = MAGIC_W4 if kind == "w4" else MAGIC_W2
    struct.pack_into("<IIqqiIQ", hdr, 8, VERSION, HEADER_BYTES, N, K, n_out, G, L["total"])
    for i in range(5):
        struct.pack_into("<QQ", hdr, 48 + 16 * i, L["offsets"][i], L["strides"][i])
    blob[:HEADER_BYTES] = np.frombuffer(bytes(hdr), dtype=np.uint8)
    for i, data in enumerate(sec_rows):
        data = np.ascontiguousarray(data).view(np.uint8).reshape(N, -1)
        o, ld = L["offsets"][i], L["strides"][i]
        view = blob[o:o + N * ld].reshape(N, ld)
        view[:, :data.shape[1]] = data
    if n_out:
        o = L["offsets"][3]
        blob[o:o + 4 * n_out] = np.ascontiguousarray(idx.astype("<i4")).view(np.uint8)
        o, ld = L["offsets"][4], L["strides"][4]
        view = blob[o:o + N * ld].reshape(N, ld)
        view[:, :2 * n_out] = np.ascontiguousarray(vals16.astype("<f2")).view(np.uint8).reshape(N, 2 * n_out)
    return blob


def read_header(blob: np.ndarray) -> dict:
    b = bytes(blob[:HEADER_BYTES])
    magic = b[0:8]
    version, hbytes, N, K, n_out, group, total = struct.unpack_from("<IIqqiIQ", b, 8)
    secs = [struct.unpack_from("<QQ", b, 48 + 16 * i) for i in range(5)]
    return {"magic": magic, "version": version, "header_bytes": hbytes, "N": N, "K": K,
            "n_out": n_out, "group": group, "total": total,
            "offsets": [s[0] for s in secs], "strides": [s[1] for s in secs]}


def _section(blob: np.ndarray, hdr: dict, i: int, row_bytes: int) -> np.ndarray:
    o, ld, N = hdr["offsets"][i], hdr["strides"][i], hdr["N"]
    return blob[o:o + N * ld].reshape(N, ld)[:, :row_bytes]


# ---------------------------------------------------------------------------
# outlier selection
# ---------------------------------------------------------------------------

def column_norms(W: np.ndarray) -> np.ndarray:
    """||W[:, j]||_2 in FP64, the sum of squares taken row by row in order."""
    W = np.asarray(W)
    acc = np.zeros(W.shape[1], dtype=F64)
    for n in range(W.shape[0]):
        r = W[n].astype(F64)
        acc = acc + r * r
    return np.sqrt(acc)


def population_kurtosis(S: np.ndarray) -> float:
    """kappa = (1/K) sum z_j^4 with z_j = (S_j - mu)/sigma, population moments
    (SPECTRA Proposition 1).  A constant vector has no defined kurtosis; it is
    taken as 0 here (no excess)."""
    S = np.asarray(S, dtype=F64)
    K = S.size
    mu = seq_sum_vector(S) / K
    d = S - mu
    var = seq_sum_vector(d * d) / K
    sigma = math.sqrt(var)
    if sigma == 0.0:
        return 0.0
    z = d / sigma
    z2 = z * z
    return seq_sum_vector(z2 * z2) / K


def outlier_ratio(kappa: float) -> float:
    """r = clamp(0.01 (1 + 0.15 ln(1 + max(0, kappa - 3))), 0.005, 0.03)
    (SPECTRA section 3.3, with r_base = 0.01)."""
    r = 0.01 * (1.0 + 0.15 * math.log(1.0 + max(0.0, kappa - 3.0)))
    return min(max(r, 0.005), 0.03)


def top_indices(score: np.ndarray, n: int) -> np.ndarray:
    """The n largest scores, ties broken towards the lower index, returned ascending."""
    score = np.asarray(score, dtype=F64)
    order = sorted(range(score.size), key=lambda j: (-score[j], j))
    return np.array(sorted(order[:n]), dtype=np.int32)


def select_outliers_w4(W: np.ndarray) -> np.ndarray:
    """Saliency S_j = ||W[:,j]||_2 (gamma = 1, no preceding norm), kurtosis-adaptive
    ratio r, n_out = floor(r K) largest-saliency columns (SPECTRA sections 3.2-3.3)."""
    S = column_norms(W)
    r = outlier_ratio(population_kurtosis(S))
    n_out = int(math.floor(r * W.shape[1]))
    return top_indices(S, n_out)


def impact_scores(W: np.ndarray, Xprof: np.ndarray) -> np.ndarray:
    """I_c = ||W[:,c]||_2 * mean_p |x_{p,c}| (otf-llm section 4)."""
    Xa = np.abs(np.asarray(Xprof, dtype=np.float16).astype(F64))
    acc = np.zeros(Xa.shape[1], dtype=F64)
    for p in range(Xa.shape[0]):
        acc = acc + Xa[p]
    return column_norms(W) * (acc / Xa.shape[0])


def select_outliers_impact(W: np.ndarray, Xprof: np.ndarray, frac: float = W2_OUTLIER_FRAC) -> np.ndarray:
    n_out = int(math.floor(frac * W.shape[1]))
    return top_indices(impact_scores(W, Xprof), n_out)


def _split_outliers(W: np.ndarray, idx) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    idx = np.asarray(idx if idx is not None else [], dtype=np.int32)
    W = np.asarray(W, dtype=np.float32)
    vals16 = fp16_round(W[:, idx].astype(F64)) if idx.size else np.zeros((W.shape[0], 0), np.float16)
    Wd = W.copy()
    if idx.size:
        Wd[:, idx] = 0.0
    return Wd, idx, vals16


# ---------------------------------------------------------------------------
# 4-bit asymmetric Group-32
# ---------------------------------------------------------------------------

def quantise_w4(Wd: np.ndarray):
    """Per (row, group of 32 along K): wmin, wmax, s, z, q (SPECTRA 3.4, App. A Prop 2).

    Returns q (N, K/32, 32) uint8, z (N, K/32) uint8, s (N, K/32) FP64 (unrounded)."""
    N, K = Wd.shape
    Wg = np.asarray(Wd, dtype=F64).reshape(N, K // G, G)
    wmin = Wg.min(axis=2)
    wmax = Wg.max(axis=2)
    s = np.maximum((wmax - wmin) / 15.0, EPS_SCALE)
    z = np.clip(np.rint(-wmin / s), 0.0, 15.0)
    q = np.clip(np.rint(Wg / s[..., None] + z[..., None]), 0.0, 15.0)
    return q.astype(np.uint8), z.astype(np.uint8), s


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Byte k of a 32-group = q_k | q_{k+16} << 4, k in [0, 16)  (SPECTRA 3.4)."""
    N, ng, _ = q.shape
    return (q[..., :16] | (q[..., 16:] << 4)).astype(np.uint8).reshape(N, ng * 16)


def pack_zero_points(z: np.ndarray) -> np.ndarray:
    """PackedZero[i, m] = z_{2m} | z_{2m+1} << 4  (SPECTRA 3.4)."""
    return (z[:, 0::2] | (z[:, 1::2] << 4)).astype(np.uint8)


def pack_w4(W: np.ndarray, idx=None) -> np.ndarray:
    """Quantise and pack an N x K FP32 matrix (K % 64 == 0) into a 4-bit blob."""
    N, K = W.shape
    assert K % 64 == 0
    Wd, idx, vals16 = _split_outliers(W, idx)
    q, z, s = quantise_w4(Wd)
    s16 = fp16_round(s)
    return _write_blob("w4", N, K, idx, [pack_nibbles(q), s16.astype("<f2"), pack_zero_points(z)], vals16)


def unpack_w4(blob: np.ndarray):
    """Inverse of the layout: q (N,K) uint8, z (N,K/32) uint8, s16 (N,K/32) FP64,
    idx (n_out,) int32, vals (N,n_out) FP64."""
    h = read_header(blob)
    assert h["magic"] == MAGIC_W4
    N, K, n_out = h["N"], h["K"], h["n_out"]
    qb = _section(blob, h, 0, K // 2).reshape(N, K // 32, 16)
    q = np.concatenate([qb & 0x0F, qb >> 4], axis=2).reshape(N, K)
    s16 = np.ascontiguousarray(_section(blob, h, 1, K // 16)).view("<f2").astype(F64)
    zb = _section(blob, h, 2, K // 64)
    z = np.stack([zb & 0x0F, zb >> 4], axis=2).reshape(N, K // 32)
    idx, vals = _unpack_outliers(blob, h)
    return q, z, s16, idx, vals


def _unpack_outliers(blob, h):
    N, n_out = h["N"], h["n_out"]
    if n_out == 0:
        return np.zeros(0, np.int32), np.zeros((N, 0), F64)
    o = h["offsets"][3]
    idx = np.ascontiguousarray(blob[o:o + 4 * n_out]).view("<i4").astype(np.int32)
    vals = np.ascontiguousarray(_section(blob, h, 4, 2 * n_out)).view("<f2").astype(F64)
    return idx, vals


def dequant_w4(blob: np.ndarray, rows=None) -> np.ndarray:
    """W_hat = (q - z) * s16 in FP64, from the packed bytes.  Optional row subset."""
    q, z, s16, _, _ = unpack_w4(blob)
    if rows is not None:
        q, z, s16 = q[rows], z[rows], s16[rows]
    N, K = q.shape
    qg = q.reshape(N, K // G, G).astype(F64)
    return ((qg - z[..., None].astype(F64)) * s16[..., None]).reshape(N, K)


# ---------------------------------------------------------------------------
# 2-bit Lloyd-Max codebook, Group-32, OLS (S, Z)
# ---------------------------------------------------------------------------

def assign_codes(Wg: np.ndarray) -> np.ndarray:
    """Nearest FP16 centroid of each standardised weight; ties to the lower code.

    Wg: (..., 32) FP64 groups.  Standardisation uses the group mean and the
    population standard deviation (a reading; the otf-llm page only says the
    weights are assigned to centroids)."""
    mu = seq_sum_last(Wg) / G
    d = Wg - mu[..., None]
    sigma = np.sqrt(seq_sum_last(d * d) / G)
    safe = np.where(sigma > 0, sigma, 1.0)
    u = np.where(sigma[..., None] > 0, d / safe[..., None], 0.0)
    dist = np.abs(u[..., None] - C16)          # (..., 32, 4)
    return np.argmin(dist, axis=-1).astype(np.uint8)   # first minimum = lower code


def ols_fit(Wg: np.ndarray, q: np.ndarray):
    """S = sum (w - wbar)(c - cbar) / (sum (c - cbar)^2 + eps),  Z = wbar - S cbar
    (otf-llm section 3), all in FP64, sums sequential."""
    Cq = C16[q]
    wbar = seq_sum_last(Wg) / G
    cbar = seq_sum_last(Cq) / G
    dw = Wg - wbar[..., None]
    dc = Cq - cbar[..., None]
    S = seq_sum_last(dw * dc) / (seq_sum_last(dc * dc) + EPS_OLS)
    Z = wbar - S * cbar
    return S, Z


def quantise_w2(Wd: np.ndarray):
    N, K = Wd.shape
    Wg = np.asarray(Wd, dtype=F64).reshape(N, K // G, G)
    q = assign_codes(Wg)
    S, Z = ols_fit(Wg, q)
    return q.reshape(N, K), S, Z


def pack_crumbs(q: np.ndarray) -> np.ndarray:
    """byte = q0 | q1 << 2 | q2 << 4 | q3 << 6 for four consecutive k (otf-llm section 5)."""
    N, K = q.shape
    q4 = q.reshape(N, K // 4, 4).astype(np.uint8)
    return (q4[..., 0] | (q4[..., 1] << 2) | (q4[..., 2] << 4) | (q4[..., 3] << 6)).astype(np.uint8)


def pack_w2cb(W: np.ndarray, idx=None) -> np.ndarray:
    N, K = W.shape
    assert K % 64 == 0
    Wd, idx, vals16 = _split_outliers(W, idx)
    q, S, Z = quantise_w2(Wd)
    return _write_blob("w2", N, K, idx, [pack_crumbs(q), fp16_round(S).astype("<f2"),
                                          fp16_round(Z).astype("<f2")], vals16)


def unpack_w2(blob: np.ndarray):
    h = read_header(blob)
    assert h["magic"] == MAGIC_W2
    N, K = h["N"], h["K"]
    cb = _section(blob, h, 0, K // 4)
    q = np.stack([(cb >> (2 * j)) & 3 for j in range(4)], axis=2).reshape(N, K)
    S16 = np.ascontiguousarray(_section(blob, h, 1, K // 16)).view("<f2").astype(F64)
    Z16 = np.ascontiguousarray(_section(blob, h, 2, K // 16)).view("<f2").astype(F64)
    idx, vals = _unpack_outliers(blob, h)
    return q, S16, Z16, idx, vals


def dequant_w2(blob: np.ndarray, rows=None) -> np.ndarray:
    """W_hat = S16 * C16[q] + Z16 in FP64, from the packed bytes."""
    q, S16, Z16, _, _ = unpack_w2(blob)
    if rows is not None:
        q, S16, Z16 = q[rows], S16[rows], Z16[rows]
    N, K = q.shape
    Cq = C16[q].reshape(N, K // G, G)
    return (S16[..., None] * Cq + Z16[..., None]).reshape(N, K)


# ---------------------------------------------------------------------------
# GEMV / small-M GEMM
# ---------------------------------------------------------------------------

def dequant(blob: np.ndarray, rows=None) -> np.ndarray:
    magic = bytes(blob[:8])
    return dequant_w4(blob, rows) if magic == MAGIC_W4 else dequant_w2(blob, rows)


def outliers(blob: np.ndarray):
    h = read_header(blob)
    return _unpack_outliers(blob, h)


def gemm(blob: np.ndarray, X: np.ndarray, rows=None) -> np.ndarray:
    """Y[m, n] = sum_{k not outlier} W_hat[n,k] x[m,k] + sum_j vals[n,j] x[m, idx_j], FP64.

    X: (M, K) or (K,) FP16.  rows: optional subset of output rows."""
    X = np.asarray(X, dtype=np.float16).astype(F64)
    squeeze = X.ndim == 1
    X = np.atleast_2d(X)
    Wh = dequant(blob, rows)
    idx, vals = outliers(blob)
    if rows is not None:
        vals = vals[rows]
    Xb = X.copy()
    if idx.size:
        Xb[:, idx] = 0.0
    Y = Xb @ Wh.T
    if idx.size:
        Y = Y + X[:, idx] @ vals.T
    return Y[0] if squeeze else Y


def gemv(blob: np.ndarray, x: np.ndarray, rows=None) -> np.ndarray:
    return gemm(blob, np.asarray(x).reshape(-1), rows)


def within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, fp16_out: bool = False) -> np.ndarray:
    """The acceptance bound |y_gpu - y_ref| <= 2e-3 rms(y_ref) + 1e-3 |y_ref|
    (+ half an FP16 ulp of y_ref when the output was rounded to FP16)."""
    y_ref = np.asarray(y_ref, dtype=F64)
    y_gpu = np.asarray(y_gpu, dtype=F64)
    rms = math.sqrt(float(np.mean(y_ref * y_ref))) if y_ref.size else 0.0
    bound = 2e-3 * rms + 1e-3 * np.abs(y_ref)
    if fp16_out:
        bound = bound + 0.5 * fp16_ulp(y_ref)
    return np.abs(y_gpu - y_ref) <= bound


def fp16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of FP16 numbers at |v| (2^-24 in the subnormal range)."""
    a = np.abs(np.asarray(v, dtype=F64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -14.0)
    return np.ldexp(1.0, (e - 10).astype(int))
