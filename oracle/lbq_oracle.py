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

Blob format (version 2), all integers little-endian, written here from the
layout description, independently of the C++ packer:
  [0:8)    magic b"LBQW4G32" (4-bit) or b"LBQW2C32" (2-bit codebook)
  [8:12)   u32 version = 2           [12:16)  u32 header bytes = 128
  [16:24)  i64 N                     [24:32)  i64 K
  [32:36)  i32 n_out                 [36:40)  u32 group size = 32
  [40:48)  u64 total blob bytes
  [48:56)  u64 offset of the row-block area (256)
  [56:64)  u64 bytes per row block
  [64:72)  u64 bytes per dense record   [72:80)  u64 dense records per row block
  [80:88)  u64 bytes per full outlier record [88:96)  u64 outlier records per row block
  [96:104) u64 offset of the outlier index array (n_out int32)
  [104:128) zero
Rows are taken 4 at a time (a row block; rows past N are zero).  A row block
holds ceil(K/1024) dense records, one per block of 32 groups along K (groups
past K/32 are zero), then ceil(n_out/256) outlier records.  Inside a record,
each of the three parts is row-major over (row 0..3, group 0..31):
  4-bit  record (2368 B): qweight 16 B per group (byte k = q_k | q_{k+16} << 4),
         then FP16 scale per group, then zero points z_{2m} | z_{2m+1} << 4 per byte;
  2-bit  record (1536 B): codes 8 B per group (byte = q0 | q1<<2 | q2<<4 | q3<<6),
         then FP16 S per group, then FP16 Z per group;
  outlier record j: W[n, idx_c] in FP16 for its columns c = 256 j .. 256 j + w_j - 1,
         row-major over (row 0..3, column); w_j = 256 except for the last record,
         whose width is rounded up to a multiple of 8 columns (columns past n_out
         are zero), so a row block's outlier records take 8 * round_up(n_out, 8) bytes.
The idx array starts on a 256-byte boundary after the row-block area.
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
MAGIC_W4 = b"LBQW4G32"
MAGIC_W2 = b"LBQW2C32"
VERSION = 2

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


REC_GROUPS = 32          # groups per dense record (1024 k)
ROWS_PER_BLOCK = 4
OUT_COLS = 256           # outlier columns per full outlier record
OUT_COL_ALIGN = 8        # the last outlier record's width is a multiple of this


def record_parts(kind: str) -> tuple:
    """Bytes per row of the three parts of a dense record: packed, scale/S, zero/Z."""
    if kind == "w4":
        return 16 * REC_GROUPS, 2 * REC_GROUPS, REC_GROUPS // 2
    if kind == "w2":
        return 8 * REC_GROUPS, 2 * REC_GROUPS, 2 * REC_GROUPS
    raise ValueError(kind)


def layout(kind: str, N: int, K: int, n_out: int) -> dict:
    """Sizes and offsets of a blob (see module docstring)."""
    parts = record_parts(kind)
    rec = ROWS_PER_BLOCK * sum(parts)
    nrec = -(-K // (REC_GROUPS * G))
    out_rec = ROWS_PER_BLOCK * OUT_COLS * 2 if n_out else 0
    n_outrec = -(-n_out // OUT_COLS)
    out_cols = _up(n_out, OUT_COL_ALIGN)                # columns stored, last record trimmed
    rb_bytes = nrec * rec + ROWS_PER_BLOCK * 2 * out_cols
    n_rb = -(-N // ROWS_PER_BLOCK)
    area = SECTION_ALIGN
    idx_off = _up(area + n_rb * rb_bytes, SECTION_ALIGN)
    total = _up(idx_off + 4 * n_out, SECTION_ALIGN)
    return {"area": area, "rb_bytes": rb_bytes, "rec_bytes": rec, "recs": nrec, "out_rec_bytes": out_rec,
            "out_recs": n_outrec, "idx": idx_off, "total": total, "n_rb": n_rb, "out_cols": out_cols}


def outlier_widths(n_out: int) -> list:
    """Columns of each outlier record of a row block (the last one trimmed)."""
    cols = _up(n_out, OUT_COL_ALIGN)
    return [min(OUT_COLS, cols - OUT_COLS * j) for j in range(-(-n_out // OUT_COLS))]


def _pad2(a: np.ndarray, rows: int, cols: int) -> np.ndarray:
    out = np.zeros((rows, cols), dtype=a.dtype)
    out[:a.shape[0], :a.shape[1]] = a
    return out


def _write_blob(kind: str, N: int, K: int, idx: np.ndarray, part_rows: list, vals16: np.ndarray) -> np.ndarray:
    """part_rows: the three per-row byte arrays (N x bytes) in the pages' layout."""
    n_out = int(idx.size)
    L = layout(kind, N, K, n_out)
    n_rb, nrec = L["n_rb"], L["recs"]
    rows = n_rb * ROWS_PER_BLOCK
    chunks = []
    for data, per_row in zip(part_rows, record_parts(kind)):
        b = np.ascontiguousarray(data).view(np.uint8).reshape(N, -1)
        b = _pad2(b, rows, nrec * per_row)
        # (row block, row, record, bytes) -> (row block, record, row, bytes)
        chunks.append(b.reshape(n_rb, ROWS_PER_BLOCK, nrec, per_row).transpose(0, 2, 1, 3)
                      .reshape(n_rb, nrec, ROWS_PER_BLOCK * per_row))
    dense = np.concatenate(chunks, axis=2).reshape(n_rb, nrec * L["rec_bytes"])
    pieces = [dense]
    if n_out:
        v = _pad2(np.ascontiguousarray(vals16.astype("<f2")).view(np.uint8).reshape(N, 2 * n_out),
                  rows, 2 * L["out_cols"]).reshape(n_rb, ROWS_PER_BLOCK, 2 * L["out_cols"])
        c0 = 0
        for w in outlier_widths(n_out):
            # record: (row 0..3, its w columns), row-major
            pieces.append(v[:, :, 2 * c0:2 * (c0 + w)].reshape(n_rb, ROWS_PER_BLOCK * 2 * w))
            c0 += w
    area = np.concatenate(pieces, axis=1)
    blob = np.zeros(L["total"], dtype=np.uint8)
    blob[L["area"]:L["area"] + area.size] = area.reshape(-1)
    hdr = bytearray(HEADER_BYTES)
    hdr[0:8] = MAGIC_W4 if kind == "w4" else MAGIC_W2
    struct.pack_into("<IIqqiIQ", hdr, 8, VERSION, HEADER_BYTES, N, K, n_out, G, L["total"])
    struct.pack_into("<7Q", hdr, 48, L["area"], L["rb_bytes"], L["rec_bytes"], L["recs"], L["out_rec_bytes"],
                     L["out_recs"], L["idx"])
    blob[:HEADER_BYTES] = np.frombuffer(bytes(hdr), dtype=np.uint8)
    if n_out:
        blob[L["idx"]:L["idx"] + 4 * n_out] = np.ascontiguousarray(idx.astype("<i4")).view(np.uint8)
    return blob


def read_header(blob: np.ndarray) -> dict:
    b = bytes(blob[:HEADER_BYTES])
    version, hbytes, N, K, n_out, group, total = struct.unpack_from("<IIqqiIQ", b, 8)
    area, rb_bytes, rec, recs, out_rec, out_recs, idx = struct.unpack_from("<7Q", b, 48)
    return {"magic": b[0:8], "version": version, "header_bytes": hbytes, "N": N, "K": K, "n_out": n_out,
            "group": group, "total": total, "area": area, "rb_bytes": rb_bytes, "rec_bytes": rec, "recs": recs,
            "out_rec_bytes": out_rec, "out_recs": out_recs, "idx": idx}


def _read_parts(blob: np.ndarray, kind: str):
    """The three per-row byte arrays (N x bytes, pages' layout), idx and vals."""
    h = read_header(blob)
    N, n_out = h["N"], h["n_out"]
    n_rb = -(-N // ROWS_PER_BLOCK)
    area = blob[h["area"]:h["area"] + n_rb * h["rb_bytes"]].reshape(n_rb, h["rb_bytes"])
    nrec = h["recs"]
    dense = area[:, :nrec * h["rec_bytes"]].reshape(n_rb, nrec, h["rec_bytes"])
    out, off = [], 0
    for per_row in record_parts(kind):
        w = ROWS_PER_BLOCK * per_row
        p = dense[:, :, off:off + w].reshape(n_rb, nrec, ROWS_PER_BLOCK, per_row).transpose(0, 2, 1, 3)
        out.append(np.ascontiguousarray(p.reshape(n_rb * ROWS_PER_BLOCK, nrec * per_row)[:N]))
        off += w
    if n_out:
        cols, off = [], nrec * h["rec_bytes"]
        for w in outlier_widths(n_out):
            cols.append(area[:, off:off + ROWS_PER_BLOCK * 2 * w].reshape(n_rb, ROWS_PER_BLOCK, 2 * w))
            off += ROWS_PER_BLOCK * 2 * w
        v = np.concatenate(cols, axis=2).reshape(n_rb * ROWS_PER_BLOCK, -1)[:N, :2 * n_out]
        vals = np.ascontiguousarray(v).view("<f2").astype(F64)
        idx = np.ascontiguousarray(blob[h["idx"]:h["idx"] + 4 * n_out]).view("<i4").astype(np.int32)
    else:
        vals = np.zeros((N, 0), F64)
        idx = np.zeros(0, np.int32)
    return h, out, idx, vals


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
    h, (qb, sb, zb), idx, vals = _read_parts(blob, "w4")
    assert h["magic"] == MAGIC_W4
    N, K = h["N"], h["K"]
    qb = qb[:, :K // 2].reshape(N, K // 32, 16)
    q = np.concatenate([qb & 0x0F, qb >> 4], axis=2).reshape(N, K)
    s16 = np.ascontiguousarray(sb[:, :K // 16]).view("<f2").astype(F64)
    zb = zb[:, :K // 64]
    z = np.stack([zb & 0x0F, zb >> 4], axis=2).reshape(N, K // 32)
    return q, z, s16, idx, vals


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
    h, (cb, Sb, Zb), idx, vals = _read_parts(blob, "w2")
    assert h["magic"] == MAGIC_W2
    N, K = h["N"], h["K"]
    cb = cb[:, :K // 4]
    q = np.stack([(cb >> (2 * j)) & 3 for j in range(4)], axis=2).reshape(N, K)
    S16 = np.ascontiguousarray(Sb[:, :K // 16]).view("<f2").astype(F64)
    Z16 = np.ascontiguousarray(Zb[:, :K // 16]).view("<f2").astype(F64)
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
    kind = "w4" if bytes(blob[:8]) == MAGIC_W4 else "w2"
    _, _, idx, vals = _read_parts(blob, kind)
    return idx, vals


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


# ---------------------------------------------------------------------------
# Selective weight refinement (StrataFlux paper, section 3 "Designing Precision
# for Selective Refinement": "Weight Refinement", Eq. 2 and "Channel selection";
# Appendix "StrataFlux Implementation": exact radix-sort selection)
#
#   y' = W_hat x + sum_{i in S(x)} x_i C[:, i]
#   S(x): per chunk of 1,024 consecutive input channels, the k channels with the
#         largest |x_i| (ties to the lower index; a chunk shorter than k gives all)
#   C:    the refinement matrix, 4-bit integers with scale factors.
# Readings (listed in the design notes): C is the 4-bit encoding of the weight
# residual R = W - W_hat_eff (no refinement fitting: that needs calibration
# data), quantised per input channel with the 4-bit Group-32 quantiser above
# over groups of 32 consecutive output rows; each channel's column is one
# contiguous record so that a selected column is fetched in one piece.
# ---------------------------------------------------------------------------

REFINE_CHUNK = 1024
MAGIC_RF = b"LBQRFW4C"
RF_VERSION = 1
RF_HEADER = 64


def refine_column_bytes(N: int) -> int:
    """One column record: N/2 nibble bytes, N/32 FP16 scales, N/64 zero bytes, padded to 16."""
    assert N % 64 == 0 and N > 0
    return _up(N // 2 + N // 16 + N // 64, 16)


def refine_layout(N: int, K: int) -> dict:
    cb = refine_column_bytes(N)
    return {"column_bytes": cb, "header": RF_HEADER, "total": RF_HEADER + K * cb,
            "codes": 0, "scales": N // 2, "zeros": N // 2 + N // 16}


def dequant_eff(blob: np.ndarray) -> np.ndarray:
    """The matrix the resident GEMV applies, FP64: the dense dequantised weights,
    with each outlier column replaced by its exact FP16 values."""
    Wh = dequant(blob)
    idx, vals = outliers(blob)
    if idx.size:
        Wh[:, idx] = vals
    return Wh


def pack_refine(R: np.ndarray) -> np.ndarray:
    """Quantise the N x K FP32 residual column by column (groups of 32 rows) and
    write the refinement blob:
      [0:8) magic b"LBQRFW4C"  [8:12) u32 version 1  [12:16) u32 header bytes 64
      [16:24) i64 N  [24:32) i64 K  [32:36) u32 group 32  [36:40) u32 column bytes
      [40:48) u64 total bytes  [48:64) zero
      then column i at 64 + i * column_bytes: nibbles (byte b of group g =
      q_{32g+b} | q_{32g+b+16} << 4), FP16 scales, zero points z_{2m} | z_{2m+1} << 4."""
    R = np.asarray(R, dtype=np.float32)
    N, K = R.shape
    L = refine_layout(N, K)
    q, z, s = quantise_w4(R.astype(F64).T)           # rows = input channels, groups along N
    s16 = fp16_round(s)
    codes, zeros = pack_nibbles(q), pack_zero_points(z)
    blob = np.zeros(L["total"], dtype=np.uint8)
    blob[0:8] = np.frombuffer(MAGIC_RF, dtype=np.uint8)
    hdr = np.array([RF_VERSION, RF_HEADER], dtype="<u4").view(np.uint8)
    blob[8:16] = hdr
    blob[16:32] = np.array([N, K], dtype="<i8").view(np.uint8)
    blob[32:40] = np.array([G, L["column_bytes"]], dtype="<u4").view(np.uint8)
    blob[40:48] = np.array([L["total"]], dtype="<u8").view(np.uint8)
    cb = L["column_bytes"]
    cols = blob[RF_HEADER:].reshape(K, cb)
    cols[:, 0:N // 2] = codes
    cols[:, N // 2:N // 2 + N // 16] = np.ascontiguousarray(s16.astype("<f2")).view(np.uint8).reshape(K, N // 16)
    cols[:, N // 2 + N // 16:N // 2 + N // 16 + N // 64] = zeros
    return blob


def unpack_refine(blob: np.ndarray, cols=None) -> np.ndarray:
    """C (N x K, FP64) = (q - z) * s16 of every column record (or only of the
    listed columns, in that order: N x len(cols))."""
    assert bytes(blob[:8]) == MAGIC_RF
    N = int(blob[16:24].view("<i8")[0])
    K = int(blob[24:32].view("<i8")[0])
    cb = int(blob[36:40].view("<u4")[0])
    sel = np.arange(K) if cols is None else np.asarray(cols, dtype=np.int64)
    K = sel.size
    cols = blob[RF_HEADER:].reshape(-1, cb)[sel]
    qb = cols[:, :N // 2].reshape(K, N // 32, 16)
    q = np.concatenate([qb & 0x0F, qb >> 4], axis=2).astype(F64)          # (K, N/32, 32)
    s16 = np.ascontiguousarray(cols[:, N // 2:N // 2 + N // 16]).view("<f2").astype(F64)
    zb = cols[:, N // 2 + N // 16:N // 2 + N // 16 + N // 64]
    z = np.stack([zb & 0x0F, zb >> 4], axis=2).reshape(K, N // 32).astype(F64)
    return ((q - z[..., None]) * s16[..., None]).reshape(K, N).T


def select_refine(x: np.ndarray, k: int) -> np.ndarray:
    """S(x): per chunk of 1,024 channels the min(k, chunk length) largest |x_i|,
    ties to the lower index; ascending channel indices.

    |x_i| is ranked by the magnitude field of x_i's FP16 encoding (the 15 bits
    below the sign): for finite values that order is the order of |x_i|, and it
    also places the non-finite values, which the pages leave open: an infinity
    ranks above every finite value and a NaN above an infinity."""
    a = (np.asarray(x, dtype=np.float16).reshape(-1).view(np.uint16) & 0x7FFF).astype(F64)
    out = []
    for c0 in range(0, a.size, REFINE_CHUNK):
        chunk = a[c0:c0 + REFINE_CHUNK]
        out.append(top_indices(chunk, min(k, chunk.size)) + c0)
    return np.concatenate(out).astype(np.int32) if out else np.zeros(0, np.int32)


def refine_apply(blob: np.ndarray, x: np.ndarray, idx: np.ndarray, y: np.ndarray) -> np.ndarray:
    """y + sum_j x_{idx_j} C[:, idx_j], FP64, terms added in the order of idx."""
    idx = np.asarray(idx, dtype=np.int64)
    C = unpack_refine(blob, idx)                       # the selected columns only
    xv = np.asarray(x, dtype=np.float16).astype(F64).reshape(-1)
    out = np.asarray(y, dtype=F64).copy()
    for j, i in enumerate(idx):
        out = out + xv[i] * C[:, j]
    return out


# ---------------------------------------------------------------------------
# Fused embedding row gather (SPECTRA article, section 4.3 "SpectraFusedEmbedding:
# Dynamic Row-Gather Dequantization"): only the rows of the requested token ids
# are dequantised.  Reading: an output row is the row of the matrix the blob
# applies (outlier columns exact), in FP64, rounded once to the output type.
# ---------------------------------------------------------------------------

def embed(blob: np.ndarray, ids, out_dtype=np.float16) -> np.ndarray:
    ids = np.asarray(ids, dtype=np.int64)
    rows = dequant(blob, ids)
    idx, vals = outliers(blob)
    if idx.size:
        rows[:, idx] = vals[ids]
    return fp16_round(rows) if out_dtype == np.float16 else rows.astype(np.float32)


# ---------------------------------------------------------------------------
# 4-bit Group-32 KV cache (SPECTRA article, section 4.5 "Group-32 Microscaled
# 4-Bit Key-Value Cache": key and value states quantised into asymmetric 4-bit
# Group-32 blocks in place).  Readings: the quantiser of section 3.4 applied to
# the FP16 states (FP64 statistics, round half to even); each cached token row
# of `width` = heads x head_dim values is one record: width/2 nibble bytes,
# width/32 FP16 scales, width/64 zero-point bytes, padded to 16 bytes; a read
# returns (q - z) * s16 rounded once to FP16.
# ---------------------------------------------------------------------------

def kv_record_bytes(width: int) -> int:
    assert width % 64 == 0 and width > 0
    return _up(width // 2 + width // 16 + width // 64, 16)


def kv_quantize(X: np.ndarray) -> np.ndarray:
    """Records (rows x kv_record_bytes) of FP16 rows X (rows x width)."""
    X = np.asarray(X, dtype=np.float16)
    rows, width = X.shape
    q, z, s = quantise_w4(X.astype(F64))
    out = np.zeros((rows, kv_record_bytes(width)), dtype=np.uint8)
    out[:, :width // 2] = pack_nibbles(q)
    out[:, width // 2:width // 2 + width // 16] = \
        np.ascontiguousarray(fp16_round(s).astype("<f2")).view(np.uint8).reshape(rows, width // 16)
    out[:, width // 2 + width // 16:width // 2 + width // 16 + width // 64] = pack_zero_points(z)
    return out


def kv_dequant(rec: np.ndarray, width: int) -> np.ndarray:
    """FP16 rows (rows x width) read back from records."""
    rec = np.asarray(rec, dtype=np.uint8)
    rows = rec.shape[0]
    qb = rec[:, :width // 2].reshape(rows, width // 32, 16)
    q = np.concatenate([qb & 0x0F, qb >> 4], axis=2).astype(F64)
    s16 = np.ascontiguousarray(rec[:, width // 2:width // 2 + width // 16]).view("<f2").astype(F64)
    zb = rec[:, width // 2 + width // 16:width // 2 + width // 16 + width // 64]
    z = np.stack([zb & 0x0F, zb >> 4], axis=2).reshape(rows, width // 32).astype(F64)
    return fp16_round(((q - z[..., None]) * s16[..., None]).reshape(rows, width))
