"""The C++ packers and outlier selectors against the oracle, byte for byte (CPU)."""
import numpy as np
import pytest

from bit_weight_only_lbq_gb300 import synth
from oracle import lbq_oracle as O

from degenerate_inputs import degenerate_matrix


@pytest.mark.parametrize("N,K", [(1, 64), (3, 128), (17, 192), (64, 1024), (33, 4160)])
def test_w4_pack_bitexact(lbq, N, K):
    W = synth.random_matrix(N, K, seed=N * 7 + K, scale=0.02)
    assert np.array_equal(lbq.pack_w4(W), O.pack_w4(W))


@pytest.mark.parametrize("N,K", [(1, 64), (3, 128), (17, 192), (64, 1024), (33, 4160)])
def test_w2_pack_bitexact(lbq, N, K):
    W = synth.random_matrix(N, K, seed=N * 5 + K, scale=0.02)
    assert np.array_equal(lbq.pack_w2cb(W), O.pack_w2cb(W))


def test_pack_with_outliers_bitexact(lbq):
    W = synth.weights_heavy_cols(40, 1024, workload=synth.WL_LLAMA8B_W4, layer_id=99)
    idx = O.select_outliers_w4(W)
    assert np.array_equal(lbq.select_outliers_w4(W), idx)
    assert np.array_equal(lbq.pack_w4(W, idx), O.pack_w4(W, idx))
    X = synth.profile_vectors(1024, workload=synth.WL_LLAMA8B_W2, layer_id=99)
    idx2 = O.select_outliers_impact(W, X)
    assert np.array_equal(lbq.select_outliers_impact(W, X), idx2)
    assert len(idx2) == int(0.035 * 1024)
    assert np.array_equal(lbq.pack_w2cb(W, idx2), O.pack_w2cb(W, idx2))


def test_golden_groups_through_cpp(lbq, golden):
    g = golden("w4_worked_example.txt")
    w = np.array([float(v) for v in g["w_group0"] + g["w_group1"]], dtype=np.float32)[None, :]
    blob = lbq.pack_w4(w)
    rec = lbq.blob_layout(lbq.LBQ_KIND_W4, 1, 64, 0)["area"]
    assert blob[rec:rec + 32].tolist() == [int(v, 16) for v in g["qweight_bytes"]]
    assert blob[rec + 2304] == int(g["zero_bytes"][0], 16)
    g2 = golden("w2_worked_example.txt")
    w = np.empty((1, 64), np.float32)
    w[0, :32] = [O.C16[int(c)] / 16 + 0.125 for c in g2["codes_group0"]]
    w[0, 32:] = 0.25
    blob = lbq.pack_w2cb(w)
    rec = lbq.blob_layout(lbq.LBQ_KIND_W2CB, 1, 64, 0)["area"]
    assert blob[rec:rec + 16].tolist() == [int(v, 16) for v in g2["code_bytes"]]
    assert blob[rec + 1024:rec + 1028].view("<u2").tolist() == [int(v, 16) for v in g2["S_f16_bits"]]
    assert blob[rec + 1280:rec + 1284].view("<u2").tolist() == [int(v, 16) for v in g2["Z_f16_bits"]]


def test_layouts_match_oracle(lbq):
    for kind, name in ((lbq.LBQ_KIND_W4, "w4"), (lbq.LBQ_KIND_W2CB, "w2")):
        for N, K, n in ((1, 64, 0), (3, 64, 2), (1000, 4160, 143), (7, 65536, 8192)):
            a = lbq.blob_layout(kind, N, K, n)
            b = O.layout(name, N, K, n)
            assert a == {k: b[k] for k in a}


def test_llama8b_qproj_rows_bitexact(lbq):
    """A slice of the Llama-3-8B q_proj (full K = 4096) with the W4 outlier variant."""
    W = synth.weights_heavy_cols(4096, 4096, workload=synth.WL_LLAMA8B_W4, layer_id=0)[:256]
    idx = lbq.select_outliers_w4(W)
    assert np.array_equal(idx, O.select_outliers_w4(W))
    assert np.array_equal(lbq.pack_w4(W, idx), O.pack_w4(W, idx))


@pytest.mark.parametrize("kind", ["w4", "w2"])
@pytest.mark.parametrize("N,K,n_out", [(4, 64, 0), (17, 192, 7), (64, 1088, 40), (33, 4160, 300)])
def test_dequant_host_matches_oracle(lbq, kind, N, K, n_out):
    """lbq_dequant_host: the matrix a blob applies, FP64 then one FP32 rounding."""
    W = synth.random_matrix(N, K, seed=N + K + n_out, scale=0.02)
    idx = np.sort(np.random.default_rng(N).choice(K, size=n_out, replace=False)).astype(np.int32)
    pack, opack = (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)
    got = lbq.dequant_host(pack(W, idx))
    assert np.array_equal(got, O.dequant_eff(opack(W, idx)).astype(np.float32))


@pytest.mark.parametrize("N,K", [(64, 1), (64, 3), (128, 1088), (192, 2049), (4096, 17)])
def test_refine_pack_bitexact(lbq, N, K):
    R = synth.random_matrix(N, K, seed=N * 3 + K, scale=1e-3)
    R[:, 0] = 0.25                                   # a constant column (reconstructs to 0)
    blob = lbq.pack_refine(R)
    assert blob.size == lbq.lib().lbq_refine_packed_bytes(N, K) == O.refine_layout(N, K)["total"]
    assert np.array_equal(blob, O.pack_refine(R))


def test_refine_golden_through_cpp(lbq, golden):
    g = golden("refine_column_example.txt")
    q0 = np.array([int(t) for t in g["col0_q_group0"]])
    R = np.zeros((64, 2), np.float32)
    R[:32, 0] = (q0 - 3) / 1024.0
    R[:, 1] = 0.5
    blob = lbq.pack_refine(R)
    cb = int(g["column_bytes"][0])
    assert blob[:64].tolist() == [int(v, 16) for v in g["header"]]
    assert blob[64:64 + cb].tolist() == [int(v, 16) for v in g["col0_record"]]
    assert blob[64 + cb:64 + 2 * cb].tolist() == [int(v, 16) for v in g["col1_record"]]


def test_refine_host_argument_checks(lbq):
    L = lbq.lib()
    assert L.lbq_refine_packed_bytes(96, 4) == 0           # N % 64
    assert L.lbq_refine_packed_bytes(64, 0) == 0
    assert L.lbq_refine_packed_bytes(64, 65537) == 0
    assert L.lbq_refine_selected_count(2112, 8) == 8 + 8 + 8
    assert L.lbq_refine_selected_count(2112, 100) == 100 + 100 + 64
    assert L.lbq_refine_selected_count(64, 0) == 0 and L.lbq_refine_selected_count(64, 257) == 0
    R = np.full((64, 2), np.nan, np.float32)
    buf = np.empty(L.lbq_refine_packed_bytes(64, 2), np.uint8)
    assert L.lbq_pack_refine(R.ctypes.data, 64, 2, buf.ctypes.data, buf.size) == 9   # LBQ_ERR_VALUE
    assert L.lbq_pack_refine(R.ctypes.data, 64, 2, buf.ctypes.data, buf.size - 1) == 5  # too small
    bad = np.zeros(256, np.uint8)
    out = np.empty((1, 64), np.float32)
    assert L.lbq_dequant_host(bad.ctypes.data, bad.size, out.ctypes.data) == 6        # LBQ_ERR_FORMAT


@pytest.mark.parametrize("family", ["mixed", "tiny", "large"])
def test_degenerate_groups_bitexact(lbq, family):
    """Zero, constant, one-sided, exact-tie, lone-spike, two-valued, sub-FP16 and
    large groups, a ragged last record: the C++ packers and the host dequantiser
    byte-identical to the oracle."""
    W = degenerate_matrix(6, 384, family)
    assert np.array_equal(lbq.pack_w4(W), O.pack_w4(W))
    assert np.array_equal(lbq.pack_w2cb(W), O.pack_w2cb(W))
    idx = np.array([0, 40, 200, 233, 383], np.int32)         # outlier columns inside degenerate groups
    assert np.array_equal(lbq.pack_w4(W, idx), O.pack_w4(W, idx))
    assert np.array_equal(lbq.pack_w2cb(W, idx), O.pack_w2cb(W, idx))
    # and the host dequantiser reads those bytes as the oracle does
    for kind, pack in (("w4", O.pack_w4), ("w2", O.pack_w2cb)):
        blob = pack(W, idx)
        assert np.array_equal(lbq.dequant_host(blob), O.dequant_eff(blob).astype(np.float32)), kind


def test_dequant_host_rejects_bad_blobs(lbq):
    """Bad blobs get the C call's statuses before anything is sized from the header:
    shorter than the header, or than the header says (N inflated, truncated):
    LBQ_ERR_BUFFER_TOO_SMALL; not this library's format: LBQ_ERR_FORMAT."""
    W = synth.random_matrix(8, 128, seed=5, scale=0.02)
    for pack in (lbq.pack_w4, lbq.pack_w2cb):
        b = pack(W, np.array([3], np.int32))
        huge = b.copy()
        huge[16:24] = np.frombuffer(np.int64(10 ** 6).tobytes(), np.uint8)    # N far beyond the blob
        for bad, status in ((b[:20], 5), (b[:-16], 5), (huge, 5), (np.zeros(256, np.uint8), 6)):
            with pytest.raises(lbq.LbqError) as e:
                lbq.dequant_host(bad)
            assert e.value.status == status
        # the C entry point itself answers the same, without writing (nothing to write into)
        L = lbq.lib()
        one = np.zeros(1, np.float32)
        for bad, status in ((b[:20], 5), (b[:-16], 5), (huge, 5), (np.zeros(256, np.uint8), 6)):
            assert L.lbq_dequant_host(bad.ctypes.data, bad.size, one.ctypes.data) == status
