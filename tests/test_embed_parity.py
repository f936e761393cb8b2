"""GPU parity of the fused embedding row gather (SPECTRA article, section 4.3)
against the oracle, bit for bit: both kinds, with and without outlier columns,
FP16 and FP32 outputs, a ragged vocabulary and a partial last record,
repeated ids, and the device-side error reports; plus argument checks on CPU."""
import numpy as np
import pytest

from oracle import lbq_oracle as O

from gpu_util import to_dev


def test_gather_argument_checks_without_gpu(lbq):
    L = lbq.lib()
    assert L.lbq_embed_gather(0, None, 8, 64, 0, 16, 1, 16, 0, None) == 1
    assert L.lbq_embed_gather(5, 16, 8, 64, 0, 16, 1, 16, 0, None) == 10        # unknown kind
    assert L.lbq_embed_gather(0, 16, 8, 96, 0, 16, 1, 16, 0, None) == 2         # D % 64
    assert L.lbq_embed_gather(0, 16, 8, 64, 65, 16, 1, 16, 0, None) == 2        # n_out > D
    assert L.lbq_embed_gather(0, 16, 8, 64, 0, 16, 0, 16, 0, None) == 0         # T = 0: nothing to do


def _gather(lbq, kind, blob, V, D, n_out, ids, f16):
    torch = pytest.importorskip("torch")
    out = torch.full((len(ids), D), float("nan"), dtype=torch.float16 if f16 else torch.float32, device="cuda:0")
    k = lbq.LBQ_KIND_W4 if kind == "w4" else lbq.LBQ_KIND_W2CB
    lbq.embed_gather(k, to_dev(blob), V, D, n_out, to_dev(np.asarray(ids, np.int32)), out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["w4", "w2"])
@pytest.mark.parametrize("V,D,n_out", [(13, 64, 0), (37, 1088, 0), (37, 1088, 21), (130, 4096, 143), (9, 2112, 300)])
@pytest.mark.parametrize("f16", [True, False])
def test_gather_bitexact(lbq, kind, V, D, n_out, f16):
    rng = np.random.default_rng(V + D + n_out)
    W = (rng.standard_normal((V, D)) * 0.02).astype(np.float32)
    idx = np.sort(rng.choice(D, size=n_out, replace=False)).astype(np.int32)
    pack, opack = (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)
    ids = np.concatenate([[0, V - 1, V - 1], rng.integers(0, V, size=9)]).astype(np.int32)   # ends and repeats
    got = _gather(lbq, kind, pack(W, idx), V, D, n_out, ids, f16)
    assert lbq.device_error() == 0
    ref = O.embed(opack(W, idx), ids, out_dtype=np.float16 if f16 else np.float32)
    assert np.array_equal(got.view(np.uint16 if f16 else np.uint32), ref.view(np.uint16 if f16 else np.uint32))


@pytest.mark.gpu
def test_gather_large_table_sampled(lbq):
    """A 32768 x 4096 4-bit table (every row streams through the same kernel as a
    128,256-row vocabulary), 64 token ids."""
    rng = np.random.default_rng(5)
    V, D = 32768, 4096
    W = (rng.standard_normal((V, D), dtype=np.float32) * 0.02)
    blob = lbq.pack_w4(W)
    ids = rng.integers(0, V, size=64).astype(np.int32)
    got = _gather(lbq, "w4", blob, V, D, 0, ids, True)
    assert lbq.device_error() == 0
    ref = O.embed(O.pack_w4(W[np.sort(np.unique(ids))]), np.searchsorted(np.sort(np.unique(ids)), ids))
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))


@pytest.mark.gpu
def test_gather_reports_bad_id_and_header(lbq):
    torch = pytest.importorskip("torch")
    V, D = 8, 128
    W = (np.random.default_rng(1).standard_normal((V, D)) * 0.02).astype(np.float32)
    blob = to_dev(lbq.pack_w4(W))
    out = torch.full((2, D), 7.0, dtype=torch.float16, device="cuda:0")
    lbq.embed_gather(lbq.LBQ_KIND_W4, blob, V, D, 0, to_dev(np.array([1, V], np.int32)), out)
    assert lbq.device_error() == 9                                   # LBQ_ERR_VALUE
    assert bool((out[1] == 7.0).all())                                # that row is untouched
    lbq.embed_gather(lbq.LBQ_KIND_W4, blob, V + 4, D, 0, to_dev(np.array([1], np.int32)), out[:1])
    assert lbq.device_error() == 6                                   # LBQ_ERR_FORMAT (V differs)
