"""GPU parity of the small-M batched 4-bit GEMM (M activation rows per call)."""
import numpy as np
import pytest

from bit_weight_only_lbq_gb300 import synth
from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _gemm(lbq, blob, M, N, K, n_out, X, f32=True, ldy=None):
    ldy = ldy or N
    Y = torch.full((M, ldy), float("nan"), dtype=torch.float32 if f32 else torch.float16, device="cuda:0")
    lbq.gemm_w4a16_smallM(to_dev(blob), M, N, K, n_out, to_dev(X), X.shape[1], Y, ldy)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    return Y.float().cpu().numpy()


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 9, 16, 33, 64])
def test_small_shapes(lbq, M):
    rng = np.random.default_rng(M)
    N, K, n_out = 70, 1600 - 1600 % 64, 21
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    idx = np.sort(rng.choice(K, size=n_out, replace=False)).astype(np.int32)
    X = rng.standard_normal((M, K)).astype(np.float16)
    ref = O.gemm(O.pack_w4(W, idx), X)
    blob = lbq.pack_w4(W, idx)
    Y = _gemm(lbq, blob, M, N, K, n_out, X)
    assert_close(Y, ref, what="M=%d" % M)
    Yh = _gemm(lbq, blob, M, N, K, n_out, X, f32=False)
    assert_close(Yh, ref, fp16_out=True, what="M=%d f16" % M)


def test_leading_dimensions(lbq):
    rng = np.random.default_rng(11)
    M, N, K = 5, 40, 256
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    Xfull = rng.standard_normal((M, K + 24)).astype(np.float16)
    blob = lbq.pack_w4(W)
    Y = _gemm(lbq, blob, M, N, K, 0, Xfull, ldy=N + 3)
    ref = O.gemm(O.pack_w4(W), Xfull[:, :K])
    assert_close(Y[:, :N], ref, what="ld")
    assert np.isnan(Y[:, N:]).all()                 # padding columns untouched


@pytest.mark.parametrize("name,N,K", [("gate_proj", 14336, 4096), ("down_proj", 4096, 14336)])
@pytest.mark.parametrize("M", synth.SMALL_M_VALUES)
def test_gate_down_small_m_sampled(lbq, name, N, K, M):
    li = 4 if name == "gate_proj" else 6
    W = synth.weights_heavy_cols(N, K, workload=synth.WL_SMALL_M, layer_id=li)
    X = synth.activations(M, K, workload=synth.WL_SMALL_M, layer_id=li)
    Y = _gemm(lbq, lbq.pack_w4(W), M, N, K, 0, X)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(M).choice(N, size=128)]))
    ref = O.gemm(O.pack_w4(W[rows]), X)
    assert_close(Y[:, rows], ref, what="small M %s M=%d" % (name, M))


def test_wide_k_falls_back_to_row_passes(lbq):
    rng = np.random.default_rng(12)
    M, N, K = 3, 9, 65536
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    X = rng.standard_normal((M, K)).astype(np.float16)
    Y = _gemm(lbq, lbq.pack_w4(W), M, N, K, 0, X)
    assert_close(Y, O.gemm(O.pack_w4(W), X), what="wide K")
