"""GPU parity of the batched 2-bit codebook GEMM with FP16 outlier columns
(M activation rows per call, CUDA-core passes of 2 / 4 / 8 rows) against the
FP64 oracle, through the C ABI: element by element on ragged shapes for every
pass structure (M = 1..64, odd remainders), FP16 output, leading dimensions,
and sampled rows of the Llama-3-8B gate / down projections with the top 3.5 %
outlier columns."""
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
    lbq.gemm_w2cb_outlier_smallM(to_dev(blob), M, N, K, n_out, to_dev(X), X.shape[1], Y, ldy)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    return Y.float().cpu().numpy()


def _case(seed, M, N, K, n_out):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    X = rng.standard_normal((M, K)).astype(np.float16)
    X[:, rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
    idx = np.sort(rng.choice(K, size=n_out, replace=False)).astype(np.int32)
    return W, X, idx


@pytest.mark.parametrize("M", [2, 3, 4, 5, 8, 9, 13, 16, 33, 64])
def test_small_shapes_elementwise(lbq, M):
    N, K, n_out = 70, 2112, 77                      # ragged row block, partial record, trimmed outlier record
    W, X, idx = _case(300 + M, M, N, K, n_out)
    blob = lbq.pack_w2cb(W, idx)
    ref = O.gemm(O.pack_w2cb(W, idx), X)
    assert_close(_gemm(lbq, blob, M, N, K, n_out, X), ref, what="w2 M=%d" % M)
    assert_close(_gemm(lbq, blob, M, N, K, n_out, X, f32=False), ref, fp16_out=True, what="w2 M=%d f16" % M)


def test_leading_dimensions_and_no_outliers(lbq):
    M, N, K = 6, 129, 1024
    W, Xfull, _ = _case(7, M, N, K + 40, 0)
    W = W[:, :K].copy()
    blob = lbq.pack_w2cb(W, np.zeros(0, np.int32))
    Y = _gemm(lbq, blob, M, N, K, 0, Xfull, ldy=N + 5)
    assert_close(Y[:, :N], O.gemm(O.pack_w2cb(W, np.zeros(0, np.int32)), Xfull[:, :K]), what="w2 ld")
    assert np.isnan(Y[:, N:]).all()                 # padding columns untouched


@pytest.mark.parametrize("li", [4, 6])              # gate_proj 14336 x 4096, down_proj 4096 x 14336
@pytest.mark.parametrize("M", [4, 8])
def test_llama8b_sampled(lbq, li, M):
    name, N, K = synth.LLAMA3_8B_LINEARS[li]
    W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)
    idx = O.select_outliers_impact(W, synth.profile_vectors(K, workload=synth.WL_LLAMA8B_W2, layer_id=li))
    X = synth.activations(M, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)
    Y = _gemm(lbq, lbq.pack_w2cb(W, idx), M, N, K, len(idx), X)
    rows = np.unique(np.concatenate([[0, 1, N - 2, N - 1], np.random.default_rng(M + li).choice(N, size=128)]))
    assert_close(Y[:, rows], O.gemm(O.pack_w2cb(W[rows], idx), X), what="w2 %s M=%d" % (name, M))


def test_grouped_equals_oracle(lbq):
    M = 4
    probs, checks = [], []
    for i, (N, K, n_out) in enumerate([(37, 1088, 5), (130, 4096, 143), (64, 3072, 0)]):
        W, X, idx = _case(400 + i, M, N, K, n_out)
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda:0")
        probs.append((to_dev(lbq.pack_w2cb(W, idx)), N, K, n_out, to_dev(X), K, Y, N))
        checks.append((Y, O.gemm(O.pack_w2cb(W, idx), X)))
    lbq.gemv_grouped(lbq.LBQ_KIND_W2CB, probs, M=M)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for Y, ref in checks:
        assert_close(Y.cpu().numpy(), ref, what="w2 grouped M=4")
