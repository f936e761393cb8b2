"""GPU parity of the tensor-core small-M 4-bit GEMM (16 <= M <= 64, no outlier
columns) against the FP64 oracle, element by element: ragged row tiles (N not a
multiple of 128), partial 1024-k blocks, K split over clusters of 1..8 CTAs,
activation rows padded to the MMA width, leading dimensions, FP16 output.
The weights are dequantised to FP16 before the FP32-accumulating product, so
each weight carries one FP16 rounding; the bound stays the oracle tolerance."""
import numpy as np
import pytest

from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _case(seed, M, N, K):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    W *= rng.uniform(0.5, 2.0, size=(N, 1)).astype(np.float32)
    X = rng.standard_normal((M, K)).astype(np.float16)
    X[:, rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
    return W, X


def _run(lbq, blob, M, N, K, X, ldx=None, ldy=None, f32=True):
    ldx = ldx or K
    ldy = ldy or N
    Xp = np.zeros((M, ldx), np.float16)
    Xp[:, :K] = X
    Y = torch.full((M, ldy), float("nan"), dtype=torch.float32 if f32 else torch.float16, device="cuda:0")
    lbq.gemm_w4a16_smallM(to_dev(blob), M, N, K, 0, to_dev(Xp), ldx, Y, ldy)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    return Y.float().cpu().numpy()


# (M, N, K): N ragged against the 128-row tile; K with partial k-blocks; the
# cluster size is min(8, SMs // tiles, k-blocks), so small N spreads K over 8 CTAs
SHAPES = [(16, 128, 1024), (16, 1, 64), (17, 70, 1088), (32, 129, 3072), (33, 300, 2112), (48, 257, 4096),
          (64, 1000, 1024), (64, 128, 8192), (40, 600, 7168), (16, 4100, 1024)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_elementwise(lbq, M, N, K):
    W, X = _case(M * 7 + N + K, M, N, K)
    blob = lbq.pack_w4(W)
    ref = O.gemm(O.pack_w4(W), X)
    assert_close(_run(lbq, blob, M, N, K, X), ref, what="mma M=%d N=%d K=%d" % (M, N, K))


def test_fp16_output_and_leading_dimensions(lbq):
    M, N, K = 24, 200, 2048
    W, X = _case(5, M, N, K)
    blob = lbq.pack_w4(W)
    ref = O.gemm(O.pack_w4(W), X)
    Y = _run(lbq, blob, M, N, K, X, ldx=K + 40, ldy=N + 5, f32=False)
    assert_close(Y[:, :N], ref, fp16_out=True, what="mma f16 ld")
    assert np.isnan(Y[:, N:]).all()


def test_deterministic_across_calls(lbq):
    """Split-K partials are added in rank order: identical bits on every call."""
    M, N, K = 64, 256, 8192
    W, X = _case(9, M, N, K)
    blob = lbq.pack_w4(W)
    a = _run(lbq, blob, M, N, K, X)
    for _ in range(3):
        assert np.array_equal(_run(lbq, blob, M, N, K, X), a)


def test_grouped_and_launch_count(lbq):
    M = 32
    probs, checks = [], []
    for i, (N, K) in enumerate([(300, 2048), (129, 4096)]):
        W, X = _case(20 + i, M, N, K)
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda:0")
        probs.append((to_dev(lbq.pack_w4(W)), N, K, 0, to_dev(X), K, Y, N))
        checks.append((Y, O.gemm(O.pack_w4(W), X)))
    assert lbq.gemv_grouped_launches(lbq.LBQ_KIND_W4, probs, M=M) == 2
    lbq.gemv_grouped(lbq.LBQ_KIND_W4, probs, M=M)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for Y, ref in checks:
        assert_close(Y.cpu().numpy(), ref, what="mma grouped")
