"""GPU parity of the tensor-core small-M GEMMs (16 <= M <= 64) against the FP64
oracle, element by element, for both weight formats: 4-bit (weights dequantised
into tensor memory, 128-row tiles, K split over a cluster when the tiles leave
SMs idle) and 2-bit codebook (weights as the 256-wide operand in shared memory, 256-row
tiles and 256-k chunks split over a cluster, each CTA's range spanning at most
two tiles with one accumulator each; taller matrices go in slabs of tiles, one
launch each; the exact FP16 outlier columns are extra 64-column stages of the
same accumulation, their values copied straight into the operand stage and the
activations gathered by index).  The 4-bit kernel adds the outlier columns
in its epilogue (FP32 FMAs on the CUDA cores, by the CTA that writes y).  The
shapes cover: N ragged against both tile
sizes (and smaller than one row block), K with a partial 1024-k record and a
partial chunk, M from 16 to 64, CTA ranges that span two tiles, a single tile
whose K is split over a whole cluster, two slabs, leading dimensions, FP16
output, repeatable bits; with outliers: one column, a trimmed last outlier
record (8 columns wide), exactly one full record, two and four records, every
column an outlier, the first and last channel.
The weights are dequantised to FP16 before the FP32-accumulating product, so
each weight carries one FP16 rounding; the bound stays the oracle tolerance."""
import numpy as np
import pytest

from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

NONE = np.zeros(0, np.int32)


def _case(seed, M, N, K):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    W *= rng.uniform(0.5, 2.0, size=(N, 1)).astype(np.float32)
    X = rng.standard_normal((M, K)).astype(np.float16)
    X[:, rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
    return W, X


def _pack(lbq, kind, W):
    return (lbq.pack_w4(W), O.pack_w4(W)) if kind == "w4" else (lbq.pack_w2cb(W, NONE), O.pack_w2cb(W, NONE))


def _run(lbq, kind, blob, M, N, K, X, ldx=None, ldy=None, f32=True):
    ldx = ldx or K
    ldy = ldy or N
    Xp = np.zeros((M, ldx), np.float16)
    Xp[:, :K] = X
    Y = torch.full((M, ldy), float("nan"), dtype=torch.float32 if f32 else torch.float16, device="cuda:0")
    f = lbq.gemm_w4a16_smallM if kind == "w4" else lbq.gemm_w2cb_outlier_smallM
    f(to_dev(blob), M, N, K, 0, to_dev(Xp), ldx, Y, ldy)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    return Y.float().cpu().numpy()


# (M, N, K): ragged tiles, partial records, one tile split over a cluster, many
# tiles (2-bit: CTA ranges that span two tiles, both accumulators in use; 4-bit:
# a CTA per tile, 80-112 tiles), and more tiles than one launch takes (two slabs)
SHAPES = [(16, 256, 1024), (16, 1, 64), (17, 70, 1088), (32, 257, 3072), (33, 300, 2112), (48, 513, 4096),
          (64, 1000, 1024), (64, 256, 8192), (40, 600, 7168), (16, 4100, 1024), (24, 9000, 2048),
          (64, 14336, 1024), (20, 4096, 4096), (16, 80000, 64), (16, 14336, 1024), (32, 10000, 2048)]


@pytest.mark.parametrize("kind", ["w4", "w2"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_elementwise(lbq, kind, M, N, K):
    W, X = _case(M * 7 + N + K, M, N, K)
    blob, ref_blob = _pack(lbq, kind, W)
    ref = O.gemm(ref_blob, X)
    assert_close(_run(lbq, kind, blob, M, N, K, X), ref, what="mma %s M=%d N=%d K=%d" % (kind, M, N, K))


@pytest.mark.parametrize("kind", ["w4", "w2"])
def test_fp16_output_and_leading_dimensions(lbq, kind):
    M, N, K = 24, 200, 2048
    W, X = _case(5, M, N, K)
    blob, ref_blob = _pack(lbq, kind, W)
    ref = O.gemm(ref_blob, X)
    Y = _run(lbq, kind, blob, M, N, K, X, ldx=K + 40, ldy=N + 5, f32=False)
    assert_close(Y[:, :N], ref, fp16_out=True, what="mma %s f16 ld" % kind)
    assert np.isnan(Y[:, N:]).all()


@pytest.mark.parametrize("kind", ["w4", "w2"])
def test_deterministic_across_calls(lbq, kind):
    """Split-K partials are added in rank order: identical bits on every call."""
    M, N, K = 64, 256, 8192
    W, X = _case(9, M, N, K)
    blob, _ = _pack(lbq, kind, W)
    a = _run(lbq, kind, blob, M, N, K, X)
    for _ in range(3):
        assert np.array_equal(_run(lbq, kind, blob, M, N, K, X), a)


def test_grouped_and_launch_count(lbq):
    M = 32
    probs, checks = [], []
    for i, (N, K) in enumerate([(300, 2048), (129, 4096)]):
        W, X = _case(20 + i, M, N, K)
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda:0")
        probs.append((to_dev(lbq.pack_w4(W)), N, K, 0, to_dev(X), K, Y, N))
        checks.append((Y, O.gemm(O.pack_w4(W), X)))
    assert lbq.gemv_grouped_launches(lbq.LBQ_KIND_W4, probs, M=M) == 2
    big = [(probs[0][0], 80000, 64, 0, probs[0][4], 64, probs[0][6], 80000)]
    assert lbq.gemv_grouped_launches(lbq.LBQ_KIND_W2CB, big, M=16) == 2   # 2-bit: two slabs of tiles
    lbq.gemv_grouped(lbq.LBQ_KIND_W4, probs, M=M)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for Y, ref in checks:
        assert_close(Y.cpu().numpy(), ref, what="mma grouped")


def _idx(seed, K, n_out):
    rng = np.random.default_rng(seed)
    if n_out >= 2:   # the first and the last channel are always among them
        rest = rng.choice(np.arange(1, K - 1), size=n_out - 2, replace=False)
        return np.sort(np.concatenate([[0, K - 1], rest])).astype(np.int32)
    return np.sort(rng.choice(K, size=n_out, replace=False)).astype(np.int32)


def _run_out(lbq, blob, M, N, K, n_out, X, f32=True, kind="w2"):
    Y = torch.full((M, N), float("nan"), dtype=torch.float32 if f32 else torch.float16, device="cuda:0")
    f = lbq.gemm_w4a16_smallM if kind == "w4" else lbq.gemm_w2cb_outlier_smallM
    f(to_dev(blob), M, N, K, n_out, to_dev(X), K, Y, N)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    return Y.float().cpu().numpy()


# (M, N, K, n_out): one outlier column; 77 (a trimmed last record, two 64-column
# stages); 256 (one full record); 257 (a full record and an 8-column one); 501 over
# two records at K = 14336; 1000 (four records, four outlier chunks); every column
# an outlier; outliers with two tiles per CTA range (2-bit at 9000 and 10000
# rows) and with two slabs
OUT_SHAPES = [(16, 300, 1024, 1), (17, 70, 2112, 77), (32, 513, 4096, 256), (64, 257, 2048, 257),
              (16, 512, 14336, 501), (40, 1000, 4096, 1000), (24, 100, 128, 128), (48, 9000, 2048, 61),
              (16, 80000, 64, 9), (32, 10000, 2048, 61)]


@pytest.mark.parametrize("kind", ["w2", "w4"])
@pytest.mark.parametrize("M,N,K,n_out", OUT_SHAPES)
def test_outliers_elementwise(lbq, kind, M, N, K, n_out):
    """2-bit: outlier stages of the tensor-core accumulation; 4-bit: outlier
    columns added in the tensor-core kernel's epilogue (both one launch per slab
    or problem)."""
    W, X = _case(M * 5 + N + K + n_out, M, N, K)
    idx = _idx(n_out + K, K, n_out)
    X[:, idx[: max(1, n_out // 3)]] *= 30   # large activations on outlier channels too
    pack, opack = (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)
    ref = O.gemm(opack(W, idx), X)
    y = _run_out(lbq, pack(W, idx), M, N, K, n_out, X, kind=kind)
    assert_close(y, ref, what="mma %s M=%d N=%d K=%d n_out=%d" % (kind, M, N, K, n_out))


@pytest.mark.parametrize("kind", ["w2", "w4"])
def test_outliers_fp16_output_and_repeatable(lbq, kind):
    M, N, K, n_out = 33, 700, 3072, 143
    W, X = _case(77, M, N, K)
    idx = _idx(78, K, n_out)
    pack, opack = (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)
    blob = pack(W, idx)
    ref = O.gemm(opack(W, idx), X)
    assert_close(_run_out(lbq, blob, M, N, K, n_out, X, f32=False, kind=kind), ref, fp16_out=True,
                 what="mma %s outliers f16" % kind)
    a = _run_out(lbq, blob, M, N, K, n_out, X, kind=kind)
    for _ in range(2):
        assert np.array_equal(_run_out(lbq, blob, M, N, K, n_out, X, kind=kind), a)


def test_w2_outliers_launch_count(lbq):
    """Outlier stages add chunks to every tile but no launches."""
    W, X = _case(3, 16, 80000, 64)
    idx = _idx(4, 64, 9)
    big = [(to_dev(lbq.pack_w2cb(W, idx)), 80000, 64, 9, to_dev(X), 64,
            torch.empty((16, 80000), dtype=torch.float32, device="cuda:0"), 80000)]
    assert lbq.gemv_grouped_launches(lbq.LBQ_KIND_W2CB, big, M=16) == 2
