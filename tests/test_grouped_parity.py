"""GPU parity of grouped launches (several independent problems in one kernel)
against the FP64 oracle, through the C ABI: ragged mixed shapes element by
element, small M, and a group too wide for one launch (split into back-to-back
launches).  The full-size layer sweeps are checked on every row in
test_fullsize_parity.py."""
import numpy as np
import pytest

from bit_weight_only_lbq_gb300 import synth
from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MIXED = [(37, 1088, 0), (257, 2112, 5), (1, 64, 0), (130, 4096, 143), (64, 3072, 300), (4, 64, 64), (1029, 1024, 0)]


def _problem(rng, N, K, n_out, M=1):
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    X = rng.standard_normal((M, K)).astype(np.float16)
    X[:, rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
    idx = np.sort(rng.choice(K, size=n_out, replace=False)).astype(np.int32)
    return W, X, idx


def _sampled_rows(N, rng, n=160):
    rows = np.unique(np.concatenate([[0, 1, 2, 3, N - 4, N - 3, N - 2, N - 1], rng.choice(N, size=min(n, N))]))
    return rows[(rows >= 0) & (rows < N)]


@pytest.mark.parametrize("kind", ["w4", "w2"])
@pytest.mark.parametrize("f32", [True, False])
def test_mixed_group_elementwise(lbq, kind, f32):
    rng = np.random.default_rng(11 if kind == "w4" else 12)
    pack, opack = (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)
    probs, refs, ys, keep = [], [], [], []
    for (N, K, n_out) in MIXED:
        W, X, idx = _problem(rng, N, K, n_out)
        blob, x = to_dev(pack(W, idx)), to_dev(X[0])
        y = torch.full((N,), float("nan"), dtype=torch.float32 if f32 else torch.float16, device="cuda:0")
        probs.append((blob, N, K, n_out, x, y))
        keep += [blob, x]
        ys.append(y)
        refs.append(O.gemv(opack(W, idx), X[0]))
    lbq.gemv_grouped(lbq.LBQ_KIND_W4 if kind == "w4" else lbq.LBQ_KIND_W2CB, probs)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for (N, K, n_out), y, ref in zip(MIXED, ys, refs):
        assert_close(y.float().cpu().numpy(), ref, fp16_out=not f32, what="%s group %dx%d/%d" % (kind, N, K, n_out))


@pytest.mark.parametrize("M", [2, 3, 8, 13])
def test_small_m_group_elementwise(lbq, M):
    rng = np.random.default_rng(40 + M)
    shapes = [(37, 1088, 0), (130, 4096, 143), (64, 3072, 300)]
    probs, checks = [], []
    for (N, K, n_out) in shapes:
        W, X, idx = _problem(rng, N, K, n_out, M)
        ldx, ldy = K + 8, N + 3
        Xp = np.zeros((M, ldx), np.float16)
        Xp[:, :K] = X
        Y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda:0")
        probs.append((to_dev(lbq.pack_w4(W, idx)), N, K, n_out, to_dev(Xp), ldx, Y, ldy))
        checks.append((Y, N, O.gemm(O.pack_w4(W, idx), X)))
    lbq.gemv_grouped(lbq.LBQ_KIND_W4, probs, M=M)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for Y, N, ref in checks:
        Yc = Y.cpu().numpy()
        assert_close(Yc[:, :N], ref, what="smallM group M=%d" % M)
        assert np.isnan(Yc[:, N:]).all()          # padding columns untouched


def test_group_split_when_too_wide(lbq):
    """Two K=65536 problems whose activations cannot share a CTA's shared memory:
    the library splits the group into back-to-back launches."""
    rng = np.random.default_rng(13)
    K = 65536
    probs, checks = [], []
    for N in (808, 812):
        W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        x = rng.standard_normal(K).astype(np.float16)
        idx = np.sort(rng.choice(K, size=300, replace=False)).astype(np.int32)
        y = torch.empty(N, dtype=torch.float32, device="cuda:0")
        probs.append((to_dev(lbq.pack_w4(W, idx)), N, K, len(idx), to_dev(x), y))
        rows = _sampled_rows(N, rng, n=24)
        checks.append((y, rows, O.gemv(O.pack_w4(W[rows], idx), x)))
    assert lbq.gemv_grouped_launches(lbq.LBQ_KIND_W4, probs) == 2
    lbq.gemv_grouped(lbq.LBQ_KIND_W4, probs)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for y, rows, ref in checks:
        assert_close(y.cpu().numpy()[rows], ref, what="split group")


def test_max_group_of_tiny_problems(lbq):
    rng = np.random.default_rng(14)
    probs, checks = [], []
    for p in range(lbq.LBQ_MAX_GROUP):
        N, K = 1 + p % 5, 64 * (1 + p % 3)
        W, X, idx = _problem(rng, N, K, p % 2)
        y = torch.empty(N, dtype=torch.float32, device="cuda:0")
        probs.append((to_dev(lbq.pack_w2cb(W, idx)), N, K, len(idx), to_dev(X[0]), y))
        checks.append((y, O.gemv(O.pack_w2cb(W, idx), X[0])))
    lbq.gemv_grouped(lbq.LBQ_KIND_W2CB, probs)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for y, ref in checks:
        assert_close(y.cpu().numpy(), ref, what="tiny group")
