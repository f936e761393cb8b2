"""GPU parity on degenerate weight groups (zero, constant, one-sided, exact
rounding ties, a lone spike, two-valued, sub-FP16-normal and large groups)
through every product entry point: the M = 1 GEMVs and the small-M GEMMs, on
the CUDA cores (M < 16) and on the tensor cores (M >= 16), with outlier
columns placed inside degenerate groups.  N is ragged against the 4-row block
and K holds a full 1024-k record and a partial one.

On the tensor cores each dequantised weight is rounded once to FP16 before the
FP32-accumulating product (the dequantised FP16 tile of the SPECTRA article,
section 4.2 "Batched Tensor Core W4A16 GEMM").  Below the FP16 normal range
(2^-14) that rounding is absolute, at most 2^-25 a weight, which the relative
tolerance does not cover when every weight is that small: for the sub-normal
family on the tensor cores the bound adds sum_k |x_k| |fp16(w_k) - w_k| to each
output's tolerance (w the oracle's dequantised weight)."""
import numpy as np
import pytest

from oracle import lbq_oracle as O

from degenerate_inputs import degenerate_matrix
from gpu_util import assert_close, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N, K = 42, 1408
IDX = np.array([0, 40, 200, 233, 383, 1024, 1407], np.int32)
FAMILIES = ["mixed", "tiny", "large"]


def _inputs(family, M, seed):
    W = degenerate_matrix(N, K, family)
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((M, K)).astype(np.float16)
    X[:, [5, 700]] *= 100                                   # spike channels
    return W, X


def _packers(lbq, kind):
    return (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("kind", ["w4", "w2"])
def test_degenerate_gemv(lbq, kind, family):
    W, X = _inputs(family, 1, 1)
    pack, opack = _packers(lbq, kind)
    y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda:0")
    f = lbq.gemv_w4a16 if kind == "w4" else lbq.gemv_w2cb_outlier
    f(to_dev(pack(W, IDX)), N, K, len(IDX), to_dev(X[0]), y)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    assert_close(y.cpu().numpy(), O.gemv(opack(W, IDX), X[0]), what="%s %s M=1" % (kind, family))


@pytest.mark.parametrize("family", FAMILIES)
@pytest.mark.parametrize("kind", ["w4", "w2"])
@pytest.mark.parametrize("M", [4, 9, 16, 33])
def test_degenerate_gemm(lbq, kind, family, M):
    W, X = _inputs(family, M, M)
    pack, opack = _packers(lbq, kind)
    oblob = opack(W, IDX)
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda:0")
    f = lbq.gemm_w4a16_smallM if kind == "w4" else lbq.gemm_w2cb_outlier_smallM
    f(to_dev(pack(W, IDX)), M, N, K, len(IDX), to_dev(X), K, Y, N)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    Y = Y.cpu().numpy().astype(np.float64)
    ref = O.gemm(oblob, X)
    what = "%s %s M=%d" % (kind, family, M)
    if M >= 16 and family == "tiny":
        Wd = O.dequant(oblob)
        Wd[:, O.outliers(oblob)[0]] = 0.0                   # the dense part skips the outlier columns
        r16 = np.abs(O.fp16_round(Wd).astype(np.float64) - Wd)
        slack = np.abs(X.astype(np.float64)) @ r16.T
        rms = float(np.sqrt(np.mean(ref * ref)))
        bound = 2e-3 * rms + 1e-3 * np.abs(ref) + slack
        err = np.abs(Y - ref)
        assert np.all(np.isfinite(Y)) and np.all(err <= bound), (
            what, float(np.max(err - bound)), float(np.max(slack)), rms)
    else:
        assert_close(Y, ref, what=what)
