"""GPU parity of EVERY output row, at full size, for the launches the bench
times: the Llama-3-8B layer sweep of seven 4-bit linears (one grouped launch),
the same layer in the 2-bit codebook format with its 3.5 % profile-selected
outlier columns (one grouped launch), the 4-bit gate + down projections at
M = 4 activation rows (one grouped launch) and on the tensor cores at M = 16
and 32, the 2-bit gate with its outlier columns on the tensor cores at M = 16,
and the Llama-3-70B layer (one
grouped launch) and lm_head (one call).  Inputs are the bench's own seeded
synthetic weights and activations (rank 0).  The oracle is computed over row
chunks by worker processes (exact: rows are independent in the blob format).
Covers every row block at every CTA and warp split boundary by construction."""
import numpy as np
import pytest

from bit_weight_only_lbq_gb300 import synth
from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev
import oracle_rows

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def ex():
    with oracle_rows.pool() as e:
        yield e


def _sweep(lbq, ex, kind, linears, wl, M=1, fp16_out=False):
    probs, checks, keep = [], [], []
    for li, (name, N, K) in linears:
        W = synth.weights_heavy_cols(N, K, workload=wl, layer_id=li)
        if M == 1:
            X = synth.activations(1, K, workload=wl, layer_id=li)
        else:
            X = synth.activations(M, K, workload=wl, layer_id=li)
        if kind == "w2":
            idx = O.select_outliers_impact(W, synth.profile_vectors(K, workload=wl, layer_id=li))
            blob = lbq.pack_w2cb(W, idx)
        else:
            idx = np.zeros(0, np.int32)
            blob = lbq.pack_w4(W)
        fut = oracle_rows.submit(ex, kind, W, idx, X)
        del W
        y = torch.full((M, N), float("nan"), dtype=torch.float16 if fp16_out else torch.float32, device="cuda:0")
        b, x = to_dev(blob), to_dev(X)
        keep += [b, x]
        probs.append((b, N, K, len(idx), x, K, y, N))
        checks.append((name, y, fut))
    lk = lbq.LBQ_KIND_W2CB if kind == "w2" else lbq.LBQ_KIND_W4
    assert lbq.gemv_grouped_launches(lk, probs, M=M) == 1
    lbq.gemv_grouped(lk, probs, M=M, pdl=True)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for name, y, fut in checks:
        assert_close(y.float().cpu().numpy(), oracle_rows.collect(fut), fp16_out=fp16_out,
                     what="%s %s every row" % (kind, name))


def test_w4_layer_sweep_every_row(lbq, ex):
    _sweep(lbq, ex, "w4", list(enumerate(synth.LLAMA3_8B_LINEARS)), wl=synth.WL_LLAMA8B_W4)


def test_w2_layer_sweep_every_row(lbq, ex):
    _sweep(lbq, ex, "w2", list(enumerate(synth.LLAMA3_8B_LINEARS)), wl=synth.WL_LLAMA8B_W2)


def test_w4_small_m_gate_down_every_row(lbq, ex):
    _sweep(lbq, ex, "w4", [(li, synth.LLAMA3_8B_LINEARS[li]) for li in (4, 6)], wl=synth.WL_SMALL_M, M=4)


@pytest.mark.parametrize("M", [16, 32])
def test_w4_tensor_core_gate_down_every_row(lbq, ex, M):
    """The 4-bit tensor-core kernel at full size: gate (112 tiles, a CTA each)
    and down (K split over clusters of 4), every row."""
    for li in (4, 6):
        name, N, K = synth.LLAMA3_8B_LINEARS[li]
        W = synth.weights_heavy_cols(N, K, workload=synth.WL_SMALL_M, layer_id=li)
        X = synth.activations(M, K, workload=synth.WL_SMALL_M, layer_id=li)
        fut = oracle_rows.submit(ex, "w4", W, np.zeros(0, np.int32), X)
        blob = lbq.pack_w4(W)
        del W
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda:0")
        b, x = to_dev(blob), to_dev(X)
        lbq.gemm_w4a16_smallM(b, M, N, K, 0, x, K, y, N)
        torch.cuda.synchronize()
        assert lbq.device_error() == 0
        assert_close(y.cpu().numpy(), oracle_rows.collect(fut), what="w4 tensor cores %s M=%d every row" % (name, M))


def test_w2_tensor_core_gate_with_outliers_every_row(lbq, ex):
    """The 2-bit tensor-core kernel at full size with its profile-selected 3.5 %
    outlier columns (gate projection, M = 16: CTA ranges over two tiles, outlier
    stages at every tile's end), every row."""
    M = 16
    li = 4
    name, N, K = synth.LLAMA3_8B_LINEARS[li]
    W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)
    idx = O.select_outliers_impact(W, synth.profile_vectors(K, workload=synth.WL_LLAMA8B_W2, layer_id=li))
    X = synth.activations(M, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)
    fut = oracle_rows.submit(ex, "w2", W, idx, X)
    blob = lbq.pack_w2cb(W, idx)
    del W
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda:0")
    lbq.gemm_w2cb_outlier_smallM(to_dev(blob), M, N, K, len(idx), to_dev(X), K, y, N)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    assert_close(y.cpu().numpy(), oracle_rows.collect(fut), what="w2 tensor cores %s M=%d every row" % (name, M))


def test_70b_layer_every_row(lbq, ex):
    _sweep(lbq, ex, "w4", list(enumerate(synth.LLAMA3_70B_LINEARS)), wl=synth.WL_LLAMA70B, fp16_out=True)


def test_70b_lm_head_every_row(lbq, ex):
    name, N, K = synth.LLAMA3_70B_LM_HEAD
    W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA70B, layer_id=99)
    x = synth.activations(1, K, workload=synth.WL_LLAMA70B, layer_id=K)
    fut = oracle_rows.submit(ex, "w4", W, np.zeros(0, np.int32), x, chunk=4096)
    blob = to_dev(lbq.pack_w4(W))
    del W
    y = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda:0")
    lbq.gemv_w4a16(blob, N, K, 0, to_dev(x[0]), y, pdl=True)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    assert_close(y.cpu().numpy()[None, :], oracle_rows.collect(fut), what="70B lm_head every row")
