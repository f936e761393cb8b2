"""GPU parity of selective weight refinement (StrataFlux paper, section 3
"Weight Refinement", Eq. 2, and "Channel selection") against the oracle,
through the C ABI: the selected channels bit for bit (ties, short last chunks,
k above a chunk's length), the applied correction element by element, the
refinement of the Llama-3-8B projections after their 4-bit GEMV on sampled
rows, FP16 outputs, and the device-side error reports."""
import numpy as np
import pytest

from bit_weight_only_lbq_gb300 import synth
from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _select(lbq, x, k):
    K = x.size
    n = lbq.refine_selected_count(K, k)
    idx = torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda:0")
    lbq.refine_select(to_dev(x), K, k, idx)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    return idx[:n].cpu().numpy()


@pytest.mark.parametrize("K,k", [(64, 1), (64, 100), (1024, 8), (1088, 5), (2048, 256), (4096, 16),
                                 (14336, 16), (14400, 33)])
def test_selection_bitexact(lbq, K, k):
    rng = np.random.default_rng(K * 3 + k)
    x = (rng.standard_normal(K) * 2).astype(np.float16)
    x[rng.choice(K, size=K // 4, replace=False)] = np.float16(0.5)     # many ties in |x|
    x[rng.choice(K, size=K // 8, replace=False)] = np.float16(-0.5)
    x[rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
    assert np.array_equal(_select(lbq, x, k), O.select_refine(x, k))


def test_selection_of_non_finite_values(lbq):
    x = (np.random.default_rng(5).standard_normal(3000) * 2).astype(np.float16)
    x[17], x[400] = np.float16(np.inf), np.float16(-np.inf)
    x[900], x[2100] = np.float16(np.nan), np.float16(65504.0)
    for k in (1, 2, 3, 8):
        assert np.array_equal(_select(lbq, x, k), O.select_refine(x, k))


def test_selection_of_zeros_and_signed_zero(lbq):
    x = np.zeros(3000, np.float16)
    x[1500] = np.float16(-0.0)
    x[2999] = np.float16(1e-7)                      # FP16 subnormal
    assert np.array_equal(_select(lbq, x, 3), O.select_refine(x, 3))


@pytest.mark.parametrize("N,K,k", [(64, 64, 1), (128, 1088, 7), (320, 2112, 64), (4096, 4096, 16),
                                   (320, 4096, 100), (256, 14336, 16),    # > 128 columns: 32 warps
                                   (64, 8192, 256)])                      # > 1024 columns: two index blocks
@pytest.mark.parametrize("f32", [True, False])
def test_apply_elementwise(lbq, N, K, k, f32):
    rng = np.random.default_rng(N + K + k)
    R = (rng.standard_normal((N, K)) * 1e-3).astype(np.float32)
    blob = lbq.pack_refine(R)
    x = rng.standard_normal(K).astype(np.float16)
    x[rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
    idx = O.select_refine(x, k)
    y0 = (rng.standard_normal(N) * 0.3).astype(np.float32 if f32 else np.float16)
    y = torch.from_numpy(y0.copy()).cuda()
    lbq.refine_apply(to_dev(blob), N, K, to_dev(x), to_dev(idx), idx.size, y)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    ref = O.refine_apply(blob, x, idx, y0.astype(np.float64))
    assert_close(y.float().cpu().numpy(), ref, fp16_out=not f32, what="refine N=%d K=%d k=%d" % (N, K, k))


@pytest.mark.parametrize("li", [0, 4, 6])                      # q_proj, gate_proj, down_proj
def test_llama8b_gemv_then_refinement(lbq, li):
    """4-bit GEMV, then select + apply on the same stream: y' = W_hat x + sum x_i C[:, i]."""
    name, N, K = synth.LLAMA3_8B_LINEARS[li]
    W = synth.weights_heavy_cols(N, K, workload=synth.WL_LLAMA8B_W4, layer_id=li)
    x = synth.activations(1, K, workload=synth.WL_LLAMA8B_W4, layer_id=li)[0]
    base = lbq.pack_w4(W)
    # the residual from the oracle's own 4-bit packing (identical bytes, pinned on CPU)
    R = (W.astype(np.float64) - O.dequant_eff(O.pack_w4(W))).astype(np.float32)
    ref_blob = lbq.pack_refine(R)
    k = 16
    n_sel = lbq.refine_selected_count(K, k)
    y = torch.empty(N, dtype=torch.float32, device="cuda:0")
    idx = torch.empty(n_sel, dtype=torch.int32, device="cuda:0")
    d_x = to_dev(x)
    lbq.gemv_w4a16(to_dev(base), N, K, 0, d_x, y)
    lbq.refine_select(d_x, K, k, idx)
    lbq.refine_apply(to_dev(ref_blob), N, K, d_x, idx, n_sel, y)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    sel = O.select_refine(x, k)
    assert np.array_equal(idx.cpu().numpy(), sel)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(li).choice(N, size=160)]))
    y_base = O.gemv(O.pack_w4(W[rows]), x)
    # columns are quantised independently: the oracle packs just the selected ones
    C_sel = O.unpack_refine(O.pack_refine(np.ascontiguousarray(R[:, sel])))[rows]
    ref = y_base.copy()
    for j, i in enumerate(sel):
        ref = ref + np.float64(x[i]) * C_sel[:, j]
    assert_close(y.cpu().numpy()[rows], ref, what="refined %s" % name)
    # the refinement moves the output towards the unquantised product
    exact = W[rows].astype(np.float64) @ x.astype(np.float64)
    assert np.linalg.norm(ref - exact) < np.linalg.norm(y_base - exact)


def test_apply_reports_bad_index_and_header(lbq):
    N, K = 64, 128
    R = np.zeros((N, K), np.float32)
    blob = lbq.pack_refine(R)
    x = to_dev(np.ones(K, np.float16))
    y = torch.zeros(N, dtype=torch.float32, device="cuda:0")
    bad_idx = to_dev(np.array([3, K + 5], np.int32))
    lbq.refine_apply(to_dev(blob), N, K, x, bad_idx, 2, y)
    assert lbq.device_error() == 9                                   # LBQ_ERR_VALUE
    lbq.refine_apply(to_dev(blob), N, K - 64, x, to_dev(np.array([1], np.int32)), 1, y)   # K differs from the blob
    assert lbq.device_error() == 6                                   # LBQ_ERR_FORMAT
    assert np.array_equal(y.cpu().numpy(), np.zeros(N, np.float32))    # a zero residual adds nothing

