"""GPU parity of the fused kernels against the FP64 oracle, through the C ABI.

Small shapes span several tiles and ragged tails and are compared element by
element; the full-size decode configurations are compared on sampled rows that
the oracle packs and evaluates itself (the bytes are identical; see the
bit-exact packing tests)."""
import numpy as np
import pytest

from bit_weight_only_lbq_gb300 import synth
from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _run(lbq, kind, blob, N, K, n_out, x, f32=True, pdl=False):
    y = torch.empty(N, dtype=torch.float32 if f32 else torch.float16, device="cuda:0")
    f = lbq.gemv_w4a16 if kind == "w4" else lbq.gemv_w2cb_outlier
    f(to_dev(blob), N, K, n_out, to_dev(x), y, pdl=pdl)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    return y.float().cpu().numpy()


SMALL = [(1, 64, 0), (3, 128, 0), (37, 1088, 0), (257, 2112, 5), (130, 4096, 143), (9, 64, 64), (64, 3072, 300)]


@pytest.mark.parametrize("N,K,n_out", SMALL)
@pytest.mark.parametrize("kind", ["w4", "w2"])
def test_small_shapes_elementwise(lbq, kind, N, K, n_out):
    rng = np.random.default_rng(N * 31 + K + n_out)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal(K).astype(np.float16)
    x[rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
    idx = np.sort(rng.choice(K, size=n_out, replace=False)).astype(np.int32)
    pack, opack = (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)
    ref = O.gemv(opack(W, idx), x)
    blob = pack(W, idx)
    assert_close(_run(lbq, kind, blob, N, K, n_out, x), ref, what="%s f32" % kind)
    assert_close(_run(lbq, kind, blob, N, K, n_out, x, f32=False), ref, fp16_out=True, what="%s f16" % kind)


def _sampled_rows(N, rng, n=192):
    rows = np.unique(np.concatenate([[0, 1, 2, 3, N - 4, N - 3, N - 2, N - 1], rng.choice(N, size=min(n, N))]))
    return rows[(rows >= 0) & (rows < N)]


def _layer_weights(wl, N, K, layer):
    if wl == synth.WL_SINGLE_4096:
        return synth.weights_row_scaled(N, K)
    return synth.weights_heavy_cols(N, K, workload=wl, layer_id=layer)


@pytest.mark.parametrize("li", range(len(synth.LLAMA3_8B_LINEARS)))
def test_llama8b_w4_linears_sampled(lbq, li):
    name, N, K = synth.LLAMA3_8B_LINEARS[li]
    W = _layer_weights(synth.WL_LLAMA8B_W4, N, K, li)
    x = synth.activations(1, K, workload=synth.WL_LLAMA8B_W4, layer_id=li)[0]
    rng = np.random.default_rng(li)
    rows = _sampled_rows(N, rng)
    for with_outliers in (False, True):
        idx = O.select_outliers_w4(W) if with_outliers else np.zeros(0, np.int32)
        y = _run(lbq, "w4", lbq.pack_w4(W, idx), N, K, len(idx), x)
        ref = O.gemv(O.pack_w4(W[rows], idx), x)
        assert_close(y[rows], ref, what="llama8b w4 %s outliers=%s" % (name, with_outliers))


@pytest.mark.parametrize("li", range(len(synth.LLAMA3_8B_LINEARS)))
def test_llama8b_w2_linears_sampled(lbq, li):
    name, N, K = synth.LLAMA3_8B_LINEARS[li]
    W = _layer_weights(synth.WL_LLAMA8B_W2, N, K, li)
    x = synth.activations(1, K, workload=synth.WL_LLAMA8B_W2, layer_id=li)[0]
    prof = synth.profile_vectors(K, workload=synth.WL_LLAMA8B_W2, layer_id=li)
    idx = O.select_outliers_impact(W, prof)
    assert len(idx) == int(0.035 * K)
    rows = _sampled_rows(N, np.random.default_rng(100 + li))
    y = _run(lbq, "w2", lbq.pack_w2cb(W, idx), N, K, len(idx), x)
    assert_close(y[rows], O.gemv(O.pack_w2cb(W[rows], idx), x), what="llama8b w2 %s" % name)


def test_single_4096_full_elementwise(lbq):
    W = synth.weights_row_scaled()
    x = synth.activations(1, 4096, workload=synth.WL_SINGLE_4096, layer_id=0)[0]
    blob = lbq.pack_w4(W)
    ref = O.gemv(O.pack_w4(W), x)
    assert_close(_run(lbq, "w4", blob, 4096, 4096, 0, x), ref, what="single 4096 f32")
    assert_close(_run(lbq, "w4", blob, 4096, 4096, 0, x, f32=False), ref, fp16_out=True, what="single 4096 f16")


def test_large_single_problem_elementwise(lbq):
    """One large 4-bit problem (one-record items on 16 warps) with a K of 17
    records per row block and outlier records after the dense ones; every row
    compared."""
    rng = np.random.default_rng(21)
    N, K = 2300, 17408                        # 575 row blocks x 17 records: >= 4 per warp
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal(K).astype(np.float16)
    x[rng.choice(K, size=K // 200, replace=False)] *= 100
    for n_out in (0, 300):
        idx = np.sort(rng.choice(K, size=n_out, replace=False)).astype(np.int32)
        y = _run(lbq, "w4", lbq.pack_w4(W, idx), N, K, n_out, x)
        assert_close(y, O.gemv(O.pack_w4(W, idx), x), what="large single n_out=%d" % n_out)


def test_max_k_and_max_outliers(lbq):
    rng = np.random.default_rng(5)
    for kind in ("w4", "w2"):
        N, K = 9, 65536
        W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
        x = rng.standard_normal(K).astype(np.float16)
        idx = np.sort(rng.choice(K, size=8192, replace=False)).astype(np.int32)
        pack, opack = (lbq.pack_w4, O.pack_w4) if kind == "w4" else (lbq.pack_w2cb, O.pack_w2cb)
        assert_close(_run(lbq, kind, pack(W, idx), N, K, 8192, x), O.gemv(opack(W, idx), x), what=kind + " maxK")


def test_header_mismatch_reported(lbq):
    rng = np.random.default_rng(6)
    W = (rng.standard_normal((8, 128)) * 0.02).astype(np.float32)
    blob = to_dev(lbq.pack_w2cb(W))
    x = to_dev(rng.standard_normal(128).astype(np.float16))
    y = torch.empty(8, dtype=torch.float32, device="cuda:0")
    lbq.gemv_w4a16(blob, 8, 128, 0, x, y)           # a 2-bit blob passed to the 4-bit kernel
    assert lbq.device_error() == 6                  # LBQ_ERR_FORMAT
    assert lbq.device_error() == 0                  # cleared


def test_pdl_back_to_back_and_graph(lbq):
    """Chained GEMVs (y of one is x of the next) with programmatic dependent
    launch, eagerly and captured in a CUDA graph."""
    rng = np.random.default_rng(7)
    K = 2048
    Ws = [(rng.standard_normal((K, K)) * 0.02).astype(np.float32) for _ in range(3)]
    blobs = [to_dev(lbq.pack_w4(W)) for W in Ws]
    x0 = rng.standard_normal(K).astype(np.float16)
    bufs = [to_dev(x0)] + [torch.empty(K, dtype=torch.float16, device="cuda:0") for _ in range(3)]

    def chain():
        for i in range(3):
            lbq.gemv_w4a16(blobs[i], K, K, 0, bufs[i], bufs[i + 1], pdl=True)

    chain()
    torch.cuda.synchronize()
    eager = [b.clone() for b in bufs[1:]]
    # reference: each stage from the GPU's own FP16 input of that stage
    xs = [x0] + [e.cpu().numpy() for e in eager[:-1]]
    for i in range(3):
        assert_close(eager[i].float().cpu().numpy(), O.gemv(O.pack_w4(Ws[i]), xs[i]), fp16_out=True,
                     what="pdl stage %d" % i)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            chain()
    for b in bufs[1:]:
        b.zero_()
    g.replay()
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(bufs[i + 1], eager[i])
    assert lbq.device_error() == 0
