"""lbq_refine_noalloc (index scratch in a static device array) against the
two-call form with a caller-provided index buffer: identical bits on two
successive calls with different inputs; argument checks without a GPU."""
import numpy as np
import pytest

from gpu_util import to_dev


def test_noalloc_rejects_bad_shapes_without_gpu(lbq):
    L = lbq.lib()
    assert L.lbq_refine_noalloc(None, 64, 64, 1, 16, 16, 1, None) == 1          # null blob
    assert L.lbq_refine_noalloc(16, 96, 64, 1, 16, 16, 1, None) == 2            # N % 64
    assert L.lbq_refine_noalloc(16, 64, 64, 0, 16, 16, 1, None) == 2            # k < 1
    assert L.lbq_refine_noalloc(16, 64, 64, 257, 16, 16, 1, None) == 2          # k > 256
    assert L.lbq_refine_noalloc(16, 64, 65537, 4, 16, 16, 1, None) == 2         # K > 65536
    assert L.lbq_refine_noalloc(16, 64, 64, 4, 16, 16, 7, None) == 10           # y dtype
    assert L.lbq_refine_noalloc(8, 64, 64, 4, 16, 16, 1, None) == 3             # blob not 16-byte aligned


# (N, K, k, FP32 y): 224 columns (the 32-warp apply), a partial last chunk with
# FP16 y (the 8-warp apply, the last chunk holding min(rest, k) channels), 64
# columns, and the largest selection the static array holds (64 chunks x 256)
NOALLOC_CASES = [(4096, 14336, 16, True), (256, 1500, 8, False), (512, 4096, 16, True), (64, 65536, 256, True)]


@pytest.mark.gpu
@pytest.mark.parametrize("N,K,k,f32", NOALLOC_CASES)
def test_noalloc_matches_two_call_form(lbq, N, K, k, f32):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(77 + K + k)
    R = (rng.standard_normal((N, K)) * 1e-3).astype(np.float32)
    blob = to_dev(lbq.pack_refine(R))
    n_sel = lbq.refine_selected_count(K, k)
    ydt = torch.float32 if f32 else torch.float16
    for call in range(2):                                    # the scratch is reused by the second call
        x = rng.standard_normal(K).astype(np.float16)
        x[rng.choice(K, size=max(1, K // 200), replace=False)] *= 100
        y0 = torch.from_numpy((rng.standard_normal(N) * 0.3).astype(np.float32)).to(ydt)
        d_x = to_dev(x)
        y_ref = y0.clone().cuda()
        idx = torch.empty(n_sel, dtype=torch.int32, device="cuda:0")
        lbq.refine_select(d_x, K, k, idx)
        lbq.refine_apply(blob, N, K, d_x, idx, n_sel, y_ref)
        y_na = y0.clone().cuda()
        lbq.refine_noalloc(blob, N, K, k, d_x, y_na)
        torch.cuda.synchronize()
        assert lbq.device_error() == 0
        assert torch.equal(y_na, y_ref), "call %d" % call
        assert not torch.equal(y_na, y0.cuda())              # the correction did something
