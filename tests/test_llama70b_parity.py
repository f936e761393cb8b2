"""GPU parity at the full Llama-3-70B decode sizes, in the launch configuration
the bench times for them: one layer's seven 4-bit linears (q/o 8192 x 8192,
k/v 1024 x 8192, gate/up 28672 x 8192, down 8192 x 28672) as ONE grouped
launch, and the 128256 x 8192 lm_head as one call, W4A16 Group-32 (SPECTRA
article, sections 3.4 and 4.1).  Sampled output rows (the first, the last and
random ones) are compared with the oracle, which packs exactly those rows
(groups run along K, so a row's codes do not depend on the other rows)."""
import numpy as np
import pytest

from bit_weight_only_lbq_gb300 import synth
from oracle import lbq_oracle as O

from gpu_util import assert_close, to_dev

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _rows(N, seed, n=48):
    r = np.random.default_rng(seed).choice(N, size=n, replace=False)
    return np.unique(np.concatenate([[0, N - 1], r]))


def test_70b_layer_one_grouped_launch_sampled(lbq):
    probs, refs = [], []
    for li, (name, N, K) in enumerate(synth.LLAMA3_70B_LINEARS):
        W = synth.weights_heavy_cols(N, K, config_id=5, layer_id=li)
        x = synth.activations(1, K, config_id=5, layer_id=K)[0]
        rows = _rows(N, li)
        refs.append((name, rows, O.gemv(O.pack_w4(np.ascontiguousarray(W[rows])), x)))
        blob = to_dev(lbq.pack_w4(W))
        del W
        probs.append((blob, N, K, 0, to_dev(x), torch.empty(N, dtype=torch.float16, device="cuda:0")))
    assert lbq.gemv_grouped_launches(lbq.LBQ_KIND_W4, probs) == 1
    lbq.gemv_grouped(lbq.LBQ_KIND_W4, probs, pdl=True)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    for (name, rows, ref), p in zip(refs, probs):
        assert_close(p[5].float().cpu().numpy()[rows], ref, fp16_out=True, what="70B %s" % name)


def test_70b_lm_head_sampled(lbq):
    name, N, K = synth.LLAMA3_70B_LM_HEAD
    W = synth.weights_heavy_cols(N, K, config_id=5, layer_id=99)
    x = synth.activations(1, K, config_id=5, layer_id=K)[0]
    rows = _rows(N, 99, n=96)
    ref = O.gemv(O.pack_w4(np.ascontiguousarray(W[rows])), x)
    blob = to_dev(lbq.pack_w4(W))
    del W
    y = torch.empty(N, dtype=torch.float32, device="cuda:0")
    lbq.gemv_w4a16(blob, N, K, 0, to_dev(x), y, pdl=True)
    torch.cuda.synchronize()
    assert lbq.device_error() == 0
    assert_close(y.cpu().numpy()[rows], ref, what="70B lm_head")
