"""GPU parity of the 4-bit Group-32 KV cache (SPECTRA article, section 4.5)
against the oracle, bit for bit: records written by quantise-on-write (one
token at a time and in blocks, at any position, from strided rows), and the
FP16 rows read back; plus argument checks on CPU."""
import numpy as np
import pytest

from oracle import lbq_oracle as O

from gpu_util import to_dev


def test_kv_argument_checks_without_gpu(lbq):
    L = lbq.lib()
    assert L.lbq_kv_record_bytes(1024) == O.kv_record_bytes(1024) == 592
    assert L.lbq_kv_record_bytes(64) == 48 and L.lbq_kv_record_bytes(96) == 0
    assert L.lbq_kv_quantize(16, 64, 1, 96, 16, 0, None) == 2          # width % 64
    assert L.lbq_kv_quantize(16, 32, 1, 64, 16, 0, None) == 2          # ldx < width
    assert L.lbq_kv_quantize(None, 64, 1, 64, 16, 0, None) == 1
    assert L.lbq_kv_quantize(16, 64, 0, 64, 16, 0, None) == 0          # nothing to write
    assert L.lbq_kv_dequant(16, 0, 1, 64, 16, 60, None) == 2           # ldo < width


def _states(rng, rows, width):
    X = (rng.standard_normal((rows, width)) * 2).astype(np.float16)
    X[:, rng.choice(width, size=max(1, width // 100), replace=False)] *= 50     # outlier channels
    X[0, :32] = np.float16(0.0)                                                   # a zero group
    if rows > 2:
        X[2, 32:64] = np.float16(-1.25)                                           # a constant group
    if rows > 3:
        # ties of w / s + z on .5 (s = 1 exactly): round half to even decides the codes
        X[1, :32] = np.float16(0.0)
        X[1, :6] = np.array([0.0, 15.0, 7.5, 2.5, 0.5, 13.5], np.float16)
        # z itself on a tie: wmin = -7.5, s = 1, z = round(7.5) = 8
        X[3, :32] = np.float16(1.0)
        X[3, :4] = np.array([-7.5, 7.5, -2.5, 0.0], np.float16)
        # FP16 subnormals and a negative zero
        X[1, 32:64] = (np.arange(32) * 2.0 ** -24).astype(np.float16)
        X[1, 40] = np.float16(-0.0)
    return X


@pytest.mark.gpu
@pytest.mark.parametrize("width", [64, 1024, 4160])
def test_quantize_on_write_bitexact(lbq, width):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(width)
    T, rb = 37, lbq.kv_record_bytes(width)
    X = _states(rng, T, width)
    cache = torch.full((T + 5, rb), 0xAB, dtype=torch.uint8, device="cuda:0")
    # rows 0..9 one token at a time (decode appends), then the rest as a block
    # from a strided view (prefill), written at an offset of 5 records
    for t in range(10):
        lbq.kv_quantize(to_dev(X[t:t + 1]), 1, width, cache, 5 + t)
    Xs = np.zeros((T - 10, width + 24), np.float16)
    Xs[:, :width] = X[10:]
    lbq.kv_quantize(to_dev(Xs), T - 10, width, cache, 15, ldx=width + 24)
    torch.cuda.synchronize()
    got = cache.cpu().numpy()
    assert np.array_equal(got[5:], O.kv_quantize(X))
    assert (got[:5] == 0xAB).all()                                     # records outside the range untouched
    out = torch.full((T, width + 8), float("nan"), dtype=torch.float16, device="cuda:0")
    lbq.kv_dequant(cache, 5, T, width, out, ldo=width + 8)
    torch.cuda.synchronize()
    back = out.cpu().numpy()
    ref = O.kv_dequant(O.kv_quantize(X), width)
    assert np.array_equal(back[:, :width].view(np.uint16), ref.view(np.uint16))
    assert np.isnan(back[:, width:].astype(np.float32)).all()
