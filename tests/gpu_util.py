"""Helpers shared by the GPU tests: device placement and oracle comparison."""
import numpy as np

from oracle import lbq_oracle as O


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda:0")


def assert_close(y_gpu, y_ref, fp16_out=False, what=""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    ok = O.within_tolerance(y_gpu, y_ref, fp16_out=fp16_out)
    if not ok.all():
        bad = np.flatnonzero(~ok.reshape(-1))[:5]
        yr = np.asarray(y_ref).reshape(-1)
        yg = y_gpu.reshape(-1)
        raise AssertionError("%s: %d/%d outside tolerance; first %s: gpu %s ref %s" % (
            what, int((~ok).sum()), ok.size, bad.tolist(), yg[bad].tolist(), yr[bad].tolist()))
    # report headroom: max |err| / bound
    return float(np.max(np.abs(y_gpu - y_ref)))
