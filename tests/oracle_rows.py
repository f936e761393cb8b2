"""Every-row oracle references for the full-size parity tests.

Rows of a weight matrix are independent under the blob format (groups run along
K), so the oracle's product over a matrix is exactly the concatenation of its
products over row chunks: O.pack_*(W[r0:r1]) followed by O.gemm.  The chunks are
computed by a pool of worker processes started with `spawn` (the test process
already holds a CUDA context), each running the plain FP64 oracle unchanged."""
import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def _chunk_ref(kind, W, idx, X):
    from oracle import lbq_oracle as O
    blob = O.pack_w4(W, idx) if kind == "w4" else O.pack_w2cb(W, idx)
    return np.asarray(O.gemm(blob, X), dtype=np.float64)


def pool(workers=None):
    n = workers or max(1, min(16, os.cpu_count() or 1))
    return ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))


def submit(ex, kind, W, idx, X, chunk=2048):
    """Queue the oracle product of the whole matrix (M x N, FP64) in row chunks."""
    X = np.atleast_2d(X)
    idx = np.asarray(idx, np.int32)
    return [ex.submit(_chunk_ref, kind, np.ascontiguousarray(W[r0:r0 + chunk]), idx, X)
            for r0 in range(0, W.shape[0], chunk)]


def collect(futs):
    return np.concatenate([f.result() for f in futs], axis=1)
