"""Seeded synthetic inputs for the low-bit decode GEMV workloads.

This module only draws random numbers: weights, activations, profile vectors
and the fixed "spike" channels.  It holds none of the quantisation or GEMV
arithmetic, so both the CPU oracle (through the tests) and the CUDA path can
be fed from it without sharing any of the method's code.

Distributions follow the synthetic workloads of the SPECTRA article (wpnews.pro,
"Compress any LLM 3x ...", section 5.7 "Experiment A": Gaussian 2048x2048
matrices) and the five decode workloads this library is measured on (the
WL_* ids below):

* weights  W ~ N(0, 0.02^2), FP32, N x K row-major (one output per row);
  the single 4096 x 4096 GEMV additionally scales each row's std by U(0.5, 2);
  the others scale floor(0.01 K) randomly chosen input columns by 20;
* activations x ~ N(0, 1) rounded to FP16, with floor(0.005 K) fixed
  "spike" channels multiplied by 100 (the emergent activation spikes the
  otf-llm page, section 4 "Profile-Guided Activation Outliers", describes);
* the otf-llm calibration profile is replaced by 64 seeded vectors drawn
  like x, sharing the same spike channels.

Seeds: numpy PCG64 through ``SeedSequence([workload, layer_id, role_id])``,
except the single 4096 x 4096 GEMV's weight matrix, which uses plain seed 0.
"""
from __future__ import annotations

import numpy as np

# role ids inside a SeedSequence triple
ROLE_WEIGHT = 0
ROLE_X = 1
ROLE_SPIKES = 2
ROLE_HEAVY_COLS = 3
ROLE_PROFILE = 4
ROLE_ROWSCALE = 5

# workload ids (the first word of every seed)
WL_SINGLE_4096 = 1      # one W4A16 GEMV, 4096 x 4096, M = 1
WL_LLAMA8B_W4 = 2       # the seven Llama-3-8B decode linears, 4-bit, M = 1
WL_LLAMA8B_W2 = 3       # the same shapes, 2-bit codebook with 3.5 % FP16 outlier columns
WL_SMALL_M = 4          # batched 4-bit gate and down projections, M = 2..64
WL_LLAMA70B = 5         # the Llama-3-70B full-model decode weight sweep

W_STD = 0.02
SPIKE_FRAC = 0.005
SPIKE_MULT = 100.0
HEAVY_COL_FRAC = 0.01
HEAVY_COL_MULT = 20.0
PROFILE_VECTORS = 64

# (name, N, K): one output per row, K input features
LLAMA3_8B_LINEARS = (
    ("q_proj", 4096, 4096),
    ("k_proj", 1024, 4096),
    ("v_proj", 1024, 4096),
    ("o_proj", 4096, 4096),
    ("gate_proj", 14336, 4096),
    ("up_proj", 14336, 4096),
    ("down_proj", 4096, 14336),
)

LLAMA3_70B_LINEARS = (
    ("q_proj", 8192, 8192),
    ("k_proj", 1024, 8192),
    ("v_proj", 1024, 8192),
    ("o_proj", 8192, 8192),
    ("gate_proj", 28672, 8192),
    ("up_proj", 28672, 8192),
    ("down_proj", 8192, 28672),
)
LLAMA3_70B_LAYERS = 80
LLAMA3_70B_LM_HEAD = ("lm_head", 128256, 8192)

SMALL_M_VALUES = (2, 4, 8, 16, 32, 64)


def rng(workload: int, layer_id: int, role_id: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([workload, layer_id, role_id]))


def gaussian_weights(N: int, K: int, g: np.random.Generator, std: float = W_STD) -> np.ndarray:
    """N x K float32 with i.i.d. N(0, std^2) entries."""
    W = g.standard_normal((N, K), dtype=np.float32)
    W *= np.float32(std)
    return W


def weights_row_scaled(N: int = 4096, K: int = 4096) -> np.ndarray:
    """The single 4096 x 4096 GEMV's matrix: N(0, 0.02^2), seed 0, each row's std
    scaled by U(0.5, 2)."""
    g = np.random.default_rng(0)
    W = gaussian_weights(N, K, g)
    row_scale = rng(WL_SINGLE_4096, 0, ROLE_ROWSCALE).uniform(0.5, 2.0, size=(N, 1)).astype(np.float32)
    W *= row_scale
    return W


def heavy_columns(K: int, workload: int, layer_id: int) -> np.ndarray:
    n = int(HEAVY_COL_FRAC * K)
    cols = rng(workload, layer_id, ROLE_HEAVY_COLS).choice(K, size=n, replace=False)
    return np.sort(cols).astype(np.int64)


def weights_heavy_cols(N: int, K: int, workload: int, layer_id: int) -> np.ndarray:
    """N(0, 0.02^2) with floor(0.01 K) input columns multiplied by 20."""
    W = gaussian_weights(N, K, rng(workload, layer_id, ROLE_WEIGHT))
    W[:, heavy_columns(K, workload, layer_id)] *= np.float32(HEAVY_COL_MULT)
    return W


def spike_channels(K: int, workload: int) -> np.ndarray:
    """floor(0.005 K) fixed activation spike channels for a given width K."""
    n = int(SPIKE_FRAC * K)
    ch = rng(workload, K, ROLE_SPIKES).choice(K, size=n, replace=False)
    return np.sort(ch).astype(np.int64)


def activations(M: int, K: int, workload: int, layer_id: int, stream: int = 0) -> np.ndarray:
    """M x K float16: N(0,1) with the fixed spike channels scaled by 100."""
    g = rng(workload, layer_id, ROLE_X * 1000 + stream)
    X = g.standard_normal((M, K))
    X[:, spike_channels(K, workload)] *= SPIKE_MULT
    return X.astype(np.float16)


def profile_vectors(K: int, workload: int, layer_id: int, P: int = PROFILE_VECTORS) -> np.ndarray:
    """P x K float16 calibration stand-in, drawn like the activations."""
    g = rng(workload, layer_id, ROLE_PROFILE)
    X = g.standard_normal((P, K))
    X[:, spike_channels(K, workload)] *= SPIKE_MULT
    return X.astype(np.float16)


def random_matrix(N: int, K: int, seed: int, scale: float = 1.0) -> np.ndarray:
    """Small generic test matrix, float32."""
    g = np.random.default_rng(seed)
    return (g.standard_normal((N, K)) * scale).astype(np.float32)


def random_vector_f16(K: int, seed: int, M: int | None = None) -> np.ndarray:
    g = np.random.default_rng(seed)
    shape = (K,) if M is None else (M, K)
    return g.standard_normal(shape).astype(np.float16)
