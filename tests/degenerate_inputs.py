"""Weight matrices built from degenerate Group-32 groups, for the packer and
kernel parity tests.  Inputs only: no quantisation or GEMV arithmetic here."""
import numpy as np

G = 32


def mixed_groups(seed: int = 11) -> list:
    """Groups of 32 that each hit one corner of the quantisers, at ordinary
    weight magnitudes."""
    r = np.random.default_rng(seed)
    ramp = np.arange(G, dtype=np.float64)
    return [
        np.zeros(G),                                         # all zero: scale floor, q = z
        np.full(G, 0.3),                                     # constant positive
        np.full(G, -0.7),                                    # constant negative
        np.linspace(1.0, 4.0, G),                            # one-sided: z clamps to 0
        np.linspace(-4.0, -1.0, G),                          # one-sided: z clamps to 15
        np.concatenate([[0.0, 15.0], (ramp[:30] % 15) + 0.5]),   # s = 1: every other value a tie
        np.where(ramp == 17, 0.5, 0.0),                      # a lone spike
        np.where(ramp % 2 == 0, 0.1, -0.1),                  # two values: the outer centroids
        r.standard_normal(G) * 0.02,
    ]


def tiny_groups(seed: int = 12) -> list:
    """Groups whose scales fall below the FP16 normal range (or to zero)."""
    r = np.random.default_rng(seed)
    return [
        r.standard_normal(G) * 1e-7,
        r.standard_normal(G) * 1e-4,
        np.full(G, 1e-30),
        np.linspace(0.0, 3e-6, G),
    ]


def large_groups(seed: int = 13) -> list:
    """Groups of large magnitude whose dequantised values stay inside FP16."""
    r = np.random.default_rng(seed)
    return [
        r.uniform(-3.0e4, 3.0e4, G),
        np.linspace(0.0, 3.0e4, G),
        np.full(G, -2.0e4),
    ]


def degenerate_matrix(N: int, K: int, family: str = "mixed") -> np.ndarray:
    """N x K FP32 (K a multiple of 32): row i cycles the family's groups along K
    starting from group i, reversed on every other pass, negated on odd rows."""
    groups = {"mixed": mixed_groups, "tiny": tiny_groups, "large": large_groups}[family]()
    ng, L = K // G, len(groups)
    rows = []
    for i in range(N):
        parts = []
        for g in range(ng):
            v = groups[(g + i) % L]
            parts.append(v[::-1] if (g // L) % 2 else v)
        row = np.concatenate(parts)
        rows.append(-row if i % 2 else row)
    return np.stack(rows).astype(np.float32)
