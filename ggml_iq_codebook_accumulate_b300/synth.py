"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the benchmark.

This module holds none of the method's arithmetic: it only draws numbers (numpy's PCG64 generator
with fixed seeds) and rounds them to the storage dtype.  The pages measure on real checkpoints and
calibration sets that are not available here; these draws stand in for them with the shapes and
value distributions the workloads name:

* weights: Student-t with 4 degrees of freedom scaled by 0.02 (or N(0, 0.02) for the small case);
* activations: N(0, 1) times a per-column log-normal(0, 1) scale;
* router: a random permutation of the experts, Zipf(1.2) weights over the first ranks and weight 0
  for the idle tail, top-k distinct experts per token drawn without replacement;
* codebooks: distinct 8-vectors drawn without replacement from the 3^8 combinations of the format's
  value set ({8, 25, 43} for IQ2, {-1, 0, 1} for IQ1), in draw order.
"""
from __future__ import annotations

import numpy as np

FORMATS = ("IQ2_XXS", "IQ2_XS", "IQ2_S", "IQ1_S", "IQ1_M")
GRID_ENTRIES = {"IQ2_XXS": 256, "IQ2_XS": 512, "IQ2_S": 1024, "IQ1_S": 2048, "IQ1_M": 2048}
IQ2_VALUES = (8.0, 25.0, 43.0)
IQ1_VALUES = (-1.0, 0.0, 1.0)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round fp32 to the nearest bf16 (ties to even); returns the bf16 bit patterns (uint16)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_dtype(x: np.ndarray, dtype: str):
    """Returns (storage array, exact fp32 values).  dtype 'f32' or 'bf16' (storage = uint16 bits)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x, x
    if dtype == "bf16":
        h = bf16_round(x)
        return h, bf16_to_f32(h)
    raise ValueError(dtype)


def grid(fmt: str, seed: int | None = None, values=None) -> np.ndarray:
    """Synthetic codebook [entries, 8] fp32 for ``fmt`` (seed defaults to 1000 + format index):
    distinct 8-vectors over ``values`` (default: the format's value set), drawn without
    replacement."""
    n = GRID_ENTRIES[fmt]
    if seed is None:
        seed = 1000 + FORMATS.index(fmt)
    if values is None:
        values = IQ1_VALUES if fmt.startswith("IQ1") else IQ2_VALUES
    vals = np.array(values, np.float32)
    m = len(vals)
    rng = np.random.default_rng(seed)
    codes = rng.choice(m ** 8, size=n, replace=False)
    digits = np.stack([(codes // m ** i) % m for i in range(8)], axis=1)
    return vals[digits].astype(np.float32)


def weight_normal(rows: int, cols: int, seed: int, std: float = 0.02) -> np.ndarray:
    return (np.random.default_rng(seed).standard_normal((rows, cols)) * std).astype(np.float32)


def weight_t4(rows: int, cols: int, seed: int, scale: float = 0.02) -> np.ndarray:
    return (np.random.default_rng(seed).standard_t(4, size=(rows, cols)) * scale).astype(np.float32)


def activations(tokens: int, cols: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    s = np.exp(rng.standard_normal(cols))
    return (rng.standard_normal((tokens, cols)) * s[None, :]).astype(np.float32)


def router(tokens: int, num_experts: int = 128, top_k: int = 8, alpha: float = 1.2, idle: int = 8,
           seed: int = 2) -> np.ndarray:
    """Top-k expert ids [tokens, top_k] int32: a random permutation of the experts ranks them; rank
    r (1-based) has weight r^-alpha for r <= E - idle and 0 after; each token draws top_k distinct
    experts without replacement (Gumbel top-k, which samples exactly that law)."""
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_experts)
    ranks = np.arange(1, num_experts + 1, dtype=np.float64)
    w = np.where(ranks <= num_experts - idle, ranks ** (-alpha), 0.0)
    logp = np.full(num_experts, -np.inf)
    logp[perm] = np.log(np.where(w > 0, w, 1.0)) + np.where(w > 0, 0.0, -np.inf)
    g = rng.gumbel(size=(tokens, num_experts))
    key = logp[None, :] + g
    ids = np.argsort(-key, axis=1, kind="stable")[:, :top_k]
    return ids.astype(np.int32)
