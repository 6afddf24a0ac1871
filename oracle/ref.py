"""Dense brute force of the LoRA delta -- TEST INFRASTRUCTURE.

Used only to pin the paged oracle: it takes the dense weight matrices
straight from the generator (never from pool pages or a page table) and
evaluates y_in + s * (x @ A) @ B with numpy fp64 matmuls, token by token
with each token's own adapter.
"""
from __future__ import annotations

import numpy as np


def dense_delta(x: np.ndarray, A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """(x @ A) @ B in fp64 for x [n, H_in], A [H_in, r], B [r, H_out]."""
    return (x.astype(np.float64) @ A.astype(np.float64)) @ B.astype(np.float64)


def brute_force(token_adapter, x_vals, y_vals, dense_weights, s: float) -> np.ndarray:
    """Exact fp64 y_in + s (x A_a) B_a per token; tokens with id -1 keep y_in.

    dense_weights[a] = (A [H_in, r], B [r, H_out]) as fp64 arrays.
    """
    out = np.array(y_vals, dtype=np.float64, copy=True)
    for i, a in enumerate(np.asarray(token_adapter)):
        if a < 0:
            continue
        A, B = dense_weights[int(a)]
        out[i] = y_vals[i] + s * dense_delta(x_vals[i:i + 1], A, B)[0]
    return out
