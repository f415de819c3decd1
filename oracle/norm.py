"""L2 normalisation of q and k rows, in fp64 (oracle side).

TEST INFRASTRUCTURE ONLY.

The sliding-window paragraph of the talk "Qwen系列模型线性注意力高性能优化实践"
states that every key k_t is L2-normalised before it enters the recurrence
(that is what bounds the factor I - beta k k^T); models of this family normalise
the queries the same way.  The pages give no epsilon; the reading taken here is

    x_hat = x / sqrt(sum_d x_d^2 + eps),   eps = 1e-6,

which is the exact unit vector for any row whose squared norm is far above
eps and maps a zero row to zero.  Computed row by row in fp64 from the values
the device sees.

Its backward (the chain rule through x_hat = x / n, n = sqrt(|x|^2 + eps)):
the Jacobian is I / n - x x^T / n^3, so for an upstream gradient dy

    dx = dy / n - x (x . dy) / n^3.
"""
from __future__ import annotations

import numpy as np

__all__ = ["L2NORM_EPS", "l2_normalize", "l2_normalize_backward"]

L2NORM_EPS = 1e-6


def l2_normalize(x, eps: float = L2NORM_EPS) -> np.ndarray:
    """Rows over the last axis scaled to unit L2 norm (fp64)."""
    a = np.asarray(x, dtype=np.float64)
    ss = np.sum(a * a, axis=-1, keepdims=True)   # squared norm of each row
    return a / np.sqrt(ss + eps)


def l2_normalize_backward(x, dy, eps: float = L2NORM_EPS) -> np.ndarray:
    """Gradient with respect to the rows x of <l2_normalize(x), dy> (fp64)."""
    a = np.asarray(x, dtype=np.float64)
    g = np.asarray(dy, dtype=np.float64)
    n = np.sqrt(np.sum(a * a, axis=-1, keepdims=True) + eps)
    xdy = np.sum(a * g, axis=-1, keepdims=True)
    return g / n - a * xdy / n ** 3
