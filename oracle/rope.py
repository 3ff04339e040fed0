"""RoPE realignment of reused keys -- the plain definition.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

The news summary's Elastic Sparsity recovery starts with "RoPE position
alignment": KV computed for a segment at one position is reused at another,
so the rotation the keys carry must move with them.  The pages give no
formula; this oracle takes the standard rotary embedding (frequencies
theta^(-2i/d), i < d/2) with the "rotate half" pairing of element i with
element i + d/2, which is the reading the library documents.  Moving a key by
delta positions is then the plane rotation by a_i = delta * theta^(-2i/d) of
every pair:

    k'[i]       = k[i] cos a_i - k[i + d/2] sin a_i
    k'[i + d/2] = k[i + d/2] cos a_i + k[i] sin a_i

computed here in float64.  Pins (tests/test_rope_oracle.py) check it against
an independent complex-exponential statement of absolute RoPE, composition,
inverse, norms and hand-derived special angles.
"""
from __future__ import annotations

import numpy as np


def angles(d: int, delta: int, theta: float = 10000.0) -> np.ndarray:
    """a_i = delta * theta^(-2i/d) for i < d/2, float64."""
    i = np.arange(d // 2, dtype=np.float64)
    return float(delta) * np.power(float(theta), -2.0 * i / d)


def realign(k: np.ndarray, delta: int, theta: float = 10000.0) -> np.ndarray:
    """Rotate key rows k[..., d] by `delta` positions (float64 result)."""
    k = np.asarray(k, dtype=np.float64)
    d = k.shape[-1]
    a = angles(d, delta, theta)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = k[..., : d // 2], k[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
