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


def angles_f32(d: int, delta: int, theta: float = 10000.0):
    """cos and sin of a_i = delta * theta^(-2i/d) as float32: the angle is
    formed and reduced modulo 2*pi in float64 (exact reduction), its cos and
    sin taken in float64 and rounded once to float32."""
    i = np.arange(d // 2, dtype=np.float64)
    a = np.fmod(float(delta) * np.power(float(theta), -2.0 * i / d), 2.0 * np.pi)
    return np.cos(a).astype(np.float32), np.sin(a).astype(np.float32)


def realign_fp8(codes: np.ndarray, scale: np.ndarray, delta: int, theta: float = 10000.0) -> np.ndarray:
    """Rotate FP8 (E4M3) key rows codes[..., d] (uint8) with per-channel
    scales scale[d] by `delta` positions and quantise the result again.

    The rotation of the stored values (code * scale) is the formula above,
    evaluated in float32 (the precision the codes are decided in): every
    product and every sum rounded once, no fused multiply-add,

        x = code_i * s_i,  y = code_{i+d/2} * s_{i+d/2}
        x' = (x c_i) - (y s_i'),  y' = (y c_i) + (x s_i')

    (c, s' the float32 cos / sin of angles_f32), and each result is written
    back as a new code: E4M3(v * fp32(1 / scale)) (oracle/fp8.py)."""
    from oracle import fp8
    codes = np.asarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    h = d // 2
    s = np.asarray(scale, dtype=np.float32)
    c, sn = angles_f32(d, delta, theta)
    v = (fp8.decode(codes).astype(np.float32) * s).astype(np.float32)
    x, y = v[..., :h], v[..., h:]
    xn = (x * c).astype(np.float32) - (y * sn).astype(np.float32)
    yn = (y * c).astype(np.float32) + (x * sn).astype(np.float32)
    out = np.concatenate([xn.astype(np.float32), yn.astype(np.float32)], axis=-1)
    return fp8.quantize(out.astype(np.float64), s)
