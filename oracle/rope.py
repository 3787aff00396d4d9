"""Rotary position embedding (RoPE) of query and key rows, alone and fused
with a row gather.  Test infrastructure only.

Source: guijiagi.com tag page "Ring Attention", article on the evolution of
long-context techniques, section 1.2 "RoPE: rotary position embedding":
* RoPE(x, m) = x e^{i m theta}: the vector at position m is rotated in the
  complex plane, with theta_i = 10000^(-2i/d);
* Re<RoPE(q, m), RoPE(k, n)> depends on m - n only;
* the real form used with it: x * cos + rotate_half(x) * sin, where
  rotate_half cuts the head dimension into halves (x1, x2) and returns
  (-x2, x1), and cos and sin have one row per position and d columns.

Readings where the page is silent (also listed in the design notes):
* i runs over 0 .. d/2 - 1, so theta_0 = 1;
* the base 10000 is a parameter (the page names other bases in its
  extrapolation table, e.g. NTK-aware scaling changes it);
* column j of cos / sin holds cos / sin(m * theta_{j mod d/2}).  With
  rotate_half this is the only layout under which the real form is the
  complex rotation of the first formula: component j (j < d/2) is the real
  part and component j + d/2 the imaginary part of the j-th complex number;
* the rotation covers the whole head dimension (d even);
* the position of a row is given explicitly (one integer per token), as the
  row's index inside its own sequence.

Parity status: pinned (complex-rotation form, relative-position identity,
hand-worked values, identity at position 0, norm preservation).
"""

from __future__ import annotations

import numpy as np


def rope_theta(d: int, base: float = 10000.0):
    """theta_i = base^(-2i/d), i = 0 .. d/2 - 1 (float64)."""
    if d < 2 or d % 2:
        raise ValueError("head dim must be even")
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(np.float64(base), -2.0 * i / d)


def rope_cos_sin(positions, d: int, base: float = 10000.0):
    """cos, sin tables of shape [len(positions), d]: column j uses theta_{j mod d/2}."""
    m = np.asarray(positions, dtype=np.float64)
    ang = m[:, None] * rope_theta(d, base)[None, :]
    ang = np.concatenate([ang, ang], axis=1)
    return np.cos(ang), np.sin(ang)


def rotate_half(x):
    """(x1, x2) -> (-x2, x1) over the last axis."""
    x = np.asarray(x)
    h = x.shape[-1] // 2
    return np.concatenate([-x[..., h:], x[..., :h]], axis=-1)


def apply_rope(x, positions, base: float = 10000.0):
    """x: [n, H, d] rows of one tensor (Q or K); positions: [n] -> rotated rows (float64)."""
    x = np.asarray(x, dtype=np.float64)
    n, _, d = x.shape
    if len(positions) != n:
        raise ValueError("one position per row")
    cos, sin = rope_cos_sin(positions, d, base)
    return x * cos[:, None, :] + rotate_half(x) * sin[:, None, :]


def rope_gather(x, perm, positions, base: float = 10000.0):
    """Row gather fused with the rotation: out[i] = RoPE(x[perm[i]], positions[perm[i]]),
    or a zero row where perm[i] < 0 (a padding slot of the zigzag layout).

    positions holds one position per SOURCE row, so a row keeps the position it
    had before the partition moved it."""
    x = np.asarray(x, dtype=np.float64)
    perm = np.asarray(perm, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    out = np.zeros((len(perm),) + x.shape[1:], dtype=np.float64)
    ok = perm >= 0
    src = perm[ok]
    out[ok] = apply_rope(x[src], positions[src], base)
    return out
