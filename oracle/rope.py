"""Rotary position embedding, rotate-half convention, in float64.

Test infrastructure only (see the package docstring).

Follows the helexa continuous-batching PR, slice 1 ("rope: batch_cos_sin
gathers cos/sin at arbitrary per-row positions ... rotate-half"): every batch
row carries its own position, cos/sin are taken at that position, and the head
vector is split into a first and a second half that are rotated against each
other.  The pages give no formula for the frequencies; the plainest reading,
stated as ours, is the usual one: pair ``i`` (``0 <= i < d/2``) turns by
``theta_i = position * base**(-2 i / d)``.
"""
import numpy as np


def inverse_frequencies(d, base):
    """``base**(-2 i / d)`` for ``i = 0 .. d/2 - 1`` in float64."""
    i = np.arange(d // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * i / d)


def rope_rotate_half(x, position, base):
    """Rotate head vectors ``x[..., d]`` that all sit at one ``position``.

    For each pair ``(x[i], x[i + d/2])``::

        x'[i]       = x[i]       * cos(theta_i) - x[i + d/2] * sin(theta_i)
        x'[i + d/2] = x[i + d/2] * cos(theta_i) + x[i]       * sin(theta_i)
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    if d % 2:
        raise ValueError("head_dim must be even")
    half = d // 2
    theta = float(position) * inverse_frequencies(d, base)
    c, s = np.cos(theta), np.sin(theta)
    first, second = x[..., :half], x[..., half:]
    out = np.empty_like(x)
    out[..., :half] = first * c - second * s
    out[..., half:] = second * c + first * s
    return out
