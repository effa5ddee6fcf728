"""Rounding of float64 values onto the storage grids used by the decode step.

Test infrastructure only (see the package docstring).

The decode step stores its rotated query/key and its output in the storage
type T of the inputs (float32 or bfloat16).  The oracle computes in float64 and
rounds once, to nearest with ties to even, when a value is materialised in T.
"""
import numpy as np

# bfloat16: 8 significant bits (7 stored + implicit), exponent range of float32.
_BF16_SIG_BITS = 8
_BF16_MIN_NORMAL_EXP = -126


def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 value (ties to even).

    Written from the format's definition: a normal bfloat16 value is
    ``1.f * 2**e`` with a 7-bit fraction, so the spacing of representable values
    at exponent ``e`` is ``2**(e - 7)``; below the smallest normal exponent the
    spacing stays at ``2**(-126 - 7)``.  Rounding is a division by the spacing,
    ``rint`` (ties to even) and a multiplication, all exact in float64.
    Values beyond the bfloat16 range are not expected here and are not clamped
    to infinity.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    _, e = np.frexp(x[nz])            # x = m * 2**e with 0.5 <= |m| < 1
    exp_unbiased = np.maximum(e - 1, _BF16_MIN_NORMAL_EXP)
    spacing = np.ldexp(1.0, exp_unbiased - (_BF16_SIG_BITS - 1))
    out[nz] = np.rint(x[nz] / spacing) * spacing
    return out


def round_to_f32(x):
    """Round float64 values to float32 (ties to even) and return float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to(x, dtype):
    """Round onto the grid of ``dtype`` ('f32' or 'bf16')."""
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "f32":
        return round_to_f32(x)
    raise ValueError(f"unknown dtype {dtype!r}")
