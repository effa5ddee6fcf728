"""The dense right-padded batch (test infrastructure only; see the package
docstring).

helexa issue 121, slice 1: ``assemble_batch`` right-pads every sequence's KV
snapshot to the batch maximum and concatenates the rows; the padding gap of
row b is the columns ``[len_b, padded_len)``, masked with ``-inf``, and the
lockstep decode columns follow at ``padded_len, padded_len + 1, ...``.
Slice 3a: ``extract_row`` slices a row back to a contiguous snapshot, keeping
the prefix ``[0, prefix_len)`` plus the decode columns ``[padded_len,
padded_len + steps)`` and dropping the gap.  Arrays here are token-major:
a snapshot is ``[tokens, Hkv, d]``, a dense batch ``[B, cap, Hkv, d]``.  The gap
holds zeros (any finite value is inert under the mask).
"""
import numpy as np


def assemble_batch(snapshots, padded_len, cap):
    """Dense batch ``[B, cap, Hkv, d]`` of the snapshots, right-padded with zeros
    to ``padded_len``; columns from ``padded_len`` on are left at zero too."""
    hkv, d = snapshots[0].shape[1:]
    dense = np.zeros((len(snapshots), cap, hkv, d))
    for b, s in enumerate(snapshots):
        dense[b, :s.shape[0]] = s
    return dense


def extract_row(dense, row, prefix_len, padded_len, steps):
    """Contiguous snapshot ``[prefix_len + steps, Hkv, d]`` of one row."""
    return np.concatenate([dense[row, :prefix_len],
                           dense[row, padded_len:padded_len + steps]], axis=0)


def gap_bias(lens, padded_len, cap):
    """Additive mask of the dense batch: ``-inf`` on each row's gap."""
    t = np.arange(cap)[None, :]
    lens = np.asarray(lens)[:, None]
    return np.where((t >= lens) & (t < padded_len), -np.inf, 0.0)
