"""One continuous-batching decode step over a paged KV cache, in float64.

Test infrastructure only (see the package docstring).

Order of the step (neurogrid releases v0.8.0 / v0.7.0; helexa issue 121,
slice 1):

1. Rotate the new query (all ``Hq`` heads) and the new key (``Hkv`` heads) of
   each row at that row's own position with rotate-half RoPE.  Values are not
   rotated.  The rotated query and key are materialised in the storage type T
   (rounded once from float64); this is our reading of "keys are stored
   post-RoPE" for the key, and the query follows the same boundary.
2. Append: write the rotated key and the raw value of each row into the cache
   slot ``slot_mapping[b]`` (block ``slot // 16``, row ``slot % 16``).
3. Attend: each row attends over its first ``seq_lens[b]`` tokens (the new one
   included, ``kv_len = position + 1``) through its block table, with an
   optional additive bias; the output is rounded to T.
"""
import numpy as np

from .attention import decode_attention_row
from .numerics import round_to
from .rope import rope_rotate_half


def decode_step(q, k_new, v_new, positions, slot_mapping, seq_lens, block_tables,
                k_cache, v_cache, *, scale, base, dtype, attn_bias=None,
                block_size=16, want_probs=False):
    """Run one decode step.

    Arguments are numpy arrays holding the exact values of the dtype-T inputs:
    ``q [B,Hq,d]``, ``k_new, v_new [B,Hkv,d]``, ``positions [B]``,
    ``slot_mapping [B]`` (a negative slot appends nothing), ``seq_lens [B]``
    (lengths after the append), ``block_tables [B, >=max blocks]``,
    ``k_cache, v_cache [num_blocks,Hkv,block_size,d]``, ``attn_bias [B, >=seq_len]``
    or None.  Returns a dict with ``q_rot``, ``k_rot`` (rounded to T),
    ``k_cache``, ``v_cache`` (copies after the append), ``out`` ``[B,Hq,d]``
    (rounded to T) and, if asked, per-row ``probs``.
    """
    q = np.asarray(q, np.float64)
    k_new = np.asarray(k_new, np.float64)
    v_new = np.asarray(v_new, np.float64)
    B, hq, d = q.shape
    q_rot = np.zeros_like(q)
    k_rot = np.zeros_like(k_new)
    for b in range(B):
        q_rot[b] = round_to(rope_rotate_half(q[b], positions[b], base), dtype)
        k_rot[b] = round_to(rope_rotate_half(k_new[b], positions[b], base), dtype)

    k_cache = np.array(k_cache, dtype=np.float64, copy=True)
    v_cache = np.array(v_cache, dtype=np.float64, copy=True)
    for b in range(B):
        slot = int(slot_mapping[b])
        if slot < 0:
            continue
        blk, row = divmod(slot, block_size)
        k_cache[blk, :, row, :] = k_rot[b]
        v_cache[blk, :, row, :] = v_new[b]

    out = np.zeros((B, hq, d))
    probs = []
    for b in range(B):
        bias = None if attn_bias is None else attn_bias[b]
        o, p = decode_attention_row(q_rot[b], k_cache, v_cache, block_tables[b],
                                    int(seq_lens[b]), scale, bias, block_size)
        out[b] = round_to(o, dtype)
        probs.append(p)
    result = dict(q_rot=q_rot, k_rot=k_rot, k_cache=k_cache, v_cache=v_cache,
                  out=out)
    if want_probs:
        result["probs"] = probs
    return result


def prefill_kv(k, v, positions, slot_mapping, k_cache, v_cache, *, base, dtype,
               block_size=16):
    """Write the prefix keys and values of joining sequences into the cache.

    Token t's raw key ``k[t] [Hkv,d]`` is rotated at ``positions[t]`` (the
    same rotate-half RoPE and rounding to T as a decode step's new key: keys are
    stored post-RoPE, helexa issue 121 slice 1) and written with ``v[t]`` to
    slot ``slot_mapping[t]`` (a negative slot writes nothing).  Returns copies of
    ``k_cache, v_cache``.
    """
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    k_cache = np.array(k_cache, dtype=np.float64, copy=True)
    v_cache = np.array(v_cache, dtype=np.float64, copy=True)
    for t in range(k.shape[0]):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        blk, row = divmod(slot, block_size)
        k_cache[blk, :, row, :] = round_to(rope_rotate_half(k[t], positions[t], base), dtype)
        v_cache[blk, :, row, :] = v[t]
    return k_cache, v_cache
