"""Exact decode attention of one batch row over a paged KV cache, float64.

Test infrastructure only (see the package docstring).

What is computed (neurogrid releases, v0.7.0 "Paged Attention Kernel: reads
K/V via block_table indirection, GQA support"; v0.6.0 "Flash Decode"):

* The cache is a pool of fixed 16-token blocks laid out
  ``[num_blocks, Hkv, block_size, d]``; token ``t`` of a sequence lives in
  block ``block_table[t // block_size]`` at row ``t % block_size``.
* Grouped-query attention: query head ``h`` reads KV head ``h // G`` with
  ``G = Hq / Hkv`` (contiguous groups; the pages do not state the mapping, this
  is our reading).
* Scores ``s_t = (q . k_t) * scale + bias_t``; probabilities
  ``P = exp(s - max s) / sum``; output ``sum_t P_t v_t``.  This is the plain
  definition; flash decode and the split-KV merge reach the same value by a
  different summation order.
* A row whose scores are all ``-inf`` (or that has no tokens) outputs zeros,
  the zero-denominator guard of the cortex-engine writeup's block-sparse
  attention kernel.
"""
import numpy as np


def gather_sequence(cache, block_table, n_tokens, kv_head, block_size=16):
    """Keys (or values) ``[n_tokens, d]`` of one sequence and one KV head.

    ``cache`` is ``[num_blocks, Hkv, block_size, d]``; ``block_table`` lists the
    sequence's blocks in order.
    """
    t = np.arange(n_tokens)
    blocks = np.asarray(block_table)[t // block_size]
    return np.asarray(cache, dtype=np.float64)[blocks, kv_head, t % block_size]


def softmax_attention(q, keys, values, scale, bias=None):
    """One query vector against ``n`` keys/values.

    Returns ``(out [d], probs [n])``.  ``bias`` (optional, ``[n]``) is added to
    the scaled scores; ``-inf`` entries exclude a token.
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    n = keys.shape[0]
    if n == 0:
        return np.zeros(values.shape[-1]), np.zeros(0)
    s = (keys @ q) * float(scale)
    if bias is not None:
        s = s + np.asarray(bias, dtype=np.float64)
    m = s.max()
    if m == -np.inf:
        return np.zeros(values.shape[-1]), np.zeros(n)
    w = np.exp(s - m)
    probs = w / w.sum()
    return probs @ values, probs


def decode_attention_row(q_rot, k_cache, v_cache, block_table, seq_len, scale,
                         bias=None, block_size=16):
    """Attention output ``[Hq, d]`` and probabilities ``[Hq, seq_len]`` of one row.

    ``q_rot`` is ``[Hq, d]`` (already rotated).  ``seq_len`` counts every token
    the row attends to, the one appended in this step included.
    """
    q_rot = np.asarray(q_rot, dtype=np.float64)
    hq, d = q_rot.shape
    hkv = k_cache.shape[1]
    group = hq // hkv
    out = np.zeros((hq, d))
    probs = np.zeros((hq, seq_len))
    row_bias = None if bias is None else np.asarray(bias, np.float64)[:seq_len]
    for g in range(hkv):
        keys = gather_sequence(k_cache, block_table, seq_len, g, block_size)
        values = gather_sequence(v_cache, block_table, seq_len, g, block_size)
        for h in range(g * group, (g + 1) * group):
            out[h], probs[h] = softmax_attention(q_rot[h], keys, values, scale,
                                                 row_bias)
    return out, probs
