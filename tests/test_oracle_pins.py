"""Pins of the float64 oracle to facts other than itself.

Each test checks the oracle against something the pages or mathematics fix:
a library routine (torch's bfloat16 cast, torch's scaled-dot-product attention,
complex multiplication), a closed form, an invariant the pages state (ragged
lockstep equals sequential, padding under the additive mask is inert, paged
equals contiguous), or a hand-derived allocator trace in ``tests/golden``.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle.allocator import BlockAllocatorModel, OutOfBlocks, UnknownSequence
from oracle.attention import decode_attention_row, gather_sequence, softmax_attention
from oracle.numerics import round_to_bf16, round_to_f32
from oracle.rope import rope_rotate_half
from oracle.step import decode_step, prefill_kv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


# --------------------------------------------------------------------------
# rounding onto the storage grid
# --------------------------------------------------------------------------
def test_bf16_rounding_matches_torch_cast():
    x32 = rng.standard_normal(20000).astype(np.float32) * np.float32(3.0)
    # exact ties: a bfloat16 value plus half of its spacing
    b = torch.from_numpy(x32[:2000]).to(torch.bfloat16).to(torch.float64).numpy()
    spacing = np.ldexp(1.0, np.frexp(b)[1] - 8)
    ties = (b + 0.5 * spacing).astype(np.float32)
    x32 = np.concatenate([x32, ties, np.float32([0.0, -0.0, 1.0, -1.5, 1e-30])])
    expect = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = round_to_bf16(x32.astype(np.float64))
    np.testing.assert_array_equal(got, expect)


def test_f32_rounding_matches_numpy_cast():
    x = rng.standard_normal(1000) * 1e3
    np.testing.assert_array_equal(round_to_f32(x), x.astype(np.float32).astype(np.float64))


# --------------------------------------------------------------------------
# RoPE (helexa issue 121, slice 1: per-row positions, rotate-half)
# --------------------------------------------------------------------------
def test_rope_position_zero_is_identity():
    x = rng.standard_normal((5, 64))
    np.testing.assert_array_equal(rope_rotate_half(x, 0, 10000.0), x)


def test_rope_hand_worked_d4():
    # d = 4, base 10000: theta_0 = p, theta_1 = p * 10000**(-1/2) = p / 100.
    x = np.array([1.0, 2.0, 3.0, 4.0])
    p = 1
    expect = np.array([
        1 * math.cos(1) - 3 * math.sin(1),
        2 * math.cos(0.01) - 4 * math.sin(0.01),
        3 * math.cos(1) + 1 * math.sin(1),
        4 * math.cos(0.01) + 2 * math.sin(0.01),
    ])
    np.testing.assert_allclose(rope_rotate_half(x, p, 10000.0), expect, rtol=0, atol=1e-15)


@pytest.mark.parametrize("d,pos", [(64, 7), (128, 131072), (128, 2047)])
def test_rope_equals_complex_rotation(d, pos):
    """Pair (x[i], x[i+d/2]) as the complex number x[i] + i x[i+d/2] times e^{i theta}."""
    x = rng.standard_normal((3, d))
    half = d // 2
    theta = np.array([pos / (10000.0 ** (2.0 * i / d)) for i in range(half)])
    z = (x[:, :half] + 1j * x[:, half:]) * np.exp(1j * theta)
    expect = np.concatenate([z.real, z.imag], axis=1)
    np.testing.assert_allclose(rope_rotate_half(x, pos, 10000.0), expect,
                               rtol=0, atol=1e-10)


def test_rope_preserves_pair_norms():
    x = rng.standard_normal((4, 128))
    y = rope_rotate_half(x, 12345, 10000.0)
    n_x = x[:, :64] ** 2 + x[:, 64:] ** 2
    n_y = y[:, :64] ** 2 + y[:, 64:] ** 2
    np.testing.assert_allclose(n_y, n_x, rtol=1e-12)


@pytest.mark.parametrize("m,n", [(10, 3), (4096, 4000), (131072, 65536)])
def test_rope_relative_position(m, n):
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    lhs = rope_rotate_half(q, m, 10000.0) @ rope_rotate_half(k, n, 10000.0)
    rhs = rope_rotate_half(q, m - n, 10000.0) @ k
    assert abs(lhs - rhs) < 1e-9


# --------------------------------------------------------------------------
# softmax attention: closed forms
# --------------------------------------------------------------------------
def test_single_token_returns_its_value():
    q, k, v = rng.standard_normal((3, 64))
    out, p = softmax_attention(q, k[None], v[None], 0.125)
    np.testing.assert_array_equal(out, v)
    assert p.tolist() == [1.0]


def test_zero_query_averages_values():
    keys = rng.standard_normal((37, 64))
    values = rng.standard_normal((37, 64))
    out, p = softmax_attention(np.zeros(64), keys, values, 0.125)
    np.testing.assert_allclose(out, values.mean(axis=0), rtol=0, atol=1e-13)
    np.testing.assert_allclose(p, np.full(37, 1 / 37), rtol=1e-13)


def test_constant_values_pass_through():
    keys = rng.standard_normal((100, 128)) * 3
    values = np.full((100, 128), -2.5)
    out, _ = softmax_attention(rng.standard_normal(128), keys, values, 1 / math.sqrt(128))
    np.testing.assert_allclose(out, values[0], rtol=0, atol=1e-13)


def test_two_tokens_logistic_form():
    """P(token 0) = sigmoid((q.k0 - q.k1) * scale): pins the scale and the sign."""
    q, k0, k1, v0, v1 = rng.standard_normal((5, 64))
    scale = 1 / math.sqrt(64)
    out, p = softmax_attention(q, np.stack([k0, k1]), np.stack([v0, v1]), scale)
    a = 1.0 / (1.0 + math.exp(-(q @ k0 - q @ k1) * scale))
    np.testing.assert_allclose(p, [a, 1 - a], rtol=1e-13)
    np.testing.assert_allclose(out, a * v0 + (1 - a) * v1, rtol=0, atol=1e-13)


def test_probabilities_sum_to_one():
    keys = rng.standard_normal((513, 128)) * 4
    _, p = softmax_attention(rng.standard_normal(128) * 4, keys, keys, 1 / math.sqrt(128))
    assert abs(p.sum() - 1.0) < 1e-12 and (p >= 0).all()


def test_fully_masked_row_outputs_zero():
    keys = rng.standard_normal((5, 64))
    out, p = softmax_attention(keys[0], keys, keys, 0.1, bias=np.full(5, -np.inf))
    assert not np.isnan(out).any()
    np.testing.assert_array_equal(out, 0)
    np.testing.assert_array_equal(p, 0)


# --------------------------------------------------------------------------
# paged gather, GQA mapping and the invariants the pages state
# --------------------------------------------------------------------------
def _scatter_pagewise(seqs, table_rows, num_blocks, hkv, d, fill=None):
    """Place contiguous per-sequence K or V ``[Hkv, L, d]`` into a block pool,
    one 16-token page at a time (slice copies, no per-token index arithmetic)."""
    pool = np.zeros((num_blocks, hkv, 16, d)) if fill is None else fill.copy()
    for seq, table in zip(seqs, table_rows):
        L = seq.shape[1]
        for j in range(-(-L // 16)):
            chunk = seq[:, 16 * j:16 * (j + 1)]
            pool[table[j], :, :chunk.shape[1]] = chunk
    return pool


def _random_layout(lens, hkv, d, num_blocks, seed):
    r = np.random.default_rng(seed)
    ks = [r.standard_normal((hkv, L, d)) for L in lens]
    vs = [r.standard_normal((hkv, L, d)) for L in lens]
    perm = r.permutation(num_blocks)
    tables, used = [], 0
    for L in lens:
        n = -(-L // 16)
        tables.append(perm[used:used + n])
        used += n
    return ks, vs, tables


def test_paged_attention_matches_torch_sdpa():
    """Brute force with a library routine: torch's float64 SDPA on a dense,
    right-padded batch with a boolean mask, against the paged per-row oracle."""
    lens, hq, hkv, d = [6, 18, 34], 4, 2, 64
    ks, vs, tables = _random_layout(lens, hkv, d, 16, 7)
    k_pool = _scatter_pagewise(ks, tables, 16, hkv, d)
    v_pool = _scatter_pagewise(vs, tables, 16, hkv, d)
    q = rng.standard_normal((3, hq, d))
    scale = 1 / math.sqrt(d)
    S = max(lens)
    K = torch.zeros(3, hkv, S, d, dtype=torch.float64)
    V = torch.zeros(3, hkv, S, d, dtype=torch.float64)
    mask = torch.zeros(3, 1, 1, S, dtype=torch.bool)
    for b, L in enumerate(lens):
        K[b, :, :L] = torch.from_numpy(ks[b])
        V[b, :, :L] = torch.from_numpy(vs[b])
        mask[b, ..., :L] = True
    G = hq // hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, :, None, :], K.repeat_interleave(G, dim=1),
        V.repeat_interleave(G, dim=1), attn_mask=mask, scale=scale)[:, :, 0, :]
    for b, L in enumerate(lens):
        out, _ = decode_attention_row(q[b], k_pool, v_pool, tables[b], L, scale)
        np.testing.assert_allclose(out, ref[b].numpy(), rtol=0, atol=1e-12)


def test_gather_follows_block_table():
    lens, hkv, d = [40], 2, 8
    ks, _, tables = _random_layout(lens, hkv, d, 9, 3)
    pool = _scatter_pagewise(ks, tables, 9, hkv, d)
    for g in range(hkv):
        np.testing.assert_array_equal(gather_sequence(pool, tables[0], 40, g), ks[0][g])


def test_gqa_head_mapping():
    """Query head h reads KV head h // G: with V of KV head g constant g + 1,
    the output of head h is h // G + 1."""
    hq, hkv, d, L = 8, 2, 16, 20
    ks, _, tables = _random_layout([L], hkv, d, 4, 5)
    vs = [np.stack([np.full((L, d), g + 1.0) for g in range(hkv)])]
    k_pool = _scatter_pagewise(ks, tables, 4, hkv, d)
    v_pool = _scatter_pagewise(vs, tables, 4, hkv, d)
    out, _ = decode_attention_row(rng.standard_normal((hq, d)), k_pool, v_pool,
                                  tables[0], L, 0.25)
    for h in range(hq):
        np.testing.assert_allclose(out[h], h // (hq // hkv) + 1.0, atol=1e-13)


def test_block_table_permutation_invariance():
    """Paged layout under any block permutation equals the contiguous layout."""
    lens, hq, hkv, d = [45, 3, 16], 4, 2, 32
    ks, vs, tables_a = _random_layout(lens, hkv, d, 12, 11)
    contiguous, used = [], 0
    for L in lens:
        n = -(-L // 16)
        contiguous.append(np.arange(used, used + n))
        used += n
    q = rng.standard_normal((3, hq, d))
    pools = []
    for tables in (tables_a, contiguous):
        pools.append((_scatter_pagewise(ks, tables, 12, hkv, d),
                      _scatter_pagewise(vs, tables, 12, hkv, d), tables))
    for b, L in enumerate(lens):
        outs = [decode_attention_row(q[b], kp, vp, t[b], L, 0.2)[0] for kp, vp, t in pools]
        np.testing.assert_allclose(outs[0], outs[1], rtol=0, atol=1e-14)


def test_padded_batch_with_mask_equals_unpadded():
    """helexa issue 121, slice 1: right-pad each row to the batch max and mask the
    gap [prefix_len, padded_len) with an additive -inf bias; the new token goes
    after the gap.  The result equals the unpadded row."""
    prefixes, hq, hkv, d = [5, 17, 33], 4, 2, 64
    padded = max(prefixes)
    r = np.random.default_rng(21)
    q = r.standard_normal((3, hq, d))
    for b, P in enumerate(prefixes):
        k_real = r.standard_normal((hkv, P + 1, d))
        v_real = r.standard_normal((hkv, P + 1, d))
        gap_k = r.standard_normal((hkv, padded - P, d)) * 100     # finite garbage
        gap_v = r.standard_normal((hkv, padded - P, d)) * 100
        k_pad = np.concatenate([k_real[:, :P], gap_k, k_real[:, P:]], axis=1)
        v_pad = np.concatenate([v_real[:, :P], gap_v, v_real[:, P:]], axis=1)
        bias = np.zeros(padded + 1)
        bias[P:padded] = -np.inf
        t_real = np.arange(-(-(P + 1) // 16))
        t_pad = np.arange(-(-(padded + 1) // 16))
        out_real, _ = decode_attention_row(
            q[b], _scatter_pagewise([k_real], [t_real], len(t_real), hkv, d),
            _scatter_pagewise([v_real], [t_real], len(t_real), hkv, d), t_real, P + 1, 0.125)
        out_pad, p_pad = decode_attention_row(
            q[b], _scatter_pagewise([k_pad], [t_pad], len(t_pad), hkv, d),
            _scatter_pagewise([v_pad], [t_pad], len(t_pad), hkv, d), t_pad, padded + 1,
            0.125, bias=bias)
        np.testing.assert_allclose(out_pad, out_real, rtol=0, atol=1e-12)
        assert (p_pad[:, P:padded] == 0).all()


def test_ragged_batch_equals_rows_alone():
    """helexa issue 121: a ragged lockstep batch equals each sequence decoded alone."""
    lens = [6, 18, 34]
    r = np.random.default_rng(4)
    hq, hkv, d, nb = 4, 2, 64, 16
    k_cache = r.standard_normal((nb, hkv, 16, d))
    v_cache = r.standard_normal((nb, hkv, 16, d))
    q = r.standard_normal((3, hq, d))
    knew = r.standard_normal((3, hkv, d))
    vnew = r.standard_normal((3, hkv, d))
    perm = r.permutation(nb)
    tables = np.full((3, 4), -1)
    tables[0, :1] = perm[0:1]
    tables[1, :2] = perm[1:3]
    tables[2, :3] = perm[3:6]
    pos = np.array(lens) - 1
    slots = np.array([tables[b, p // 16] * 16 + p % 16 for b, p in enumerate(pos)])
    kw = dict(scale=0.125, base=10000.0, dtype="f32")
    full = decode_step(q, knew, vnew, pos, slots, lens, tables, k_cache, v_cache, **kw)
    for b in range(3):
        solo = decode_step(q[b:b + 1], knew[b:b + 1], vnew[b:b + 1], pos[b:b + 1],
                           slots[b:b + 1], lens[b:b + 1], tables[b:b + 1], k_cache,
                           v_cache, **kw)
        np.testing.assert_array_equal(solo["out"][0], full["out"][b])


# --------------------------------------------------------------------------
# the step: RoPE on q and k at the row's position, append, attend
# --------------------------------------------------------------------------
def test_step_empty_prefix_returns_new_value():
    """With no cached tokens the row attends only to its own new token."""
    r = np.random.default_rng(8)
    q = r.standard_normal((1, 8, 64))
    knew = r.standard_normal((1, 2, 64))
    vnew = round_to_bf16(r.standard_normal((1, 2, 64)))
    res = decode_step(q, knew, vnew, [0], [16 * 3], [1], np.array([[3]]),
                      np.zeros((4, 2, 16, 64)), np.zeros((4, 2, 16, 64)),
                      scale=0.125, base=10000.0, dtype="bf16")
    for h in range(8):
        np.testing.assert_array_equal(res["out"][0, h], vnew[0, h // 4])


def test_step_append_writes_only_the_slot():
    r = np.random.default_rng(9)
    k_cache = r.standard_normal((6, 2, 16, 32))
    v_cache = r.standard_normal((6, 2, 16, 32))
    q = r.standard_normal((2, 4, 32))
    knew = r.standard_normal((2, 2, 32))
    vnew = r.standard_normal((2, 2, 32))
    res = decode_step(q, knew, vnew, [20, 3], [4 * 16 + 4, 1 * 16 + 3], [21, 4],
                      np.array([[2, 4], [1, -1]]), k_cache, v_cache,
                      scale=0.2, base=10000.0, dtype="f32")
    expect_k = k_cache.copy()
    expect_v = v_cache.copy()
    expect_k[4, :, 4] = round_to_f32(rope_rotate_half(knew[0], 20, 10000.0))
    expect_k[1, :, 3] = round_to_f32(rope_rotate_half(knew[1], 3, 10000.0))
    expect_v[4, :, 4] = vnew[0]
    expect_v[1, :, 3] = vnew[1]
    np.testing.assert_array_equal(res["k_cache"], expect_k)
    np.testing.assert_array_equal(res["v_cache"], expect_v)


def test_step_keys_are_stored_post_rope():
    """Relative-position check through the cache: a key appended at position n and
    read back at step m scores like the unrotated key against R(m - n) q."""
    r = np.random.default_rng(10)
    d = 64
    k0 = r.standard_normal((1, 1, d))
    res0 = decode_step(r.standard_normal((1, 1, d)), k0, r.standard_normal((1, 1, d)),
                       [0], [0], [1], np.array([[0, 1]]), np.zeros((2, 1, 16, d)),
                       np.zeros((2, 1, 16, d)), scale=1.0, base=10000.0, dtype="f32")
    stored = res0["k_cache"][0, 0, 0]
    np.testing.assert_allclose(stored, round_to_f32(k0[0, 0]), atol=0)   # position 0
    q = r.standard_normal(d)
    m = 17
    lhs = round_to_f32(rope_rotate_half(q, m, 10000.0)) @ stored
    rhs = rope_rotate_half(q, m, 10000.0) @ k0[0, 0]
    assert abs(lhs - rhs) < 1e-5


def _complex_rotate(x, pos, base=10000.0):
    """Rotate head vectors ``x[..., d]`` at ``pos`` by complex multiplication:
    pair (x[i], x[i + d/2]) is the number x[i] + i x[i + d/2] times e^{i theta_i}."""
    d = x.shape[-1]
    half = d // 2
    theta = pos / base ** (2.0 * np.arange(half) / d)
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * theta)
    return np.concatenate([z.real, z.imag], axis=-1)


def _torch_round(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(torch.bfloat16 if dtype == "bf16" else torch.float32).double().numpy()


@pytest.mark.parametrize("dtype,L,hq,hkv,d", [("bf16", 37, 8, 2, 64), ("bf16", 300, 32, 8, 128),
                                              ("f32", 21, 4, 2, 64)])
def test_step_rotates_the_query_at_its_position(dtype, L, hq, hkv, d):
    """helexa issue 121, slice 1 (per-row cos/sin at each row's position,
    rotate-half): the step rotates the new query at ``positions[b]`` -- the
    row's cached length, one less than ``seq_lens[b]`` -- rounds it once to the
    storage type and scores the gathered keys with it.  Built without the
    oracle: the rotation by complex multiplication, the rounding by torch's
    cast, the attention by torch's float64 SDPA over a contiguous cache (an
    identity block table).  The mistakes this must catch (the query rotated at
    seq_lens, not rotated, or scored without its rounding) are shown to move
    the output by many units of the storage type's last place."""
    r = np.random.default_rng(1000 + L)
    nblk = -(-(L + 1) // 16)
    # cached keys are post-RoPE values, drawn directly; values on the grid of T
    k_cache = _torch_round(r.standard_normal((nblk, hkv, 16, d)), dtype)
    v_cache = _torch_round(r.standard_normal((nblk, hkv, 16, d)), dtype)
    # a large query makes the softmax sharp, so that the rounding of the
    # rotated query shows in the output
    q = _torch_round(r.standard_normal((1, hq, d)) * 6.0, dtype)
    knew = _torch_round(r.standard_normal((1, hkv, d)), dtype)
    vnew = _torch_round(r.standard_normal((1, hkv, d)), dtype)
    pos, scale = L, 1 / math.sqrt(d)
    res = decode_step(q, knew, vnew, [pos], [pos], [L + 1], np.arange(nblk)[None, :],
                      k_cache, v_cache, scale=scale, base=10000.0, dtype=dtype)

    def reference(q_pos, round_q=True, rotate=True):
        qr = _complex_rotate(q[0], q_pos) if rotate else q[0]
        qr = _torch_round(qr, dtype) if round_q else qr
        kr = _torch_round(_complex_rotate(knew[0], pos), dtype)
        K = k_cache.transpose(1, 0, 2, 3).reshape(hkv, nblk * 16, d).copy()
        V = v_cache.transpose(1, 0, 2, 3).reshape(hkv, nblk * 16, d).copy()
        K[:, pos], V[:, pos] = kr, vnew[0]
        G = hq // hkv
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qr)[:, None, :],
            torch.from_numpy(K[:, :L + 1]).repeat_interleave(G, dim=0),
            torch.from_numpy(V[:, :L + 1]).repeat_interleave(G, dim=0), scale=scale)[:, 0]
        return qr, _torch_round(o.numpy(), dtype)

    q_ref, out_ref = reference(pos)
    np.testing.assert_array_equal(res["q_rot"][0], q_ref)
    ulp = np.maximum(np.abs(out_ref), 2.0 ** -20) * (2.0 ** -7 if dtype == "bf16" else 2.0 ** -23)
    assert (np.abs(res["out"][0] - out_ref) <= ulp).all()
    # each plausible mistake moves the output well past that tolerance
    wrong = [reference(pos + 1)[1], reference(pos, rotate=False)[1]]
    if dtype == "bf16":
        wrong.append(reference(pos, round_q=False)[1])
    for w in wrong:
        assert (np.abs(w - out_ref) > 4 * ulp).any()


# --------------------------------------------------------------------------
# allocator model against the hand-derived trace
# --------------------------------------------------------------------------
def test_allocator_model_golden_trace():
    with open(os.path.join(GOLDEN, "allocator_trace.json")) as f:
        g = json.load(f)
    a = BlockAllocatorModel(g["num_blocks"], g["block_size"], g["max_seqs"],
                            initial_free=g["initial_free"])
    for op in g["ops"]:
        err = op.get("error")
        if op["op"] == "join":
            if err:
                with pytest.raises(OutOfBlocks):
                    a.join(op["prefix"])
            else:
                assert a.join(op["prefix"]) == op["seq_id"]
        elif op["op"] == "leave":
            if err:
                with pytest.raises(UnknownSequence):
                    a.leave(op["seq_id"])
            else:
                a.leave(op["seq_id"])
        elif op["op"] == "step":
            if err:
                before = {s: a.seq_len(s) for s in op["seq_ids"]}
                with pytest.raises(OutOfBlocks):
                    a.prepare_step(op["seq_ids"], g["bt_stride"])
                assert {s: a.seq_len(s) for s in op["seq_ids"]} == before
            else:
                pos, slots, lens, tables = a.prepare_step(op["seq_ids"], g["bt_stride"])
                assert pos.tolist() == op["positions"]
                assert slots.tolist() == op["slots"]
                assert lens.tolist() == op["seq_lens"]
                assert tables.tolist() == op["tables"]
        assert a.free == op["free_after"], op
    for sid, blocks in g["final_tables"].items():
        assert a.seq_blocks(int(sid)) == blocks
        assert a.seq_len(int(sid)) == g["final_lengths"][sid]


def test_allocator_model_conservation_under_churn():
    r = np.random.default_rng(99)
    nb = 300
    a = BlockAllocatorModel(nb, max_seqs=32, initial_free=r.permutation(nb))
    live = []
    for it in range(400):
        act = r.integers(0, 3)
        try:
            if act == 0 and len(live) < 32:
                live.append(a.join(int(r.integers(0, 100))))
            elif act == 1 and live:
                a.leave(live.pop(int(r.integers(0, len(live)))))
            elif live:
                a.prepare_step(live, 64)
        except OutOfBlocks:
            pass
        owned = [blk for s in live for blk in a.seq_blocks(s)]
        assert len(owned) == len(set(owned))
        assert sorted(owned + a.free) == list(range(nb))
        for s in live:
            assert len(a.seq_blocks(s)) == -(-a.seq_len(s) // 16)


def test_allocator_model_prefix_slots_hand_derived():
    """join(20) on the free stack [5,3,0,1,4,2] (bottom to top) pops 2 then 4, so
    tokens 14..17 live in block 2 rows 14, 15 and block 4 rows 0, 1."""
    a = BlockAllocatorModel(6, initial_free=[5, 3, 0, 1, 4, 2])
    sid = a.join(20)
    pos, slots = a.seq_slots(sid, 14, 4)
    assert pos.tolist() == [14, 15, 16, 17]
    assert slots.tolist() == [46, 47, 64, 65]
    with pytest.raises(ValueError):
        a.seq_slots(sid, 18, 3)


def test_allocator_model_slots_equal_those_of_decode_appends():
    """The slot the model names for token p is the slot a decode step assigned
    when it appended token p."""
    r = np.random.default_rng(7)
    a = BlockAllocatorModel(64, initial_free=r.permutation(64))
    s1, s2 = a.join(0), a.join(5)
    seen = {s1: [], s2: []}
    for _ in range(40):
        _, slots, _, _ = a.prepare_step([s2, s1], 8)
        seen[s2].append(int(slots[0]))
        seen[s1].append(int(slots[1]))
    assert a.seq_slots(s1, 0, 40)[1].tolist() == seen[s1]
    assert a.seq_slots(s2, 5, 40)[1].tolist() == seen[s2]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_equals_token_by_token_decode_appends(dtype):
    """Writing a prefix in one prefill leaves the cache exactly as appending its
    tokens one decode step at a time does (same rotation, same rounding)."""
    r = np.random.default_rng(3)
    nb, hkv, d, n = 8, 2, 16, 37
    rnd = round_to_f32 if dtype == "f32" else round_to_bf16
    k = rnd(r.standard_normal((n, hkv, d)))
    v = rnd(r.standard_normal((n, hkv, d)))
    kc0 = rnd(r.standard_normal((nb, hkv, 16, d)))
    vc0 = rnd(r.standard_normal((nb, hkv, 16, d)))
    a = BlockAllocatorModel(nb, initial_free=r.permutation(nb))
    sid = a.join(n)
    pos, slots = a.seq_slots(sid, 0, n)
    kc, vc = prefill_kv(k, v, pos, slots, kc0, vc0, base=10000.0, dtype=dtype)
    kd, vd = kc0, vc0
    for t in range(n):
        res = decode_step(np.zeros((1, hkv, d)), k[t:t + 1], v[t:t + 1], pos[t:t + 1],
                          slots[t:t + 1], np.array([t + 1]), np.array([a.seq_blocks(sid)]),
                          kd, vd, scale=1.0, base=10000.0, dtype=dtype)
        kd, vd = res["k_cache"], res["v_cache"]
    np.testing.assert_array_equal(kc, kd)
    np.testing.assert_array_equal(vc, vd)
    untouched = np.ones(nb, bool)
    untouched[a.seq_blocks(sid)] = False
    np.testing.assert_array_equal(kc[untouched], kc0[untouched])


def test_dense_assemble_extract_hand_example_and_round_trip():
    """Two rows of lengths 2 and 4 padded to 4: row 0's gap is columns 2..3; a
    decode column at 4 belongs to both rows; extracting drops the gap."""
    from oracle.dense import assemble_batch, extract_row, gap_bias
    a = np.arange(2 * 1 * 2, dtype=float).reshape(2, 1, 2) + 1
    b = np.arange(4 * 1 * 2, dtype=float).reshape(4, 1, 2) + 100
    dense = assemble_batch([a, b], 4, 8)
    assert dense.shape == (2, 8, 1, 2)
    np.testing.assert_array_equal(dense[0, :2], a)
    np.testing.assert_array_equal(dense[0, 2:], 0)
    np.testing.assert_array_equal(dense[1, :4], b)
    bias = gap_bias([2, 4], 4, 8)
    assert bias[0].tolist() == [0, 0, -np.inf, -np.inf, 0, 0, 0, 0]
    assert bias[1].tolist() == [0] * 8
    dense[:, 4] = [[[7, 8]], [[9, 10]]]           # one lockstep decode column
    np.testing.assert_array_equal(extract_row(dense, 0, 2, 4, 1),
                                  np.concatenate([a, [[[7, 8]]]]))
    np.testing.assert_array_equal(extract_row(dense, 1, 4, 4, 1),
                                  np.concatenate([b, [[[9, 10]]]]))
    np.testing.assert_array_equal(extract_row(assemble_batch([a, b], 4, 8), 0, 2, 4, 0), a)
