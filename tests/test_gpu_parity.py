"""GPU parity of the decode step (through the C ABI) against the float64 oracle.

Tolerances: attention output max-abs 1e-5 for float32 inputs and 2e-2 for bf16
inputs (float32 accumulation); rotated q/k within one ulp of the storage type;
allocator outputs, slot writes of V and untouched cache bytes bit-exact.
"""
import math

import numpy as np
import pytest
import torch

from helpers import (TOL, assert_out_close, assert_rope_close, dev, f64, gpu_single_step,
                     oracle_metadata, oracle_rows)
from oracle.step import decode_step
from paged_kv_decode_10_gb300 import binding, engine, workloads

pytestmark = pytest.mark.gpu


def _check_full_step(w, res, rows=None):
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    meta = oracle_metadata(w)
    for got, ref in zip(res["meta"], meta):
        np.testing.assert_array_equal(got, ref)          # a0 bit-exact
    rows = range(w.B) if rows is None else rows
    ref = oracle_rows(w, caches, tokens, meta, rows)
    out = f64(res["out"])
    worst = 0.0
    for b in rows:
        assert_rope_close(f64(res["q_rot"][b]), ref[b]["q_rot"], w.dtype)
        assert_rope_close(f64(res["k_rot"][b]), ref[b]["k_rot"], w.dtype)
        worst = max(worst, assert_out_close(out[b], ref[b]["out"], w.dtype, f"row {b}"))
    # append: V slot bit-exact, K slot = the kernel's own k_rot, everything else untouched
    pos, slots, lens, tables = meta
    k0, v0 = caches
    k1, v1 = res["k_cache"], res["v_cache"]
    touched = torch.zeros(k0.shape[0] * 16, dtype=torch.bool)
    touched[torch.from_numpy(slots)] = True
    touched = touched.view(k0.shape[0], 16)
    for b in range(w.B):
        blk, row = divmod(int(slots[b]), 16)
        assert torch.equal(v1[blk, :, row], tokens[2][b])
        assert torch.equal(k1[blk, :, row], res["k_rot"][b])
    keep = ~touched[:, None, :, None].expand_as(k0)
    assert torch.equal(k1[keep], k0[keep]) and torch.equal(v1[keep], v0[keep])
    assert res["err"] == 0
    return worst


def test_tiny_fp32_step():
    w = workloads.make_workload("tiny")
    _check_full_step(w, gpu_single_step(w))


def test_tiny_fp32_step_simt_vs_parts():
    w = workloads.make_workload("tiny")
    for parts in (1, 2, 5, 64):
        _check_full_step(w, gpu_single_step(w, num_parts=parts))


def test_decode16_bf16_step():
    w = workloads.make_workload("decode16")
    _check_full_step(w, gpu_single_step(w))


def test_decode16_bf16_simt_consumer():
    w = workloads.make_workload("decode16")
    _check_full_step(w, gpu_single_step(w, flags=binding.ATTN_SIMT))


def test_ragged64_bf16_step():
    w = workloads.make_workload("ragged64")
    _check_full_step(w, gpu_single_step(w))


def test_long131k_bf16_step():
    w = workloads.make_workload("long131k")
    res = gpu_single_step(w)
    _check_full_step(w, res)


def test_long131k_bf16_simt_consumer():
    w = workloads.make_workload("long131k")
    _check_full_step(w, gpu_single_step(w, flags=binding.ATTN_SIMT))


@pytest.mark.parametrize("parts", [1, 3, 152, 1000, 4096])
def test_split_count_invariance(parts):
    """Any partition of the pages into parts gives the same output (the LSE
    merge of any number of splits equals one split)."""
    w = workloads.make_workload("decode16")
    _check_full_step(w, gpu_single_step(w, num_parts=parts))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (16, 2)])
def test_shapes_and_ragged_tails(dtype, d, hq, hkv):
    """Lengths around page boundaries (0, 1, 15, 16, 17, 31, 32, 33 cached tokens)
    for every built head_dim / group size and both dtypes."""
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 100, 257]
    w = workloads.custom_workload("edges", lens, hq, hkv, d, dtype, seed=5)
    for flags in ([0, binding.ATTN_SIMT] if dtype == "bf16" else [0]):
        for parts in (None, 3):
            _check_full_step(w, gpu_single_step(w, num_parts=parts, flags=flags))


def test_empty_prefix_returns_new_value():
    """A row with no cached tokens attends only to its own new token: out = v."""
    w = workloads.custom_workload("fresh", [0, 0, 0], 8, 2, 128, "bf16", seed=6)
    res = gpu_single_step(w)
    v = workloads.make_new_tokens(w, 0, "cpu")[2]
    for b in range(3):
        for h in range(8):
            assert torch.equal(res["out"][b, h], v[b, h // 4])


def test_constant_values_give_constant_output():
    """V identical to c everywhere -> out == c for every row and head (pins the
    softmax normaliser and the split merge on the GPU)."""
    w = workloads.make_workload("ragged64")
    k_cache, v_cache = workloads.make_caches(w, "cpu")
    q, k, v = workloads.make_new_tokens(w, 0, "cpu")
    c = 0.375
    v_cache.fill_(c)
    v.fill_(c)
    res = gpu_single_step(w, caches=(k_cache, v_cache), tokens=(q, k, v))
    assert torch.all(res["out"] == c)


def test_ragged_batch_equals_rows_alone():
    """helexa issue 121: the ragged lockstep batch equals each row decoded alone."""
    w = workloads.make_workload("decode16")
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    full = gpu_single_step(w, caches=caches, tokens=tokens)
    meta = full["meta"]
    d = dev()
    k_cache, v_cache = (c.to(d) for c in caches)
    q, k, v = (t.to(d) for t in tokens)
    pos, slots, lens, tables = (torch.from_numpy(np.ascontiguousarray(m)).to(d) for m in meta)
    for b in range(w.B):
        q_rot, k_rot = binding.rope(q[b:b + 1], k[b:b + 1], pos[b:b + 1])
        kc, vc = k_cache.clone(), v_cache.clone()
        binding.append(k_rot, v[b:b + 1], slots[b:b + 1], kc, vc)
        out = binding.decode_attention(q_rot, kc, vc, tables[b:b + 1], lens[b:b + 1], w.scale)
        torch.cuda.synchronize()
        diff = (out[0].float().cpu() - full["out"][b].float()).abs().max().item()
        assert diff <= TOL["bf16"], (b, diff)


def test_block_table_permutation_invariance():
    """The same logical sequences stored under two different block layouts give
    the same output (paged equals contiguous)."""
    w = workloads.make_workload("decode16")
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    a = gpu_single_step(w, caches=caches, tokens=tokens)
    # relabel blocks: physical block p of layout A becomes block perm[p] of layout B
    perm = torch.from_numpy(np.random.default_rng(3).permutation(w.num_blocks))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_blocks)
    kb, vb = torch.empty_like(caches[0]), torch.empty_like(caches[1])
    kb[perm], vb[perm] = caches[0], caches[1]
    w2 = workloads.Workload(**{**w.__dict__})
    w2.free_order = perm.numpy()[w.free_order].astype(np.int32)
    b = gpu_single_step(w2, caches=(kb, vb), tokens=tokens)
    diff = (a["out"].float() - b["out"].float()).abs().max().item()
    assert diff <= TOL["bf16"]


def test_padded_batch_with_mask_equals_unpadded():
    """helexa issue 121, slice 1: rows right-padded to the batch max with a
    finite gap, an additive -inf mask over [prefix_len, padded_len), the new
    token after the gap and RoPE at the real position, equal the unpadded batch."""
    w = workloads.make_workload("tiny")
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    unpadded = gpu_single_step(w, caches=caches, tokens=tokens)
    d = dev()
    lens = [int(x) for x in w.seq_lens]
    P = max(lens)
    nb = 3 * (-(-(P + 1) // 16))
    alloc = binding.BlockAllocator(nb, 3, 4, np.arange(nb, dtype=np.int32)[::-1].copy())
    ids = [alloc.join(P) for _ in range(3)]
    _, slots, seq_lens, tables = alloc.prepare_step(ids, 4)
    # dense padded pool: real prefix, then a finite gap of garbage
    pos_u, _, _, tab_u = unpadded["meta"]
    kp = torch.randn(nb, w.Hkv, 16, w.d) * 50
    vp = torch.randn(nb, w.Hkv, 16, w.d) * 50
    for b, L in enumerate(lens):
        for t in range(L):
            src = (int(tab_u[b, t // 16]), t % 16)
            dst = (int(tables[b, t // 16]), t % 16)
            kp[dst[0], :, dst[1]] = caches[0][src[0], :, src[1]]
            vp[dst[0], :, dst[1]] = caches[1][src[0], :, src[1]]
    bias = torch.zeros(3, P + 1)
    for b, L in enumerate(lens):
        bias[b, L:P] = -math.inf
    q, k, v = (t.to(d) for t in tokens)
    positions = torch.tensor(lens, dtype=torch.int32, device=d)      # RoPE at real position
    kp, vp = kp.to(d), vp.to(d)
    q_rot, k_rot = binding.rope(q, k, positions)
    binding.append(k_rot, v, torch.from_numpy(slots).to(d), kp, vp)
    out = binding.decode_attention(q_rot, kp, vp, torch.from_numpy(tables).to(d),
                                   torch.from_numpy(seq_lens).to(d), w.scale,
                                   attn_bias=bias.to(d))
    torch.cuda.synchronize()
    assert (seq_lens == P + 1).all()
    diff = (out.cpu() - unpadded["out"]).abs().max().item()
    assert diff <= TOL["f32"], diff


def test_fully_masked_row_outputs_zero():
    w = workloads.custom_workload("masked", [40, 5], 8, 2, 64, "f32", seed=9)
    d = dev()
    caches = workloads.make_caches(w, "cpu")
    q, _, _ = workloads.make_new_tokens(w, 0, "cpu")
    meta = oracle_metadata(w)
    tables = torch.from_numpy(meta[3]).to(d)
    lens = torch.from_numpy(meta[2]).to(d)
    bias = torch.zeros(2, 64, device=d)
    bias[1, :] = -math.inf
    out = binding.decode_attention(q.to(d), caches[0].to(d), caches[1].to(d), tables, lens,
                                   w.scale, attn_bias=bias, num_parts=7)
    torch.cuda.synchronize()
    assert torch.all(out[1] == 0) and torch.isfinite(out).all()
    assert out[0].abs().sum() > 0


def test_device_error_flags_instead_of_faults():
    """Out-of-range block ids, slots and lengths are reported in the flag word
    and skipped (no access outside the buffers)."""
    w = workloads.custom_workload("bad", [20, 20], 8, 2, 128, "bf16", seed=10)
    d = dev()
    k_cache, v_cache = (c.to(d) for c in workloads.make_caches(w, "cpu"))
    q, k, v = (t.to(d) for t in workloads.make_new_tokens(w, 0, "cpu"))
    meta = oracle_metadata(w)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    tables = torch.from_numpy(meta[3]).to(d)
    tables[1, 0] = w.num_blocks + 1000
    lens = torch.from_numpy(meta[2]).to(d)
    binding.decode_attention(q, k_cache, v_cache, tables, lens, w.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & binding.DEVERR_BAD_BLOCK
    err.zero_()
    slots = torch.tensor([0, w.num_blocks * 16 + 5], dtype=torch.int64, device=d)
    kc = k_cache.clone()
    binding.append(k, v, slots, kc, v_cache.clone(), err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == binding.DEVERR_BAD_SLOT
    err.zero_()
    lens2 = lens.clone()
    lens2[0] = tables.shape[1] * 16 + 1
    out = binding.decode_attention(q, k_cache, v_cache, torch.from_numpy(meta[3]).to(d), lens2,
                                   w.scale, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & binding.DEVERR_BAD_LEN
    assert torch.all(out[0] == 0)


@pytest.mark.parametrize("name,parts", [("tiny", None), ("tiny", 7), ("decode16", None),
                                        ("ragged64", None), ("long131k", None),
                                        ("ragged64", 4096), ("decode16", 1)])
def test_planned_partition_equals_the_device_one(name, parts):
    """Attention through the host-planned partition (pkv_plan_parts, one record
    per part) is bit-identical to the partition the kernel derives itself; in
    check mode the kernel derives it too and finds no disagreement."""
    w = workloads.make_workload(name)
    res = gpu_single_step(w, num_parts=parts)
    dec = res["decoder"]
    B = w.B
    _, _, lens, tables = (np.array(x) for x in dec.last_metadata)
    plan = torch.from_numpy(binding.plan_parts(lens, w.Hkv, w.d, tables, dec.num_parts)).to(dev())
    args = (dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables, dec.seq_lens, dec.scale)
    ref = binding.decode_attention(*args, num_parts=dec.num_parts, err=dec.err)
    got = binding.decode_attention(*args, num_parts=dec.num_parts, plan=plan, err=dec.err)
    chk = binding.decode_attention(*args, num_parts=dec.num_parts, plan=plan, err=dec.err,
                                   flags=binding.ATTN_CHECK_PLAN)
    torch.cuda.synchronize()
    assert dec.device_errors() == 0
    assert torch.equal(got, ref) and torch.equal(chk, ref)
    assert torch.equal(ref.cpu(), res["out"])


def test_checked_plan_that_disagrees_is_flagged_and_not_used():
    w = workloads.make_workload("decode16")
    res = gpu_single_step(w)
    dec = res["decoder"]
    B = w.B
    _, _, lens, tables = (np.array(x) for x in dec.last_metadata)
    plan = binding.plan_parts(lens, w.Hkv, w.d, tables, dec.num_parts)
    bad = plan.copy()
    bad[5, 1] += 1            # row offset of part 5
    bad[9, 8] = bad[9, 9]     # first block id of part 9
    args = (dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables, dec.seq_lens, dec.scale)
    out = binding.decode_attention(*args, num_parts=dec.num_parts, err=dec.err,
                                   plan=torch.from_numpy(bad).to(dev()),
                                   flags=binding.ATTN_CHECK_PLAN)
    torch.cuda.synchronize()
    assert dec.device_errors() == binding.DEVERR_BAD_PLAN
    assert torch.equal(out.cpu(), res["out"])


def test_engine_without_plan_matches_engine_with_plan():
    w = workloads.make_workload("ragged64")
    res = gpu_single_step(w)
    d = dev()
    k_cache, v_cache = workloads.make_caches(w, "cpu")
    q, k, v = workloads.make_new_tokens(w, 0, "cpu")
    dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B,
                              w.max_blocks_per_seq(), initial_free=w.free_order, device=d,
                              k_cache=k_cache.to(d), v_cache=v_cache.to(d), plan=False)
    ids = [dec.join(int(L)) for L in w.seq_lens]
    out = dec.step(ids, q.to(d), k.to(d), v.to(d))
    torch.cuda.synchronize()
    assert res["decoder"].planned and not dec.planned
    assert torch.equal(out.cpu(), res["out"])


@pytest.mark.parametrize("name,flags", [("tiny", 0), ("decode16", 0), ("decode16", 1)])
def test_waits_that_give_up_report_a_timeout(name, flags):
    """With PKV_ATTN_SHORT_WAITS every wait inside the attention kernel gives up
    after ~64 clocks, long before any copy lands: the call still returns, the
    flag word carries PKV_DEVERR_TIMEOUT, the output holds only finite values
    (rows the kernel did not finish keep what the caller put there), and the
    next normal call, on a fresh workspace, is exact again (the kernel waited
    for its own copies before exiting; the context is healthy)."""
    w = workloads.make_workload(name)
    res = gpu_single_step(w, flags=flags)
    dec = res["decoder"]
    B = w.B
    d = dev()
    args = (dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables, dec.seq_lens, dec.scale)
    err = torch.zeros(1, dtype=torch.int32, device=d)
    out = torch.zeros_like(dec.out[:B])
    ws = binding.alloc_workspace(B, w.Hq, w.Hkv, w.d, dec.num_parts, d)
    binding.decode_attention(*args, num_parts=dec.num_parts, workspace=ws, out=out,
                             flags=flags | binding.ATTN_SHORT_WAITS, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & binding.DEVERR_TIMEOUT
    assert torch.isfinite(out.float()).all()
    err.zero_()
    again = binding.decode_attention(*args, num_parts=dec.num_parts, flags=flags, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(again.cpu(), res["out"])


@pytest.mark.parametrize("name,parts", [("long131k", None), ("long131k", 97), ("ragged64", None),
                                        ("decode16", 1000)])
def test_repeated_calls_on_one_workspace_are_identical(name, parts):
    """The fused merge leaves every counter of the workspace at zero: calls that
    reuse one workspace (helpers sharing a unit's merge when the grid fits on the
    GPU, the last part alone when it does not) give bit-identical outputs."""
    w = workloads.make_workload(name)
    res = gpu_single_step(w, num_parts=parts)
    dec = res["decoder"]
    B = w.B
    outs = []
    for _ in range(3):
        outs.append(binding.decode_attention(dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables,
                                             dec.seq_lens, dec.scale, num_parts=dec.num_parts,
                                             workspace=dec.workspace, err=dec.err))
    torch.cuda.synchronize()
    assert dec.device_errors() == 0
    for o in outs:
        assert torch.equal(o.cpu(), res["out"])
    region = (B * w.Hkv * 4 + 255) // 256 * 256      # the counter and done words
    assert int(dec.workspace[:2 * region].sum().item()) == 0


@pytest.mark.parametrize("flags", [0, 1])
def test_host_entry_point_matches_device_path(flags):
    """pkv_decode_step_host (host buffers in, host result out) equals the device
    call, with staging copies (0) or with the kernels reading the pinned inputs
    in place (PKV_HOST_IN_PLACE)."""
    w = workloads.make_workload("decode16")
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    ref = gpu_single_step(w, caches=caches, tokens=tokens)
    d = dev()
    bt = w.max_blocks_per_seq()
    dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                              initial_free=w.free_order, device=d,
                              k_cache=caches[0].to(d), v_cache=caches[1].to(d))
    ids = [dec.join(int(L)) for L in w.seq_lens]
    pos, slots, lens, tables = dec.alloc.prepare_step(ids, bt)
    q, k, v = tokens
    dq, dk, dv = torch.empty_like(q, device=d), torch.empty_like(k, device=d), torch.empty_like(v, device=d)
    args = dec.step_args(w.B, dq, dk, dv)
    out_h = torch.empty_like(q).pin_memory()
    pinned = [torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in (pos, slots, lens, tables)]
    io = binding.host_io(q.pin_memory(), k.pin_memory(), v.pin_memory(), *pinned, out_h,
                         flags=flags)
    binding.decode_step_host(args, io)
    assert torch.equal(out_h, ref["out"])


def _churn_case(dtype, d, hq, hkv, seed):
    r = np.random.default_rng(seed)
    B, steps, n_move = 8, 8, 2
    lens = r.integers(10, 60, size=B)
    nb = 200
    order = r.permutation(nb).astype(np.int32)
    return r, B, steps, n_move, lens, nb, order


@pytest.mark.parametrize("dtype,d,hq,hkv", [("bf16", 128, 32, 8), ("f32", 64, 8, 2),
                                            ("bf16", 64, 16, 2)])
def test_multi_step_churn_matches_oracle(dtype, d, hq, hkv):
    """Lockstep decode with rows leaving and joining between steps: each step's
    output and the allocator state match the oracle replaying the same history
    (block reuse after leave included)."""
    from oracle.allocator import BlockAllocatorModel
    r, B, steps, n_move, lens, nb, order = _churn_case(dtype, d, hq, hkv, 11)
    dv = dev()
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
    gen = torch.Generator().manual_seed(123)
    k_pool = torch.randn(nb, hkv, 16, d, generator=gen).to(tdt)
    v_pool = torch.randn(nb, hkv, 16, d, generator=gen).to(tdt)
    bt = 16
    dec = engine.PagedDecoder(nb, hq, hkv, d, dtype, B, bt, initial_free=order, device=dv,
                              num_parts=11, k_cache=k_pool.to(dv), v_cache=v_pool.to(dv))
    model = BlockAllocatorModel(nb, max_seqs=B, max_blocks_per_seq=bt, initial_free=order)
    ids = [dec.join(int(L)) for L in lens]
    assert ids == [model.join(int(L)) for L in lens]
    k_ref, v_ref = f64(k_pool), f64(v_pool)
    scale = 1 / math.sqrt(d)
    for step in range(steps):
        if step:
            leave = r.choice(B, size=n_move, replace=False)
            for row in leave:
                dec.leave(ids[row])
                model.leave(ids[row])
            for row in leave:
                pre = int(r.integers(0, 40))
                ids[row] = dec.join(pre)
                assert ids[row] == model.join(pre)
                # synthetic prefill stand-in: fresh prefix contents for the joiner
                blocks = model.seq_blocks(ids[row])
                fill_k = torch.randn(len(blocks), hkv, 16, d, generator=gen).to(tdt)
                fill_v = torch.randn(len(blocks), hkv, 16, d, generator=gen).to(tdt)
                idx = torch.tensor(blocks, dtype=torch.long)
                dec.k_cache[idx.to(dv)] = fill_k.to(dv)
                dec.v_cache[idx.to(dv)] = fill_v.to(dv)
                k_ref[blocks], v_ref[blocks] = f64(fill_k), f64(fill_v)
        q = torch.randn(B, hq, d, generator=gen).to(tdt)
        k = torch.randn(B, hkv, d, generator=gen).to(tdt)
        v = torch.randn(B, hkv, d, generator=gen).to(tdt)
        out = dec.step(ids, q.to(dv), k.to(dv), v.to(dv))
        torch.cuda.synchronize()
        pos, slots, seq_lens, tables = model.prepare_step(ids, bt)
        for got, want in zip(dec.last_metadata, (pos, slots, seq_lens, tables)):
            np.testing.assert_array_equal(got, want)
        ref = decode_step(f64(q), f64(k), f64(v), pos, slots, seq_lens, tables, k_ref, v_ref,
                          scale=scale, base=10000.0, dtype=dtype)
        k_ref, v_ref = ref["k_cache"], ref["v_cache"]
        assert_out_close(f64(out), ref["out"], dtype, f"step {step}")
        assert dec.alloc.free_stack() == model.free
    assert dec.device_errors() == 0


def test_fused_rope_append_equals_separate_calls():
    w = workloads.make_workload("ragged64")
    d = dev()
    k_cache, v_cache = (c.to(d) for c in workloads.make_caches(w, "cpu"))
    q, k, v = (t.to(d) for t in workloads.make_new_tokens(w, 0, "cpu"))
    pos, slots, _, _ = (torch.from_numpy(np.ascontiguousarray(m)).to(d)
                        for m in oracle_metadata(w))
    kc1, vc1 = k_cache.clone(), v_cache.clone()
    q1, k1 = binding.rope(q, k, pos)
    binding.append(k1, v, slots, kc1, vc1)
    kc2, vc2 = k_cache.clone(), v_cache.clone()
    q2, k2 = binding.rope_append(q, k, v, pos, slots, kc2, vc2)
    torch.cuda.synchronize()
    assert torch.equal(q1, q2) and torch.equal(k1, k2)
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)


@pytest.mark.parametrize("name,parts", [("tiny", None), ("tiny", 1000), ("decode16", 7),
                                        ("long131k", None)])
def test_separate_merge_equals_fused(name, parts):
    """a4 as its own launch (pkv_lse_merge) gives the same output as the merge
    fused into the split kernel's epilogue, and re-merging is idempotent."""
    w = workloads.make_workload(name)
    fused = gpu_single_step(w, num_parts=parts)
    sep = gpu_single_step(w, num_parts=parts, flags=binding.ATTN_SEPARATE_MERGE)
    # the fused merge may split a unit's partials among several threads and
    # CTAs: same value up to float32 summation order, i.e. within one ulp of
    # the output type
    close = 1e-6 if w.dtype == "f32" else 1e-2
    assert (fused["out"].float() - sep["out"].float()).abs().max() <= close
    _check_full_step(w, sep)
    dec = fused["decoder"]
    B = w.B
    # re-merging rewrites the multi-part units with the same values and leaves
    # the single-part units alone
    again = fused["out"].to(d := dev())
    binding.lse_merge(dec.workspace, dec.seq_lens[:B], dec.bt_stride, B, w.Hq, w.Hkv, w.d,
                      dec.num_parts, again)
    torch.cuda.synchronize()
    assert (again.cpu().float() - fused["out"].float()).abs().max() <= close


@pytest.mark.parametrize("metadata", ["copy", "mapped"])
def test_graph_replay_matches_eager_steps(metadata):
    """The captured step (metadata H2D, or none when the kernels read the pinned
    metadata in place, + rope/append + attention in one CUDA graph) gives
    bit-identical outputs and caches to the eager C ABI calls."""
    w = workloads.make_workload("decode16")
    d = dev()
    caches = workloads.make_caches(w, "cpu")
    bt = w.max_blocks_per_seq(extra_tokens=8)
    decs = []
    for mode in ("copy", metadata):
        dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                  initial_free=w.free_order, device=d,
                                  k_cache=caches[0].to(d), v_cache=caches[1].to(d),
                                  metadata=mode)
        decs.append((dec, [dec.join(int(L)) for L in w.seq_lens]))
    (eager, ids_e), (graph, ids_g) = decs
    graph.capture(w.B)
    for step in range(4):
        q, k, v = (t.to(d) for t in workloads.make_new_tokens(w, step, "cpu"))
        out_e = eager.step(ids_e, q, k, v).clone()
        graph.q_in[:w.B].copy_(q)
        graph.k_in[:w.B].copy_(k)
        graph.v_in[:w.B].copy_(v)
        graph.prepare_host(ids_g)
        out_g = graph.replay_step().clone()
        torch.cuda.synchronize()
        assert torch.equal(out_e, out_g), step
    assert torch.equal(eager.k_cache, graph.k_cache) and torch.equal(eager.v_cache, graph.v_cache)
    assert eager.device_errors() == 0 and graph.device_errors() == 0


@pytest.mark.parametrize("name", ["tiny", "decode16", "ragged64", "churn256", "long131k"])
def test_whole_step_kernel_equals_split_launch(name):
    """The one-launch step (RoPE and append inside the attention kernel) gives
    bit-identical q_rot, k_rot, caches and output to the default two launches
    (pkv_rope_append, then the attention kernel)."""
    w = workloads.make_workload(name)
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    fused = gpu_single_step(w, caches=caches, tokens=tokens, flags=binding.STEP_FUSED)
    split = gpu_single_step(w, caches=caches, tokens=tokens)
    for key in ("out", "q_rot", "k_rot", "k_cache", "v_cache"):
        assert torch.equal(fused[key], split[key]), key
    assert fused["err"] == 0 and split["err"] == 0


@pytest.mark.parametrize("seed", range(8))
def test_whole_step_kernel_random_shapes(seed):
    """The one-launch step on the random batches, head groupings, head sizes,
    dtypes and partition counts: bit-identical to the two launches."""
    lens, hq, hkv, d, dtype, parts = _random_case(seed)
    w = workloads.custom_workload(f"rand{seed}", lens, hq, hkv, d, dtype, seed=seed)
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    fused = gpu_single_step(w, caches=caches, tokens=tokens, num_parts=parts,
                            flags=binding.STEP_FUSED)
    split = gpu_single_step(w, caches=caches, tokens=tokens, num_parts=parts)
    for key in ("out", "q_rot", "k_rot", "k_cache", "v_cache"):
        assert torch.equal(fused[key], split[key]), key
    assert fused["err"] == 0 and split["err"] == 0


@pytest.mark.parametrize("name,flags", [("tiny", 0), ("ragged64", 0), ("ragged64", 4),
                                        ("long131k", 0), ("tiny", 1)])
def test_mapped_metadata_equals_device_copy(name, flags):
    """Kernels reading positions, slots, seq_lens and block tables in place from
    pinned host memory give bit-identical results to reading a device copy."""
    w = workloads.make_workload(name)
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    a = gpu_single_step(w, caches=caches, tokens=tokens, flags=flags)
    b = gpu_single_step(w, caches=caches, tokens=tokens, flags=flags, metadata="mapped")
    for key in ("out", "q_rot", "k_rot", "k_cache", "v_cache"):
        assert torch.equal(a[key], b[key]), key
    assert a["err"] == 0 and b["err"] == 0


def test_mapped_metadata_churn_eager_and_graph():
    """Rows leave and join between steps; eager steps and graph replays of a
    decoder with in-place host metadata track a device-copy decoder exactly
    (the two pinned buffers alternate, so a refill never races a running step)."""
    w = workloads.make_workload("decode16")
    d = dev()
    caches = workloads.make_caches(w, "cpu")
    bt = w.max_blocks_per_seq(extra_tokens=64)
    r = np.random.default_rng(7)
    decs = []
    for mode in ("copy", "mapped", "mapped"):
        dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                  initial_free=w.free_order, device=d,
                                  k_cache=caches[0].to(d), v_cache=caches[1].to(d),
                                  metadata=mode)
        decs.append([dec, [dec.join(int(L)) for L in w.seq_lens]])
    decs[2][0].capture(w.B)
    for step in range(6):
        if step in (2, 4):
            row = int(r.integers(0, w.B))
            pre = int(r.integers(1, 40))
            for entry in decs:
                entry[0].leave(entry[1][row])
                entry[1][row] = entry[0].join(pre)
        q, k, v = (t.to(d) for t in workloads.make_new_tokens(w, step, "cpu"))
        outs = [decs[0][0].step(decs[0][1], q, k, v).clone(),
                decs[1][0].step(decs[1][1], q, k, v).clone()]
        g = decs[2][0]
        g.q_in[:w.B].copy_(q)
        g.k_in[:w.B].copy_(k)
        g.v_in[:w.B].copy_(v)
        g.prepare_host(decs[2][1])
        outs.append(g.replay_step().clone())
        torch.cuda.synchronize()
        assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2]), step
    for dec, _ in decs[1:]:
        assert torch.equal(dec.k_cache, decs[0][0].k_cache)
        assert torch.equal(dec.v_cache, decs[0][0].v_cache)
        assert dec.device_errors() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_variants_keep_two_ctas_per_sm(d):
    """The bf16 tensor-core kernels are sized (registers, shared memory) for two
    resident CTAs per SM; the default partition is SMs x 2 parts."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert binding.default_parts(d, binding.BF16) == 2 * sms


@pytest.mark.parametrize("metadata", ["mapped", "copy"])
def test_host_step_reads_inputs_in_place(metadata):
    """The end-to-end host step (q/k/v read in place from pinned host buffers,
    output copied back inside the graph) gives the device step's outputs."""
    w = workloads.make_workload("decode16")
    d = dev()
    caches = workloads.make_caches(w, "cpu")
    bt = w.max_blocks_per_seq(extra_tokens=8)
    decs = []
    for mode in ("copy", metadata):
        dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                  initial_free=w.free_order, device=d,
                                  k_cache=caches[0].to(d), v_cache=caches[1].to(d),
                                  metadata=mode)
        decs.append((dec, [dec.join(int(L)) for L in w.seq_lens]))
    (ref, ids_r), (host, ids_h) = decs
    host.capture_host(w.B)
    for step in range(4):
        q, k, v = workloads.make_new_tokens(w, step, "cpu")
        out_r = ref.step(ids_r, q.to(d), k.to(d), v.to(d)).cpu()
        host.q_host.copy_(q)
        host.k_host.copy_(k)
        host.v_host.copy_(v)
        out_h = host.host_step(ids_h).clone()
        assert torch.equal(out_r, out_h), step
    torch.cuda.synchronize()
    assert torch.equal(ref.k_cache, host.k_cache) and torch.equal(ref.v_cache, host.v_cache)
    assert ref.device_errors() == 0 and host.device_errors() == 0


def _random_case(seed):
    r = np.random.default_rng(1000 + seed)
    hkv = int(r.choice([1, 2, 4, 8]))
    g = int(r.choice([1, 2, 4, 8]))
    d = int(r.choice([64, 128]))
    dtype = "f32" if r.random() < 0.25 else "bf16"
    B = int(r.integers(1, 24))
    # short rows (0, 1, page edges) next to long ones: the partition then cuts
    # parts inside a unit's boundary positions, and many parts span no page
    pool = [0, 1, 15, 16, 17, 31, 32, 33, int(r.integers(34, 300)), int(r.integers(300, 900))]
    lens = [int(r.choice(pool)) for _ in range(B)]
    parts = int(r.choice([1, 5, 37, 152, 304, 1000, 4096]))
    return lens, g * hkv, hkv, d, dtype, parts


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes_and_partitions_match_oracle(seed):
    """Random batches (ragged, with empty and one-token rows), head groupings,
    head sizes, dtypes and partition counts: every step matches the oracle."""
    lens, hq, hkv, d, dtype, parts = _random_case(seed)
    w = workloads.custom_workload(f"rand{seed}", lens, hq, hkv, d, dtype, seed=seed)
    res = gpu_single_step(w, num_parts=parts)
    _check_full_step(w, res)


@pytest.mark.parametrize("flags", [0, 1])
def test_step_graph_matches_host_step(flags):
    """The captured host step (pkv_step_graph) run over several steps gives the
    per-call host step's outputs and caches, with staging copies or in place."""
    w = workloads.make_workload("decode16")
    d = dev()
    caches = workloads.make_caches(w, "cpu")
    bt = w.max_blocks_per_seq(extra_tokens=8)
    runs = []
    for use_graph in (False, True):
        dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                  initial_free=w.free_order, device=d,
                                  k_cache=caches[0].to(d), v_cache=caches[1].to(d))
        ids = [dec.join(int(L)) for L in w.seq_lens]
        q0, k0, v0 = workloads.make_new_tokens(w, 0, "cpu")
        qh, kh, vh = q0.pin_memory(), k0.pin_memory(), v0.pin_memory()
        meta_h = (torch.empty(w.B, dtype=torch.int32).pin_memory(),
                  torch.empty(w.B, dtype=torch.int64).pin_memory(),
                  torch.empty(w.B, dtype=torch.int32).pin_memory(),
                  torch.empty((w.B, bt), dtype=torch.int32).pin_memory())
        meta_d = [torch.empty_like(m, device=d) for m in meta_h]
        dq, dk, dv = (torch.empty_like(t, device=d) for t in (q0, k0, v0))
        out_h = torch.empty_like(q0).pin_memory()
        args = binding.make_step_args(dq, dk, dv, dec.q_rot[:w.B], dec.k_rot[:w.B], dec.k_cache,
                                      dec.v_cache, *meta_d, dec.scale, dec.rope_base,
                                      dec.num_parts, dec.workspace, dec.out[:w.B], err=dec.err)
        io = binding.host_io(qh, kh, vh, *meta_h, out_h, flags=flags)
        graph = binding.StepGraph(args, io) if use_graph else None
        prepare = dec.alloc.step_runner(ids, bt, tuple(m.numpy() for m in meta_h))
        outs = []
        for step in range(4):
            q, k, v = workloads.make_new_tokens(w, step, "cpu")
            qh.copy_(q)
            kh.copy_(k)
            vh.copy_(v)
            prepare()
            if use_graph:
                graph.launch()
            else:
                binding.decode_step_host(args, io)
            outs.append(out_h.clone())
        if graph is not None:
            graph.close()
        torch.cuda.synchronize()
        runs.append((outs, dec.k_cache.clone(), dec.v_cache.clone(), dec.device_errors()))
    (o1, k1, v1, e1), (o2, k2, v2, e2) = runs
    for a, b in zip(o1, o2):
        assert torch.equal(a, b)
    assert torch.equal(k1, k2) and torch.equal(v1, v2) and e1 == 0 and e2 == 0


@pytest.mark.parametrize("flags,fused", [(0, False), (1, False), (1, True)])
def test_step_graph_pipelined_matches_sequential(flags, fused):
    """Two captured host steps over two sets of pinned buffers, each step
    enqueued behind the running one and the running one then waited for with
    pkv_step_graph_wait (each set's allocator step keeps its own cached row
    state, two steps stale), give the outputs and caches of one graph launched
    and waited for step by step; with PKV_STEP_FUSED in the pipelined graphs
    only (the whole step in one kernel, reading q/k/v in place), bit for bit
    too."""
    w = workloads.make_workload("decode16")
    d = dev()
    caches = workloads.make_caches(w, "cpu")
    S = 5
    bt = w.max_blocks_per_seq(extra_tokens=S + 2)
    runs = []
    for pipelined in (False, True):
        dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                  initial_free=w.free_order, device=d,
                                  k_cache=caches[0].to(d), v_cache=caches[1].to(d))
        ids = [dec.join(int(L)) for L in w.seq_lens]
        q0, k0, v0 = workloads.make_new_tokens(w, 0, "cpu")
        dq, dk, dv = (torch.empty_like(t, device=d) for t in (q0, k0, v0))
        meta_d = [torch.empty(w.B, dtype=torch.int32, device=d),
                  torch.empty(w.B, dtype=torch.int64, device=d),
                  torch.empty(w.B, dtype=torch.int32, device=d),
                  torch.empty((w.B, bt), dtype=torch.int32, device=d)]
        args = binding.make_step_args(dq, dk, dv, dec.q_rot[:w.B], dec.k_rot[:w.B], dec.k_cache,
                                      dec.v_cache, *meta_d, dec.scale, dec.rope_base,
                                      dec.num_parts, dec.workspace, dec.out[:w.B], err=dec.err,
                                      flags=binding.STEP_FUSED if fused and pipelined else 0)
        sets = []
        for _ in range(2 if pipelined else 1):
            qkv = tuple(t.pin_memory() for t in (q0, k0, v0))
            meta_h = (torch.empty(w.B, dtype=torch.int32).pin_memory(),
                      torch.empty(w.B, dtype=torch.int64).pin_memory(),
                      torch.empty(w.B, dtype=torch.int32).pin_memory(),
                      torch.empty((w.B, bt), dtype=torch.int32).pin_memory())
            out_h = torch.empty_like(q0).pin_memory()
            io = binding.host_io(*qkv, *meta_h, out_h, flags=flags)
            prepare = dec.alloc.step_runner(ids, bt, tuple(m.numpy() for m in meta_h),
                                            row_state=np.full(3 * w.B, -1, np.int32))
            sets.append((qkv, out_h, prepare, binding.StepGraph(args, io), io))
        outs = [None] * S
        for step in range(S):
            qkv, out_h, prepare, graph, _ = sets[step % len(sets)]
            for dst, src in zip(qkv, workloads.make_new_tokens(w, step, "cpu")):
                dst.copy_(src)
            prepare()
            if pipelined:
                graph.enqueue()                 # queued behind step - 1
                if step > 0:
                    prev = sets[(step - 1) % 2]
                    prev[3].wait()
                    outs[step - 1] = prev[1].clone()
            else:
                graph.launch()
                outs[step] = out_h.clone()
        if pipelined:
            sets[(S - 1) % 2][3].wait()
            outs[S - 1] = sets[(S - 1) % 2][1].clone()
        for s in sets:
            s[3].close()
        torch.cuda.synchronize()
        runs.append((outs, dec.k_cache.clone(), dec.v_cache.clone(), dec.device_errors()))
    (o1, k1, v1, e1), (o2, k2, v2, e2) = runs
    for step, (a, b) in enumerate(zip(o1, o2)):
        assert torch.equal(a, b), step
    assert torch.equal(k1, k2) and torch.equal(v1, v2) and e1 == 0 and e2 == 0
