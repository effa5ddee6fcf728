"""Host-side checks of the C ABI: exported symbols and the C++ block allocator
against the hand-derived trace and against the allocator model (bit-exact)."""
import json
import os
import re

import numpy as np
import pytest

from oracle.allocator import BlockAllocatorModel, OutOfBlocks
from oracle.allocator import UnknownSequence as ModelUnknown

HERE = os.path.dirname(__file__)
HEADER = os.path.join(os.path.dirname(HERE), "include", "pkv.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function(host_lib):
    from paged_kv_decode_10_gb300 import binding
    names = header_functions()
    assert len(names) >= 18
    for name in names:
        assert hasattr(host_lib, name), name
        assert name in binding.SIGNATURES, name
    assert host_lib.pkv_abi_version() == 5


def test_binding_constants_match_the_header():
    """Status codes, dtype codes, flag bits and error bits of the binding are the
    values the header defines."""
    from paged_kv_decode_10_gb300 import binding
    defines = dict((m.group(1), int(m.group(2))) for m in re.finditer(
        r"#define PKV_([A-Z0-9_]+)\s+(\d+)", open(HEADER).read()))
    checked = 0
    for name, value in defines.items():
        if hasattr(binding, name):
            assert getattr(binding, name) == value, name
            checked += 1
    for must in ("ATTN_SIMT", "ATTN_SEPARATE_MERGE", "STEP_FUSED", "ATTN_SHORT_WAITS",
                 "DEVERR_TIMEOUT", "ERR_CUDA", "BF16", "HOST_IN_PLACE",
                 "LAYERS_MERGE_HELPERS"):
        assert must in defines and hasattr(binding, must), must
    assert checked >= 18


def _run_trace(alloc_cls, errors):
    with open(os.path.join(HERE, "golden", "allocator_trace.json")) as f:
        g = json.load(f)
    a = alloc_cls(g)
    for op in g["ops"]:
        err = op.get("error")
        if op["op"] == "join":
            if err:
                with pytest.raises(errors["out_of_blocks"]):
                    a.join(op["prefix"])
            else:
                assert a.join(op["prefix"]) == op["seq_id"]
        elif op["op"] == "leave":
            if err:
                with pytest.raises(errors["unknown_seq"]):
                    a.leave(op["seq_id"])
            else:
                a.leave(op["seq_id"])
        else:
            if err:
                with pytest.raises(errors["out_of_blocks"]):
                    a.prepare_step(op["seq_ids"], g["bt_stride"])
            else:
                pos, slots, lens, tables = a.prepare_step(op["seq_ids"], g["bt_stride"])
                assert pos.tolist() == op["positions"]
                assert slots.tolist() == op["slots"]
                assert lens.tolist() == op["seq_lens"]
                assert tables.tolist() == op["tables"]
        assert a.free_stack() == op["free_after"], op
    for sid, blocks in g["final_tables"].items():
        assert a.seq_blocks(int(sid)) == blocks
        assert a.seq_len(int(sid)) == g["final_lengths"][sid]


def test_cpp_allocator_golden_trace(host_lib):
    from paged_kv_decode_10_gb300 import binding

    def make(g):
        return binding.BlockAllocator(g["num_blocks"], g["max_seqs"], g["bt_stride"],
                                      g["initial_free"])
    _run_trace(make, {"out_of_blocks": binding.OutOfBlocks,
                      "unknown_seq": binding.UnknownSequence})


class _ModelAdapter(BlockAllocatorModel):
    def free_stack(self):
        return list(self.free)


def test_model_allocator_golden_trace_adapter():
    _run_trace(lambda g: _ModelAdapter(g["num_blocks"], g["block_size"], g["max_seqs"],
                                       initial_free=g["initial_free"]),
               {"out_of_blocks": OutOfBlocks, "unknown_seq": ModelUnknown})


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_cpp_allocator_matches_model_under_churn(host_lib, seed):
    from paged_kv_decode_10_gb300 import binding
    r = np.random.default_rng(seed)
    nb, max_seqs, bt = 400, 24, 40
    order = r.permutation(nb).astype(np.int32)
    cpp = binding.BlockAllocator(nb, max_seqs, bt, order)
    model = BlockAllocatorModel(nb, max_seqs=max_seqs, max_blocks_per_seq=bt,
                                initial_free=order)
    live = []
    for _ in range(600):
        act = r.integers(0, 4)
        if act == 0 and len(live) < max_seqs:
            L = int(r.integers(0, 200))
            try:
                s_m = model.join(L)
            except OutOfBlocks:
                with pytest.raises(binding.OutOfBlocks):
                    cpp.join(L)
                continue
            assert cpp.join(L) == s_m
            live.append(s_m)
        elif act == 1 and live:
            s = live.pop(int(r.integers(0, len(live))))
            model.leave(s)
            cpp.leave(s)
        elif live:
            ids = [s for s in live if model.seq_len(s) < (bt - 1) * 16]
            r.shuffle(ids)
            try:
                ref = model.prepare_step(ids, bt)
            except OutOfBlocks:
                with pytest.raises(binding.OutOfBlocks):
                    cpp.prepare_step(ids, bt)
                continue
            got = cpp.prepare_step(ids, bt)
            for a_, b_ in zip(ref, got):
                np.testing.assert_array_equal(a_, b_)
        assert cpp.free_stack() == model.free
        assert cpp.num_free() == model.num_free()
        for s in live:
            assert cpp.seq_blocks(s) == model.seq_blocks(s)
            assert cpp.seq_len(s) == model.seq_len(s)
            L = model.seq_len(s)
            if L:
                start = int(r.integers(0, L))
                count = int(r.integers(0, L - start + 1))
                for a_, b_ in zip(model.seq_slots(s, start, count),
                                  cpp.seq_slots(s, start, count)):
                    np.testing.assert_array_equal(a_, b_)


def test_cpp_allocator_rejects_bad_input(host_lib):
    from paged_kv_decode_10_gb300 import binding
    with pytest.raises(binding.PkvError):
        binding.BlockAllocator(4, 2, 2, [0, 1, 1, 2])          # not a permutation
    a = binding.BlockAllocator(8, 2, 2)
    s = a.join(3)
    with pytest.raises(binding.PkvError):
        a.prepare_step([s, s], 2)                             # duplicate row
    with pytest.raises(binding.UnknownSequence):
        a.prepare_step([1], 2)
    with pytest.raises(binding.PkvError):
        a.join(33)                                            # wider than a table
    with pytest.raises(binding.UnknownSequence):
        a.leave(5)
    with pytest.raises(binding.PkvError):
        a.seq_slots(s, 2, 2)                                  # beyond the length
    with pytest.raises(binding.PkvError):
        a.seq_slots(s, -1, 1)
    with pytest.raises(binding.UnknownSequence):
        a.seq_slots(1, 0, 1)
    assert a.seq_len(s) == 3 and a.num_free() == 7


def test_pool_blocks_from_budget(host_lib):
    """Blocks that fit a byte budget: K and V, 16 tokens, every KV head and
    layer per block (floor)."""
    from paged_kv_decode_10_gb300 import binding
    per_block = 32 * 2 * 8 * 16 * 128 * 2          # 32 layers, bf16, Hkv 8, d 128
    assert binding.pool_blocks(per_block * 1000, 32, 8, 128, binding.BF16) == 1000
    assert binding.pool_blocks(per_block * 1000 - 1, 32, 8, 128, binding.BF16) == 999
    assert binding.pool_blocks(per_block - 1, 32, 8, 128, binding.BF16) == 0
    assert binding.pool_blocks(4 * 2 * 2 * 16 * 64 * 4 * 7, 4, 2, 64, binding.F32) == 7
    # a quarter of 280 GB for a 32-layer, 8-KV-head, d=128 bf16 model
    assert binding.pool_blocks(70 * 10**9, 32, 8, 128, binding.BF16) == 70 * 10**9 // per_block
    with pytest.raises(binding.PkvError):
        binding.pool_blocks(1 << 30, 0, 8, 128, binding.BF16)


def test_step_runner_matches_prepare_step(host_lib):
    """The precomputed-pointer allocator step gives prepare_step's outputs and state."""
    from paged_kv_decode_10_gb300 import binding
    order = np.random.default_rng(5).permutation(64).astype(np.int32)
    a = binding.BlockAllocator(64, 4, 16, order)
    b = binding.BlockAllocator(64, 4, 16, order)
    ids_a = [a.join(L) for L in (3, 16, 40)]
    ids_b = [b.join(L) for L in (3, 16, 40)]
    out = (np.empty(3, np.int32), np.empty(3, np.int64), np.empty(3, np.int32),
           np.empty((3, 16), np.int32))
    run = b.step_runner(ids_b, 16, out)
    for _ in range(20):
        ref = a.prepare_step(ids_a, 16)
        got = run()
        for x, y in zip(ref, got):
            np.testing.assert_array_equal(x, y)
    assert a.free_stack() == b.free_stack()


@pytest.mark.parametrize("seed", [0, 1])
def test_batched_join_leave_equal_single_calls_in_order(host_lib, seed):
    """pkv_seqs_join / pkv_seqs_leave against the allocator model doing the same
    joins and leaves one at a time: same ids, prefix slots, tables and free
    stack (bit-exact); a batch that cannot be taken whole changes nothing."""
    from paged_kv_decode_10_gb300 import binding
    r = np.random.default_rng(100 + seed)
    nb, max_seqs, bt = 300, 20, 30
    order = r.permutation(nb).astype(np.int32)
    cpp = binding.BlockAllocator(nb, max_seqs, bt, order)
    model = BlockAllocatorModel(nb, max_seqs=max_seqs, max_blocks_per_seq=bt,
                                initial_free=order)
    live = []

    def same_state():
        assert cpp.free_stack() == model.free
        for s in live:
            assert cpp.seq_blocks(s) == model.seq_blocks(s)
            assert cpp.seq_len(s) == model.seq_len(s)

    for _ in range(60):
        if live and r.random() < 0.5:
            k = int(r.integers(1, len(live) + 1))
            leave = [live[i] for i in r.choice(len(live), size=k, replace=False)]
            cpp.leave_many(leave)
            for s in leave:
                model.leave(s)
                live.remove(s)
        n = int(r.integers(0, max_seqs - len(live) + 1))
        prefixes = r.integers(0, 120, size=n).astype(np.int32)
        need = int(sum(-(-int(p) // 16) for p in prefixes))
        pos = np.full(int(prefixes.sum()) + 3, -7, np.int32)
        slots = np.full(int(prefixes.sum()) + 3, -7, np.int64)
        if need > model.num_free():
            before = cpp.free_stack()
            with pytest.raises(binding.OutOfBlocks):
                cpp.join_many(prefixes, (pos, slots))
            assert cpp.free_stack() == before and (pos == -7).all()
            same_state()
            continue
        ids = cpp.join_many(prefixes, (pos, slots))
        k = 0
        for sid, p in zip(ids, prefixes):
            assert sid == model.join(int(p))
            live.append(int(sid))
            mp, ms = model.seq_slots(int(sid), 0, int(p))
            np.testing.assert_array_equal(pos[k:k + p], mp)
            np.testing.assert_array_equal(slots[k:k + p], ms)
            k += int(p)
        assert (pos[k:] == -7).all()
        same_state()
        if live:   # a step so that lengths and tables move between batches
            ids_s = [s for s in live if model.seq_len(s) < (bt - 1) * 16]
            try:
                ref = model.prepare_step(ids_s, bt)
            except OutOfBlocks:
                continue
            for a_, b_ in zip(ref, cpp.prepare_step(ids_s, bt)):
                np.testing.assert_array_equal(a_, b_)
    # leave: an unknown or repeated id rejects the whole batch
    if len(live) >= 2:
        before = cpp.free_stack()
        with pytest.raises(binding.PkvError):
            cpp.leave_many([live[0], live[0]])
        with pytest.raises(binding.UnknownSequence):
            cpp.leave_many([live[1], max_seqs + 5])
        assert cpp.free_stack() == before
        same_state()
    # join: more joiners than free ids, or a prefix longer than a table, changes nothing
    before = cpp.free_stack()
    with pytest.raises(binding.PkvError):
        cpp.join_many([0] * (max_seqs - len(live) + 1))
    with pytest.raises(binding.PkvError):
        cpp.join_many([1, bt * 16 + 1])
    assert cpp.free_stack() == before
    same_state()


def test_binding_rejects_arrays_the_library_would_misread(host_lib):
    """Output arrays of the wrong dtype, layout or length are refused before the
    C side writes through them."""
    from paged_kv_decode_10_gb300 import binding
    a = binding.BlockAllocator(64, 4, 8)
    sid = a.join(20)
    with pytest.raises(binding.PkvError):
        a.seq_slots(sid, 0, 20, out=(np.empty(20, np.int64), np.empty(20, np.int64)))
    with pytest.raises(binding.PkvError):
        a.seq_slots(sid, 0, 20, out=(np.empty(20, np.int32), np.empty(19, np.int64)))
    with pytest.raises(binding.PkvError):
        a.join_many([5, 7], (np.empty(12, np.int32), np.empty(11, np.int64)))
    with pytest.raises(binding.PkvError):
        a.prepare_step([sid], 8, out=(np.empty(1, np.int32), np.empty(1, np.int64),
                                      np.empty(1, np.int32), np.empty((1, 16), np.int32)[:, ::2]))
    assert a.num_free() == 64 - 2          # nothing above changed the allocator
    pos, slots = a.seq_slots(sid, 0, 20)
    assert pos.tolist() == list(range(20))


def _plan_by_enumeration(lens, Hkv, d, tables, bt_stride, bias_stride, C):
    """The attention partition written out position by position: every unit
    (row, KV head) of a row with n > 0 pages is A positions without a page
    followed by its n pages, units in row-major order; part c owns positions
    [P*c // C, P*(c+1) // C).  Record fields as pkv.h states them."""
    A = 4 if d <= 64 else 2
    pos = []      # (row, KV head, page or -1)
    for b, L in enumerate(lens):
        ok = 0 <= L <= bt_stride * 16 and (bias_stride <= 0 or L <= bias_stride)
        n = -(-L // 16) if ok else 0
        for g in range(Hkv if n else 0):
            pos += [(b, g, -1)] * A + [(b, g, j) for j in range(n)]
    P = len(pos)
    out = np.zeros((C, 24), np.int64)
    for c in range(C):
        rec = [-1, 0, 0, 0, P & 0xffffffff, P >> 32, 0, 0] + [-1] * 16
        start, end = P * c // C, P * (c + 1) // C
        if start < end:
            b, g, _ = pos[start]
            pages = [j for (bb, gg, j) in pos[start:end] if (bb, gg) == (b, g) and j >= 0]
            rec[0] = b
            rec[1] = sum(1 for (bb, gg, _) in pos if bb < b) // Hkv
            rec[2] = lens[b]
            rec[3] = lens[b + 1] if b + 1 < len(lens) else 0
            for i, j in enumerate(pages[:16]):
                rec[8 + i] = tables[b][j]
        out[c] = rec
    return out


@pytest.mark.parametrize("seed", range(12))
def test_plan_parts_equals_the_partition_written_out(host_lib, seed):
    """pkv_plan_parts bit-exact against the partition enumerated position by
    position (ragged rows, empty rows, lengths the kernel rejects, a bias
    stride, fewer and more parts than positions)."""
    from paged_kv_decode_10_gb300 import binding
    r = np.random.default_rng(seed)
    B = int(r.integers(1, 14))
    Hkv = int(r.choice([1, 2, 4, 8]))
    d = int(r.choice([64, 128]))
    bt = int(r.integers(2, 40))
    lens = r.integers(0, bt * 16 + 1, size=B)
    lens[r.random(B) < 0.15] = 0
    if seed % 4 == 1:
        lens[0] = bt * 16 + 5                  # longer than the table: not counted
    bias_stride = int(r.integers(1, bt * 16)) if seed % 3 == 2 else 0
    tables = r.integers(0, 10000, size=(B, bt)).astype(np.int32)
    for C in (1, 3, 7, 64, 304, 1000):
        got = binding.plan_parts(lens.astype(np.int32), Hkv, d, tables, C, bias_stride,
                                 out=np.full((C, 24), -1, np.int32))
        want = _plan_by_enumeration([int(x) for x in lens], Hkv, d, tables.tolist(), bt,
                                    bias_stride, C)
        # (ids past a segment's last page are not written: -1 from the fill above)
        np.testing.assert_array_equal(got.astype(np.int64), want, err_msg=f"C={C}")


def test_plan_parts_rejects_bad_arguments(host_lib):
    from paged_kv_decode_10_gb300 import binding
    lens = np.array([5], np.int32)
    tables = np.zeros((1, 1), np.int32)
    with pytest.raises(binding.PkvError):
        binding.plan_parts(lens, 2, 96, tables, 4)          # head_dim not built
    with pytest.raises(binding.PkvError):
        binding.plan_parts(lens, 0, 64, tables, 4)          # no KV head


def test_prepare_step_cached_equals_prepare_step_under_churn(host_lib):
    """pkv_prepare_step_cached writing into two alternating table buffers (as the
    serving loop does) leaves every output and each buffer exactly as
    pkv_prepare_step writes them, through joins and leaves that reuse sequence
    ids and blocks, over many steps."""
    from paged_kv_decode_10_gb300 import binding
    r = np.random.default_rng(5)
    nb, B, bt = 400, 12, 12
    perm = r.permutation(nb).astype(np.int32)
    full = binding.BlockAllocator(nb, 64, bt, perm)
    cached = binding.BlockAllocator(nb, 64, bt, perm)
    lens0 = r.integers(0, 60, size=B)
    rows = [[a.join(int(L)) for L in lens0] for a in (full, cached)]
    assert rows[0] == rows[1]
    bufs = []
    for _ in range(2):
        out = (np.empty(B, np.int32), np.empty(B, np.int64), np.empty(B, np.int32),
               np.full((B, bt), 7777, np.int32))          # stale garbage to begin with
        bufs.append((out, np.full(3 * B, -1, np.int32)))
    for step in range(60):
        if step % 3 == 2:
            leave = r.choice(B, size=3, replace=False)
            prefixes = r.integers(0, 40, size=3)
            for a, ids in zip((full, cached), rows):
                a.leave_many([ids[i] for i in leave])
                for i, sid in zip(leave, a.join_many(prefixes)):
                    ids[i] = int(sid)
            assert rows[0] == rows[1]
        want = full.prepare_step(rows[0], bt)
        out, state = bufs[step % 2]
        got = cached.prepare_step_cached(rows[1], bt, out, state)
        for g, w_ in zip(got, want):
            np.testing.assert_array_equal(g, w_)
        assert full.free_stack() == cached.free_stack()
