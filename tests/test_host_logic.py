"""Host-side logic that needs no GPU: the workload recipes, the packed step
metadata layout and the benchmark's byte accounting."""
import math

import numpy as np
import pytest

from paged_kv_decode_10_gb300 import workloads


def _pages(n_tokens):
    return -(-int(n_tokens) // 16)


@pytest.mark.parametrize("name", workloads.WORKLOAD_NAMES)
def test_workload_recipe(name):
    w = workloads.make_workload(name)
    spec = {   # B, Hq, Hkv, d, dtype, length range
        "tiny": (3, 4, 2, 64, "f32", (5, 33)),
        "decode16": (16, 32, 8, 64, "bf16", (128, 2048)),
        "ragged64": (64, 32, 8, 128, "bf16", (1, 4096)),
        "churn256": (256, 32, 8, 128, "bf16", (512, 8192)),
        "long131k": (1, 32, 4, 128, "bf16", (131072, 131072)),
    }[name]
    B, Hq, Hkv, d, dtype, (lo, hi) = spec
    assert (w.B, w.Hq, w.Hkv, w.d, w.dtype) == (B, Hq, Hkv, d, dtype)
    assert len(w.seq_lens) == B and lo <= w.seq_lens.min() and w.seq_lens.max() <= hi
    assert abs(w.scale - 1 / math.sqrt(d)) < 1e-15
    if name != "tiny":
        # the pool holds 1.25x the blocks the rows need after one append
        assert w.num_blocks == math.ceil(1.25 * sum(_pages(L + 1) for L in w.seq_lens))
    # the free list is a permutation of every block
    assert sorted(w.free_order.tolist()) == list(range(w.num_blocks))
    # seeded: the same recipe twice gives the same arrays
    w2 = workloads.make_workload(name)
    np.testing.assert_array_equal(w.seq_lens, w2.seq_lens)
    np.testing.assert_array_equal(w.free_order, w2.free_order)


def test_churn_plan():
    w = workloads.make_workload("churn256")
    assert w.steps == 64 and len(w.churn) == 64
    for leave, prefixes in w.churn:
        assert len(leave) == len(prefixes) == 26            # 10% of 256, rounded
        assert len(set(leave.tolist())) == 26 and leave.min() >= 0 and leave.max() < 256
        assert prefixes.min() >= 256 and prefixes.max() <= 1024
    # the lengths follow the clipped lognormal: median near 2048
    assert 1700 < np.median(w.seq_lens) < 2400


def test_new_tokens_are_seeded_and_rounded():
    w = workloads.make_workload("decode16")
    q, k, v = workloads.make_new_tokens(w, 3, "cpu")
    q2, _, _ = workloads.make_new_tokens(w, 3, "cpu")
    q3, _, _ = workloads.make_new_tokens(w, 4, "cpu")
    assert tuple(q.shape) == (16, 32, 64) and tuple(k.shape) == tuple(v.shape) == (16, 8, 64)
    assert str(q.dtype) == "torch.bfloat16"
    assert bool((q == q2).all()) and not bool((q == q3).all())


def test_metadata_layout_is_aligned_and_disjoint():
    from paged_kv_decode_10_gb300.engine import _metadata_layout
    for B in (1, 3, 16, 255, 256):
        for bt in (1, 7, 160, 8193):
            for parts in (0, 1, 304):
                o_slots, o_pos, o_lens, o_tab, o_plan, end = _metadata_layout(B, bt, parts)
                spans = sorted([(o_slots, 8 * B), (o_pos, 4 * B), (o_lens, 4 * B),
                                (o_tab, 4 * B * bt), (o_plan, 96 * parts)])
                for (a, n), (b, _) in zip(spans, spans[1:]):
                    assert a + n <= b                   # no overlap
                assert o_slots % 8 == 0 and o_pos % 4 == 0 and o_lens % 4 == 0
                assert o_tab % 16 == 0 and o_plan % 16 == 0   # 16-byte aligned rows / records
                assert end == o_plan + 96 * parts


def test_attention_byte_accounting_hand_example():
    import bench
    # two rows of 17 and 32 tokens after the append, 4 query / 2 KV heads, d=8, 2-byte type:
    # K and V: (17 + 32) tokens * 2 heads * 8 * 2 (K and V) * 2 B = 3136
    # q in and out: 2 rows * 4 heads * 8 * 2 B * 2 = 256
    # block-table entries: (2 + 2) * 4 B = 16; seq_lens: 2 * 4 B = 8
    assert bench.attn_bytes([17, 32], 4, 2, 8, 2) == 3136 + 256 + 16 + 8


def test_roofline_peaks():
    import bench
    assert bench.NOMINAL_HBM_GBS > bench.FALLBACK_HBM_GBS > 0
    peak, kind = bench.measured_peak()
    assert peak > 0 and kind in ("measured", "fallback")


def test_long_units_rule():
    """A unit of n pages counts as long when n * num_parts >= 8 * P (P: pages
    plus 2 per unit at d = 128, 4 at d = 64, over every unit)."""
    from paged_kv_decode_10_gb300.engine import long_units
    # one 131073-token row, 4 KV heads: 8193 pages per unit, P = 4 * 8195
    assert long_units([131073], 4, 128, 304)
    assert not long_units([131073], 4, 128, 32)          # 8193 * 32 < 8 * 32780
    assert long_units([131073], 4, 128, 33)              # 8193 * 33 >= 8 * 32780
    # 64 rows of at most 4097 tokens over 304 parts: nothing spans 8 parts
    assert not long_units([4097] * 64, 8, 128, 304)
    # empty rows add nothing to P; an all-empty step has no long unit
    assert not long_units([0, 0, 4096], 1, 64, 8)        # 256 * 8 < 8 * 260
    assert long_units([0, 0, 4096], 1, 64, 9)
    assert not long_units([0, 0], 8, 128, 304)
