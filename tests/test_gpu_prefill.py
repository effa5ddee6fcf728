"""Prefix KV of joining sequences (pkv_seq_slots + pkv_prefill_kv) against the
float64 oracle, and the decode steps that follow such a prefill."""
import numpy as np
import pytest
import torch

from helpers import assert_out_close, assert_rope_close, dev, f64
from oracle.allocator import BlockAllocatorModel
from oracle.step import decode_step, prefill_kv
from paged_kv_decode_10_gb300 import binding, engine

pytestmark = pytest.mark.gpu


def _tdtype(dtype):
    return torch.float32 if dtype == "f32" else torch.bfloat16


def _joiners(r, nb, prefixes, bt):
    order = r.permutation(nb).astype(np.int32)
    alloc = binding.BlockAllocator(nb, len(prefixes) + 2, bt, order)
    model = BlockAllocatorModel(nb, max_seqs=len(prefixes) + 2, max_blocks_per_seq=bt,
                                initial_free=order)
    ids = [alloc.join(int(p)) for p in prefixes]
    assert ids == [model.join(int(p)) for p in prefixes]
    return alloc, model, ids


def _token_list(alloc, model, ids, prefixes):
    pos, slots = [], []
    for s, p in zip(ids, prefixes):
        a = alloc.seq_slots(s, 0, int(p))
        for x, y in zip(a, model.seq_slots(s, 0, int(p))):
            np.testing.assert_array_equal(x, y)
        pos.append(a[0])
        slots.append(a[1])
    return np.concatenate(pos), np.concatenate(slots)


@pytest.mark.parametrize("dtype,d,hkv", [("bf16", 128, 8), ("f32", 64, 2), ("bf16", 64, 4)])
def test_prefill_matches_oracle_and_touches_only_its_slots(dtype, d, hkv):
    r = np.random.default_rng(11)
    prefixes = [1, 16, 17, 250, 33]
    nb = 40
    alloc, model, ids = _joiners(r, nb, prefixes, 32)
    pos, slots = _token_list(alloc, model, ids, prefixes)
    T = len(pos)
    g = torch.Generator().manual_seed(5)
    td = _tdtype(dtype)
    k = torch.randn((T, hkv, d), generator=g).to(td)
    v = torch.randn((T, hkv, d), generator=g).to(td)
    kc0 = torch.randn((nb, hkv, 16, d), generator=g).to(td)
    vc0 = torch.randn((nb, hkv, 16, d), generator=g).to(td)
    D = dev()
    kc, vc = kc0.to(D), vc0.to(D)
    err = torch.zeros(1, dtype=torch.int32, device=D)
    binding.prefill_kv(k.to(D), v.to(D), torch.from_numpy(pos).to(D),
                       torch.from_numpy(slots).to(D), kc, vc, err=err)
    torch.cuda.synchronize()
    rk, rv = prefill_kv(f64(k), f64(v), pos, slots, f64(kc0), f64(vc0), base=10000.0,
                        dtype=dtype)
    assert_rope_close(f64(kc), rk, dtype)
    np.testing.assert_array_equal(f64(vc), rv)          # values are copied bit for bit
    written = np.zeros((nb, 16), bool)
    written[slots // 16, slots % 16] = True
    rows = lambda x: f64(x).transpose(0, 2, 1, 3)[~written]   # [slot, Hkv, d]
    np.testing.assert_array_equal(rows(kc), rows(kc0))
    np.testing.assert_array_equal(rows(vc), rows(vc0))
    assert int(err.item()) == 0


def test_prefill_rows_equal_decode_append_rows():
    """A prefix token's stored key is bit-identical to the key a decode step's
    append stores for the same raw key at the same position."""
    r = np.random.default_rng(2)
    w_hkv, d, nb = 8, 128, 300
    prefixes = [700, 3, 1900]
    alloc, model, ids = _joiners(r, nb, prefixes, 160)
    pos, slots = _token_list(alloc, model, ids, prefixes)
    T = len(pos)
    D = dev()
    g = torch.Generator().manual_seed(8)
    k = torch.randn((T, w_hkv, d), generator=g).to(torch.bfloat16).to(D)
    v = torch.randn((T, w_hkv, d), generator=g).to(torch.bfloat16).to(D)
    caches = [torch.zeros((nb, w_hkv, 16, d), dtype=torch.bfloat16, device=D) for _ in range(4)]
    p_d, s_d = torch.from_numpy(pos).to(D), torch.from_numpy(slots).to(D)
    binding.prefill_kv(k, v, p_d, s_d, caches[0], caches[1])
    binding.rope_append(k.clone(), k, v, p_d, s_d, caches[2], caches[3])
    torch.cuda.synchronize()
    assert torch.equal(caches[0], caches[2]) and torch.equal(caches[1], caches[3])


def test_chunked_prefill_equals_one_call():
    r = np.random.default_rng(4)
    prefixes = [300, 129]
    alloc, model, ids = _joiners(r, 60, prefixes, 32)
    pos, slots = _token_list(alloc, model, ids, prefixes)
    T = len(pos)
    D = dev()
    g = torch.Generator().manual_seed(9)
    k = torch.randn((T, 4, 64), generator=g).to(torch.bfloat16).to(D)
    v = torch.randn((T, 4, 64), generator=g).to(torch.bfloat16).to(D)
    one = [torch.zeros((60, 4, 16, 64), dtype=torch.bfloat16, device=D) for _ in range(2)]
    chunked = [torch.zeros_like(one[0]) for _ in range(2)]
    p_d, s_d = torch.from_numpy(pos).to(D), torch.from_numpy(slots).to(D)
    binding.prefill_kv(k, v, p_d, s_d, *one)
    edges = [0, 1, 8, 24, 57, 300, 301, 333, T]
    for a, b in zip(edges[:-1], edges[1:]):
        binding.prefill_kv(k[a:b], v[a:b], p_d[a:b], s_d[a:b], *chunked)
    torch.cuda.synchronize()
    assert torch.equal(one[0], chunked[0]) and torch.equal(one[1], chunked[1])


@pytest.mark.parametrize("dtype,d,hq,hkv", [("bf16", 128, 32, 8), ("f32", 64, 8, 2)])
def test_joiners_prefilled_then_decoded_match_oracle(dtype, d, hq, hkv):
    """Rows join with a prefix whose KV is written by the prefill (raw keys at
    their own positions), then decode together; every step's output matches
    the oracle replaying the same prefill and steps."""
    r = np.random.default_rng(21)
    prefixes = [37, 1, 300, 16, 129]
    B, nb, steps = len(prefixes), 80, 3
    bt = 24
    order = r.permutation(nb).astype(np.int32)
    D = dev()
    td = _tdtype(dtype)
    g = torch.Generator().manual_seed(3)
    kc0 = torch.zeros((nb, hkv, 16, d), dtype=td)
    dec = engine.PagedDecoder(nb, hq, hkv, d, dtype, B, bt, initial_free=order, device=D,
                              k_cache=kc0.to(D), v_cache=kc0.clone().to(D))
    model = BlockAllocatorModel(nb, max_seqs=B, max_blocks_per_seq=bt, initial_free=order)
    ids = [dec.join(int(p)) for p in prefixes]
    assert ids == [model.join(int(p)) for p in prefixes]
    pos, slots = _token_list(dec.alloc, model, ids, prefixes)
    T = len(pos)
    k = torch.randn((T, hkv, d), generator=g).to(td)
    v = torch.randn((T, hkv, d), generator=g).to(td)
    binding.prefill_kv(k.to(D), v.to(D), torch.from_numpy(pos).to(D),
                       torch.from_numpy(slots).to(D), dec.k_cache, dec.v_cache, err=dec.err)
    rk, rv = prefill_kv(f64(k), f64(v), pos, slots, f64(kc0), f64(kc0), base=10000.0,
                        dtype=dtype)
    for step in range(steps):
        q = torch.randn((B, hq, d), generator=g).to(td)
        kn = torch.randn((B, hkv, d), generator=g).to(td)
        vn = torch.randn((B, hkv, d), generator=g).to(td)
        out = dec.step(ids, q.to(D), kn.to(D), vn.to(D)).cpu()
        p_, s_, l_, t_ = model.prepare_step(ids, bt)
        ref = decode_step(f64(q), f64(kn), f64(vn), p_, s_, l_, t_, rk, rv,
                          scale=1.0 / np.sqrt(d), base=10000.0, dtype=dtype)
        rk, rv = ref["k_cache"], ref["v_cache"]
        assert_out_close(f64(out), ref["out"], dtype, f"step {step}")
    assert dec.device_errors() == 0


def test_prefill_skips_negative_slots_and_flags_bad_ones():
    """A negative slot writes nothing; a slot past the pool sets PKV_DEVERR_BAD_SLOT
    and is skipped; every other token is still written."""
    D = dev()
    nb, hkv, d = 8, 2, 64
    kc = torch.zeros((nb, hkv, 16, d), dtype=torch.bfloat16, device=D)
    vc = torch.zeros_like(kc)
    g = torch.Generator().manual_seed(1)
    k = torch.randn((4, hkv, d), generator=g).to(torch.bfloat16).to(D)
    v = torch.randn((4, hkv, d), generator=g).to(torch.bfloat16).to(D)
    pos = torch.tensor([0, 1, 2, 3], dtype=torch.int32, device=D)
    slots = torch.tensor([5, -1, nb * 16 + 3, 17], dtype=torch.int64, device=D)
    err = torch.zeros(1, dtype=torch.int32, device=D)
    binding.prefill_kv(k, v, pos, slots, kc, vc, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & binding.DEVERR_BAD_SLOT
    written = torch.zeros((nb, 16), dtype=torch.bool)
    written[0, 5] = written[1, 1] = True
    got = vc.transpose(1, 2).reshape(nb, 16, hkv, d).cpu()
    assert torch.equal(got[0, 5], v[0].cpu()) and torch.equal(got[1, 1], v[3].cpu())
    assert not got[~written].any()
