"""churn256 at full size (B=256, 32/8 heads, d=128, bf16) in the launch
configuration the benchmark times: the default partition, step metadata read
in place from pinned host memory, one CUDA graph replay per step, and before
every step after the first 26 rows leave and 26 join (one pkv_seqs_leave and one
pkv_seqs_join call, which also gives the joiners' prefix slots) with a prefix
whose KV pkv_prefill_kv writes into their new blocks.

The oracle cannot redo a 256-row step at this size in seconds, so it checks
sampled rows one by one: each sampled row replays its own history in float64
(its initial blocks, or its joiner prefix written by the oracle's prefill, then
one decode append per step).  The allocator's step metadata is checked
bit-exact for every row against the allocator model."""
import numpy as np
import pytest
import torch

from helpers import assert_out_close, dev, f64
from oracle.allocator import BlockAllocatorModel
from oracle.step import decode_step, prefill_kv
from paged_kv_decode_10_gb300 import binding, engine, workloads

pytestmark = pytest.mark.gpu

STEPS = 4


def _token_major(blocks_kv, n):
    """[blocks, Hkv, 16, d] -> the first n tokens as [n, Hkv, d]."""
    x = np.asarray(blocks_kv).transpose(0, 2, 1, 3)
    return x.reshape(-1, x.shape[2], x.shape[3])[:n]


def _oracle_row_step(hist, q, k, v, pos, w):
    """One decode step of a single row over its private token history."""
    n = pos + 1
    nblk = -(-n // 16)
    kc = np.zeros((nblk * 16, w.Hkv, w.d))
    vc = np.zeros_like(kc)
    kc[:pos], vc[:pos] = hist["k"], hist["v"]
    kc = kc.reshape(nblk, 16, w.Hkv, w.d).transpose(0, 2, 1, 3)
    vc = vc.reshape(nblk, 16, w.Hkv, w.d).transpose(0, 2, 1, 3)
    ref = decode_step(q[None], k[None], v[None], [pos], [pos], [n], np.arange(nblk)[None, :],
                      kc, vc, scale=w.scale, base=w.rope_base, dtype=w.dtype)
    hist["k"] = np.concatenate([hist["k"], ref["k_rot"]], 0)
    hist["v"] = np.concatenate([hist["v"], v[None]], 0)
    return ref["out"][0]


def test_churn256_graph_steps_match_oracle_on_sampled_rows():
    w = workloads.make_workload("churn256")
    D = dev()
    k0, v0 = workloads.make_caches(w, "cpu")
    bt = w.max_blocks_per_seq(extra_tokens=STEPS + 16)
    dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                              initial_free=w.free_order, device=D, k_cache=k0.to(D),
                              v_cache=v0.to(D), metadata="mapped")
    model = BlockAllocatorModel(w.num_blocks, max_seqs=w.B, max_blocks_per_seq=bt,
                                initial_free=w.free_order)
    ids = [dec.join(int(L)) for L in w.seq_lens]
    assert ids == [model.join(int(L)) for L in w.seq_lens]

    # sampled rows: some of every churn step's joiners, rows that stay, the
    # longest and the shortest initial rows
    moved = set()
    sample = []
    for s in range(1, STEPS):
        leave = [int(x) for x in w.churn[s - 1][0]]
        moved.update(leave)
        sample += leave[:3]
    stay = [b for b in range(w.B) if b not in moved]
    by_len = sorted(stay, key=lambda b: int(w.seq_lens[b]))
    sample += [by_len[0], by_len[-1], stay[len(stay) // 2]]
    sample = sorted(set(sample))
    hist = {}
    for b in sample:
        L = int(w.seq_lens[b])
        blocks = torch.tensor(model.seq_blocks(ids[b]), dtype=torch.long)
        hist[b] = dict(k=_token_major(f64(k0[blocks]), L), v=_token_major(f64(v0[blocks]), L))
    del k0, v0

    gen = torch.Generator().manual_seed(4242)
    dec.capture(w.B)
    checked = 0
    for s in range(STEPS):
        if s:
            leave, prefixes = w.churn[s - 1]
            dec.alloc.leave_many([ids[row] for row in leave])
            for row in leave:
                model.leave(ids[row])
            total = int(np.sum(prefixes))
            pos_all = np.empty(total, np.int32)
            slot_all = np.empty(total, np.int64)
            joined = dec.alloc.join_many(prefixes, (pos_all, slot_all))
            pre_k, pre_v = [], []
            k_off = 0
            for row, pre, sid in zip(leave, prefixes, joined):
                row, pre = int(row), int(pre)
                ids[row] = int(sid)
                assert ids[row] == model.join(pre)
                mp, msl = model.seq_slots(ids[row], 0, pre)
                np.testing.assert_array_equal(pos_all[k_off:k_off + pre], mp)
                np.testing.assert_array_equal(slot_all[k_off:k_off + pre], msl)
                k_off += pre
                kr = torch.randn((pre, w.Hkv, w.d), generator=gen).to(torch.bfloat16)
                vr = torch.randn((pre, w.Hkv, w.d), generator=gen).to(torch.bfloat16)
                pre_k.append(kr)
                pre_v.append(vr)
                if row in hist:
                    nblk = -(-pre // 16)
                    z = np.zeros((nblk, w.Hkv, 16, w.d))
                    kc, vc = prefill_kv(f64(kr), f64(vr), np.arange(pre), np.arange(pre), z, z,
                                        base=w.rope_base, dtype=w.dtype)
                    hist[row] = dict(k=_token_major(kc, pre), v=_token_major(vc, pre))
            binding.prefill_kv(torch.cat(pre_k).to(D), torch.cat(pre_v).to(D),
                               torch.from_numpy(pos_all).to(D), torch.from_numpy(slot_all).to(D),
                               dec.k_cache, dec.v_cache, base=w.rope_base, err=dec.err)
        q, k, v = workloads.make_new_tokens(w, s, "cpu")
        dec.q_in[:w.B].copy_(q)
        dec.k_in[:w.B].copy_(k)
        dec.v_in[:w.B].copy_(v)
        meta = [np.array(x) for x in dec.prepare_host(ids)]
        for got, want in zip(meta, model.prepare_step(ids, bt)):
            np.testing.assert_array_equal(got, want)          # a0 bit-exact, every row
        out = f64(dec.replay_step())
        torch.cuda.synchronize()
        assert np.isfinite(out).all()
        qf, kf, vf = f64(q), f64(k), f64(v)
        for b in sample:
            pos = int(meta[0][b])
            assert pos == hist[b]["k"].shape[0]
            ref = _oracle_row_step(hist[b], qf[b], kf[b], vf[b], pos, w)
            assert_out_close(out[b], ref, w.dtype, f"step {s} row {b} (position {pos})")
            checked += 1
    assert checked >= 4 * STEPS
    assert dec.device_errors() == 0
