"""The native serving loop (pkv_server) against the Python engine and the oracle.

Both drive the same continuous-batching run -- rows leave, joiners with a
prefix take their rows (prefix K/V written by the prefill kernel), every row
decodes one token per step -- from the same seeded state: outputs and caches
must be bit-identical at every step, and the last step's outputs must match
the float64 oracle on the caches they were computed from.
"""
import numpy as np
import pytest
import torch

from helpers import assert_out_close, dev, f64
from oracle.step import decode_step
from paged_kv_decode_10_gb300 import binding, engine, workloads

pytestmark = pytest.mark.gpu


def _decoder(w, caches, bt, **kw):
    d = dev()
    return engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                               initial_free=w.free_order, device=d, k_cache=caches[0].to(d),
                               v_cache=caches[1].to(d), metadata="mapped", **kw)


@pytest.mark.parametrize("dtype,d,hq,hkv", [("bf16", 128, 32, 8), ("f32", 64, 8, 2)])
def test_server_matches_engine_and_oracle(dtype, d, hq, hkv):
    r = np.random.default_rng(17)
    B, steps, move = 24, 10, 3
    lens = r.integers(40, 400, size=B)
    w = workloads.custom_workload("serve", lens, hq, hkv, d, dtype, seed=21, pool_factor=3.0)
    bt = w.max_blocks_per_seq(extra_tokens=600)
    caches = workloads.make_caches(w, "cpu")
    ref = _decoder(w, caches, bt)
    srv_dec = _decoder(w, caches, bt)
    ids = [ref.join(int(L)) for L in w.seq_lens]
    srv_ids = [srv_dec.join(int(L)) for L in w.seq_lens]
    assert ids == srv_ids
    max_prefix = move * 200
    server = binding.Server(srv_dec, srv_ids, max_prefix)
    dv = dev()
    tdt = workloads.torch_dtype(dtype)
    pos_buf = np.empty(max_prefix, np.int32)
    slot_buf = np.empty(max_prefix, np.int64)
    for s in range(steps):
        leave = np.sort(r.choice(B, size=move, replace=False)).astype(np.int32) if s else \
            np.zeros(0, np.int32)
        prefixes = r.integers(1, 200, size=len(leave)).astype(np.int32)
        n = int(prefixes.sum())
        g = torch.Generator(device=dv).manual_seed(100 + s)
        pk = torch.randn((max(n, 1), hkv, d), generator=g, device=dv).to(tdt)
        pv = torch.randn((max(n, 1), hkv, d), generator=g, device=dv).to(tdt)
        q, k, v = workloads.make_new_tokens(w, s, dv)
        # the Python engine: batched leave/join, prefill, one decode step
        if len(leave):
            ref.alloc.leave_many([ids[i] for i in leave])
            joined = ref.alloc.join_many(prefixes, (pos_buf, slot_buf))
            for i, sid in zip(leave, joined):
                ids[i] = int(sid)
            binding.prefill_kv(pk[:n], pv[:n], torch.from_numpy(pos_buf[:n]).to(dv),
                               torch.from_numpy(slot_buf[:n]).to(dv), ref.k_cache, ref.v_cache,
                               err=ref.err)
        out_ref = ref.step(ids, q, k, v)
        # the native server: one call
        server.step(leave, prefixes, pk[:n] if n else None, pv[:n] if n else None, q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(srv_dec.out[:B], out_ref), f"step {s}"
    assert ref.device_errors() == 0 and srv_dec.device_errors() == 0
    assert server.rows().tolist() == ids
    assert torch.equal(srv_dec.k_cache, ref.k_cache) and torch.equal(srv_dec.v_cache, ref.v_cache)
    # the last step against the oracle, row by row, on the caches it read (the
    # oracle re-appends the step's token, which the caches already hold)
    pos, slots, seq_lens, tables = (np.array(x) for x in ref.last_metadata)
    q64, k64, v64 = (f64(t) for t in (q, k, v))
    kc, vc = ref.k_cache.cpu(), ref.v_cache.cpu()
    got = f64(srv_dec.out[:B])
    for b in range(B):
        nblk = -(-int(seq_lens[b]) // 16)
        blocks = torch.from_numpy(tables[b, :nblk].astype(np.int64))
        j = int(pos[b]) // 16
        res = decode_step(q64[b:b + 1], k64[b:b + 1], v64[b:b + 1], pos[b:b + 1],
                          [j * 16 + int(slots[b]) % 16], seq_lens[b:b + 1],
                          np.arange(nblk)[None, :], f64(kc[blocks]), f64(vc[blocks]),
                          scale=w.scale, base=w.rope_base, dtype=dtype)
        assert_out_close(got[b], res["out"][0], dtype, f"row {b}")
    server.close()


def test_server_rejects_bad_steps():
    w = workloads.custom_workload("serve2", [30, 50, 70], 8, 2, 64, "bf16", seed=3)
    caches = workloads.make_caches(w, "cpu")
    dec = _decoder(w, caches, w.max_blocks_per_seq(extra_tokens=64))
    ids = [dec.join(int(L)) for L in w.seq_lens]
    server = binding.Server(dec, ids, 32)
    with pytest.raises(binding.PkvError):
        server.step(np.array([5], np.int32), np.array([4], np.int32))       # no row 5
    with pytest.raises(binding.PkvError):
        server.step(np.array([0, 0], np.int32), np.array([4, 4], np.int32))  # row twice
    with pytest.raises(binding.PkvError):
        server.step(np.array([1], np.int32), np.array([33], np.int32))      # prefix too long
    assert server.rows().tolist() == ids                                  # nothing changed
    server.step(np.zeros(0, np.int32), np.zeros(0, np.int32))             # still usable
    torch.cuda.synchronize()
    assert dec.device_errors() == 0
    server.close()


def test_server_churn256_full_size_matches_engine():
    """churn256 at full size (B=256, 26 leave / 26 join per step with prefixes of
    256-1024 tokens) through the native serving loop, against the Python engine
    replaying its captured graph (the launch configuration the full-size churn
    test checks against the oracle): bit-identical outputs at every step and
    identical caches and row map at the end; the last step's sampled rows also
    against the oracle on the caches they read."""
    w = workloads.make_workload("churn256")
    dv = dev()
    steps = 8
    bt = w.max_blocks_per_seq(extra_tokens=steps + 16)
    k0, v0 = workloads.make_caches(w, dv)
    decs = [engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                initial_free=w.free_order, device=dv, k_cache=k0.clone(),
                                v_cache=v0.clone(), metadata="mapped") for _ in range(2)]
    del k0, v0
    ref, srv_dec = decs
    ids = [ref.join(int(L)) for L in w.seq_lens]
    srv_ids = [srv_dec.join(int(L)) for L in w.seq_lens]
    max_prefix = max(int(np.sum(p)) for _, p in w.churn[:steps])
    server = binding.Server(srv_dec, srv_ids, max_prefix)
    ref.capture(w.B)
    gen = torch.Generator(device=dv).manual_seed(99)
    pre_k = torch.randn((max_prefix, w.Hkv, w.d), generator=gen, device=dv).to(torch.bfloat16)
    pre_v = torch.randn((max_prefix, w.Hkv, w.d), generator=gen, device=dv).to(torch.bfloat16)
    pos_buf = np.empty(max_prefix, np.int32)
    slot_buf = np.empty(max_prefix, np.int64)
    for s in range(steps):
        leave, prefixes = w.churn[s - 1] if s else (np.zeros(0, np.int64), np.zeros(0, np.int64))
        n = int(np.sum(prefixes))
        if s:
            ref.alloc.leave_many([ids[i] for i in leave])
            for i, sid in zip(leave, ref.alloc.join_many(prefixes, (pos_buf, slot_buf))):
                ids[int(i)] = int(sid)
            binding.prefill_kv(pre_k[:n], pre_v[:n], torch.from_numpy(pos_buf[:n]).to(dv),
                               torch.from_numpy(slot_buf[:n]).to(dv), ref.k_cache, ref.v_cache,
                               err=ref.err)
        q, k, v = workloads.make_new_tokens(w, s, dv)
        ref.q_in[:w.B].copy_(q)
        ref.k_in[:w.B].copy_(k)
        ref.v_in[:w.B].copy_(v)
        ref.prepare_host(ids)
        out_ref = ref.replay_step()
        server.step(leave, prefixes, pre_k[:n] if n else None, pre_v[:n] if n else None, q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(srv_dec.out[:w.B], out_ref), f"step {s}"
    assert ref.device_errors() == 0 and srv_dec.device_errors() == 0
    assert server.rows().tolist() == ids
    assert torch.equal(srv_dec.k_cache, ref.k_cache) and torch.equal(srv_dec.v_cache, ref.v_cache)
    pos, slots, seq_lens, tables = (np.array(x) for x in ref.last_metadata)
    q64, k64, v64 = (f64(t) for t in (q, k, v))
    got = f64(srv_dec.out[:w.B])
    for b in (0, 1, 100, 255):
        nblk = -(-int(seq_lens[b]) // 16)
        blocks = torch.from_numpy(tables[b, :nblk].astype(np.int64)).to(dv)
        j = int(pos[b]) // 16
        res = decode_step(q64[b:b + 1], k64[b:b + 1], v64[b:b + 1], pos[b:b + 1],
                          [j * 16 + int(slots[b]) % 16], seq_lens[b:b + 1],
                          np.arange(nblk)[None, :], f64(ref.k_cache[blocks]),
                          f64(ref.v_cache[blocks]), scale=w.scale, base=w.rope_base,
                          dtype=w.dtype)
        assert_out_close(got[b], res["out"][0], w.dtype, f"row {b}")
    server.close()
