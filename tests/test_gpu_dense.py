"""The dense right-padded comparator (assemble_batch / extract_row on the GPU)
against the oracle, and its decode steps against the unpadded oracle."""
import numpy as np
import pytest
import torch

from helpers import assert_out_close, dev, f64
from oracle.dense import assemble_batch, extract_row
from oracle.step import decode_step
from paged_kv_decode_10_gb300 import dense, engine, workloads

pytestmark = pytest.mark.gpu


def token_major(x, n=None):
    """[blocks, Hkv, 16, d] -> [blocks*16, Hkv, d] (first n tokens)."""
    t = f64(x).transpose(0, 2, 1, 3).reshape(-1, x.shape[1], x.shape[3])
    return t if n is None else t[:n]


def _snapshots(db, lens, seed):
    g = torch.Generator().manual_seed(seed)
    ks, vs = [], []
    for L in lens:
        k, v = db.new_snapshot(L)
        k.copy_(torch.randn(k.shape, generator=g).to(k.dtype))
        v.copy_(torch.randn(v.shape, generator=g).to(v.dtype))
        ks.append(k)
        vs.append(v)
    return ks, vs


@pytest.mark.parametrize("dtype,d,hkv", [("bf16", 128, 8), ("f32", 64, 2)])
def test_assemble_and_extract_are_exact_copies(dtype, d, hkv):
    lens = [5, 16, 33, 1, 40]
    cap = 64
    db = dense.DenseBatch(4 * hkv, hkv, d, dtype, len(lens), cap, dev())
    ks, vs = _snapshots(db, lens, 1)
    db.k.fill_(7.0)          # stale contents everywhere: assemble must overwrite the gap
    db.v.fill_(7.0)
    db.assemble(ks, vs, lens)
    torch.cuda.synchronize()
    P = max(lens)
    for cache, snaps in ((db.k, ks), (db.v, vs)):
        want = assemble_batch([token_major(s, L) for s, L in zip(snaps, lens)], P, cap)
        got = token_major(cache).reshape(len(lens), cap, hkv, d)
        np.testing.assert_array_equal(got[:, :P], want[:, :P])
    # two lockstep steps, then extract three rows
    g = torch.Generator().manual_seed(2)
    for _ in range(2):
        q = torch.randn((len(lens), 4 * hkv, d), generator=g).to(db.tdtype).to(dev())
        k = torch.randn((len(lens), hkv, d), generator=g).to(db.tdtype).to(dev())
        v = torch.randn((len(lens), hkv, d), generator=g).to(db.tdtype).to(dev())
        db.step(q, k, v)
    rows = [4, 0, 2]
    out_k, out_v = zip(*[db.new_snapshot(lens[r] + 2) for r in rows])
    db.extract(rows, list(out_k), list(out_v))
    torch.cuda.synchronize()
    dk = token_major(db.k).reshape(len(lens), cap, hkv, d)
    dv = token_major(db.v).reshape(len(lens), cap, hkv, d)
    for r, ok, ov in zip(rows, out_k, out_v):
        n = lens[r] + 2
        np.testing.assert_array_equal(token_major(ok, n), extract_row(dk, r, lens[r], P, 2))
        np.testing.assert_array_equal(token_major(ov, n), extract_row(dv, r, lens[r], P, 2))
    assert db.device_errors() == 0


@pytest.mark.parametrize("name", ["tiny", "decode16"])
def test_dense_steps_match_unpadded_oracle(name):
    """Right-padded rows with the gap masked give the unpadded attention (the
    padding is inert: keys are stored post-RoPE at their true positions)."""
    w = workloads.make_workload(name)
    lens = [int(x) for x in w.seq_lens]
    P = max(lens)
    steps = 3
    cap = (P + steps + 15) // 16 * 16
    db = dense.DenseBatch(w.Hq, w.Hkv, w.d, w.dtype, w.B, cap, dev())
    ks, vs = _snapshots(db, lens, 3)
    db.assemble(ks, vs, lens)
    # the oracle keeps each row unpadded in its own contiguous blocks
    nbr = -(-(P + steps) // 16)
    kc = np.zeros((w.B * nbr, w.Hkv, 16, w.d))
    vc = np.zeros_like(kc)
    for b, L in enumerate(lens):
        kt, vt = token_major(ks[b], L), token_major(vs[b], L)
        for t in range(L):
            kc[b * nbr + t // 16, :, t % 16] = kt[t]
            vc[b * nbr + t // 16, :, t % 16] = vt[t]
    tables = np.arange(w.B)[:, None] * nbr + np.arange(nbr)[None, :]
    for s in range(steps):
        q, k, v = workloads.make_new_tokens(w, s, "cpu")
        out = db.step(q.to(dev()), k.to(dev()), v.to(dev())).cpu()
        pos = np.asarray(lens) + s
        slots = tables[np.arange(w.B), pos // 16] * 16 + pos % 16
        ref = decode_step(f64(q), f64(k), f64(v), pos, slots, pos + 1, tables, kc, vc,
                          scale=1.0 / np.sqrt(w.d), base=10000.0, dtype=w.dtype)
        kc, vc = ref["k_cache"], ref["v_cache"]
        assert_out_close(f64(out), ref["out"], w.dtype, f"step {s}")
    assert db.device_errors() == 0


def test_rebatch_round_trip_matches_paged_decoder():
    """Dense lockstep decode, a leave and a join re-batched by extract +
    assemble, then more steps: every output matches the paged decoder that
    only edits block tables."""
    w = workloads.make_workload("decode16")
    lens = [int(x) for x in w.seq_lens]
    D = dev()
    bt = w.max_blocks_per_seq(extra_tokens=600)
    paged = engine.PagedDecoder(w.num_blocks + 64, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                device=D)
    paged.k_cache.zero_()
    paged.v_cache.zero_()
    ids = [paged.join(L) for L in lens]
    cap = (max(lens) + 600 + 15) // 16 * 16
    db = dense.DenseBatch(w.Hq, w.Hkv, w.d, w.dtype, w.B, cap, D)
    ks, vs = _snapshots(db, lens, 5)
    db.assemble(ks, vs, lens)

    def fill_paged(sid, k, v, n):
        """Copy a snapshot's tokens into the paged sequence's blocks."""
        blocks = paged.alloc.seq_blocks(sid)
        for j, blk in enumerate(blocks[:-(-n // 16)]):
            m = min(16, n - 16 * j)
            paged.k_cache[blk, :, :m] = k[j, :, :m]
            paged.v_cache[blk, :, :m] = v[j, :, :m]

    for b in range(w.B):
        fill_paged(ids[b], ks[b], vs[b], lens[b])
    g = torch.Generator().manual_seed(9)

    def tokens():
        return [torch.randn(s, generator=g).to(db.tdtype).to(D)
                for s in ((w.B, w.Hq, w.d), (w.B, w.Hkv, w.d), (w.B, w.Hkv, w.d))]

    def both_step(tag):
        q, k, v = tokens()
        out_d = db.step(q, k, v).clone()
        out_p = paged.step(ids, q, k, v).clone()
        err = (out_d.float() - out_p.float()).abs().max().item()
        assert err <= (1e-5 if w.dtype == "f32" else 2e-2), (tag, err)

    for s in range(3):
        both_step(f"before {s}")
    # row 5 leaves, a new sequence joins in its place: the dense batch is rebuilt
    leave = 5
    survivors = [r for r in range(w.B) if r != leave]
    cur = db.lengths()
    snaps = [db.new_snapshot(cur[r]) for r in survivors]
    db.extract(survivors, [s[0] for s in snaps], [s[1] for s in snaps])
    jk, jv = _snapshots(db, [300], 6)
    new_k = [s[0] for s in snaps]
    new_v = [s[1] for s in snaps]
    new_k.insert(leave, jk[0])
    new_v.insert(leave, jv[0])
    new_lens = [cur[r] for r in survivors]
    new_lens.insert(leave, 300)
    db.assemble(new_k, new_v, new_lens)
    paged.leave(ids[leave])
    ids[leave] = paged.join(300)
    fill_paged(ids[leave], jk[0], jv[0], 300)
    for s in range(3):
        both_step(f"after {s}")
    assert db.device_errors() == 0 and paged.device_errors() == 0
