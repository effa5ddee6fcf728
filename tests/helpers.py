"""Shared drivers for the GPU parity tests: run a step through the C ABI and
compute the same step with the float64 oracle on the same seeded inputs."""
import numpy as np
import torch

from oracle.allocator import BlockAllocatorModel
from oracle.step import decode_step
from paged_kv_decode_10_gb300 import engine, workloads

TOL = {"f32": 1e-5, "bf16": 2e-2}


def dev():
    return torch.device("cuda:0")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def storage_spacing(x, dtype):
    """Spacing of representable values of ``dtype`` at |x| (one ulp)."""
    x = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(np.where(x == 0, 1e-30, x))
    bits = 8 if dtype == "bf16" else 24
    return np.ldexp(1.0, np.maximum(e - 1, -126) - (bits - 1))


def gpu_single_step(w, num_parts=None, flags=0, caches=None, tokens=None, bt=None,
                    metadata="copy"):
    """One decode step of workload ``w`` on the GPU; every row joins with its
    cached length and is stepped once.  Returns host copies of everything."""
    d = dev()
    if caches is None:
        caches = workloads.make_caches(w, "cpu")
    if tokens is None:
        tokens = workloads.make_new_tokens(w, 0, "cpu")
    k_cache, v_cache = caches
    q, k, v = tokens
    bt = bt or w.max_blocks_per_seq()
    dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                              initial_free=w.free_order, device=d, num_parts=num_parts,
                              flags=flags, k_cache=k_cache.to(d), v_cache=v_cache.to(d),
                              metadata=metadata)
    ids = [dec.join(int(L)) for L in w.seq_lens]
    out = dec.step(ids, q.to(d), k.to(d), v.to(d))
    torch.cuda.synchronize()
    meta = [np.array(x) for x in dec.last_metadata]
    res = dict(out=out.cpu(), q_rot=dec.q_rot[:w.B].cpu(), k_rot=dec.k_rot[:w.B].cpu(),
               k_cache=dec.k_cache.cpu(), v_cache=dec.v_cache.cpu(), meta=meta,
               err=dec.device_errors(), decoder=dec)
    return res


def oracle_metadata(w, bt=None):
    bt = bt or w.max_blocks_per_seq()
    model = BlockAllocatorModel(w.num_blocks, max_seqs=w.B, max_blocks_per_seq=bt,
                                initial_free=w.free_order)
    ids = [model.join(int(L)) for L in w.seq_lens]
    return model.prepare_step(ids, bt)


def oracle_rows(w, caches, tokens, meta, rows):
    """Oracle step restricted to ``rows``: each row is computed alone over a
    private copy of just its own blocks (rows never share blocks)."""
    k_cache, v_cache = caches
    q, k, v = (f64(t) for t in tokens)
    pos, slots, lens, tables = meta
    res = {}
    for b in rows:
        n = -(-int(lens[b]) // 16)
        blocks = tables[b, :n].astype(np.int64)
        kc = f64(k_cache[torch.from_numpy(blocks)])
        vc = f64(v_cache[torch.from_numpy(blocks)])
        j = int(pos[b]) // 16
        assert blocks[j] == slots[b] // 16
        mini_slot = j * 16 + int(slots[b]) % 16
        r = decode_step(q[b:b + 1], k[b:b + 1], v[b:b + 1], pos[b:b + 1], [mini_slot],
                        lens[b:b + 1], np.arange(n)[None, :], kc, vc, scale=w.scale,
                        base=w.rope_base, dtype=w.dtype)
        res[b] = dict(out=r["out"][0], q_rot=r["q_rot"][0], k_rot=r["k_rot"][0])
    return res


def assert_rope_close(gpu, ref, dtype):
    gpu = np.asarray(gpu, np.float64)
    tol = storage_spacing(ref, dtype) + (1e-6 if dtype == "bf16" else 2e-6)
    bad = np.abs(gpu - ref) > tol
    assert not bad.any(), f"rope mismatch at {np.argwhere(bad)[:5]}: {gpu[bad][:5]} vs {ref[bad][:5]}"


def assert_out_close(gpu, ref, dtype, what=""):
    err = np.abs(np.asarray(gpu, np.float64) - ref).max()
    assert err <= TOL[dtype], f"{what} max |gpu - oracle| = {err} > {TOL[dtype]}"
    return err
