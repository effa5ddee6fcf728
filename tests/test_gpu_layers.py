"""Multi-layer decode step (per-layer caches under one set of block tables):
layer by layer through pkv_decode_step_layers equals one single-layer step per
layer, and matches the oracle."""
import numpy as np
import pytest
import torch

from helpers import assert_out_close, dev, f64
from oracle.allocator import BlockAllocatorModel
from oracle.step import decode_step
from paged_kv_decode_10_gb300 import binding, engine, workloads

pytestmark = pytest.mark.gpu


def _layer_inputs(w, L, step, device):
    toks = [workloads.make_new_tokens(w, 100 * step + l, "cpu") for l in range(L)]
    return [torch.stack([t[i] for t in toks]).to(device) for i in range(3)]


@pytest.mark.parametrize("name,L,metadata", [("decode16", 3, "mapped"), ("ragged64", 2, "copy")])
def test_layers_equal_single_layer_decoders(name, L, metadata):
    """Every layer's output and caches equal those of a one-layer decoder fed
    the same layer's inputs (eager steps, then graph replays), over steps that
    cross a block boundary."""
    _layers_against_single_layer(workloads.make_workload(name), L, metadata, None, exact=True)


@pytest.mark.parametrize("helpers,exact", [(None, True), (True, True), (False, False)])
def test_layers_with_long_rows(helpers, exact):
    """Rows whose units span many parts (the first over 30 of them).  With
    PKV_LAYERS_MERGE_HELPERS (which the decoder picks itself for such a step,
    or is told to use) each layer's merge is shared by the unit's last parts as
    in a single-layer step: bit-identical.  Without it the last part merges
    alone: the same values up to the grouping of the float32 sums, so within
    the bf16 output tolerance of the single-layer step."""
    w = workloads.custom_workload("longrows", [40000, 300, 5000], 32, 8, 128, "bf16", seed=23)
    _layers_against_single_layer(w, 2, "copy", helpers, exact)


def _layers_against_single_layer(w, L, metadata, helpers, exact):
    d = dev()
    bt = w.max_blocks_per_seq(extra_tokens=32)
    k0, v0 = workloads.make_caches(w, "cpu")
    multi = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                initial_free=w.free_order, device=d, n_layers=L,
                                metadata=metadata, layer_merge_helpers=helpers,
                                k_cache=torch.stack([k0] * L).to(d),
                                v_cache=torch.stack([v0] * L).to(d))
    singles = [engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                                   initial_free=w.free_order, device=d,
                                   k_cache=k0.to(d), v_cache=v0.to(d)) for _ in range(L)]
    ids_m = [multi.join(int(x)) for x in w.seq_lens]
    ids_s = [[s.join(int(x)) for x in w.seq_lens] for s in singles]
    multi.capture(w.B)
    for step in range(4):
        q, k, v = _layer_inputs(w, L, step, d)
        if step < 2:
            out_m = multi.step(ids_m, q, k, v).clone()
        else:
            multi.q_ins[:, :w.B].copy_(q)
            multi.k_ins[:, :w.B].copy_(k)
            multi.v_ins[:, :w.B].copy_(v)
            multi.prepare_host(ids_m)
            out_m = multi.replay_step().clone()
        for l, s in enumerate(singles):
            out_s = s.step(ids_s[l], q[l], k[l], v[l])
            torch.cuda.synchronize()
            if exact:
                assert torch.equal(out_m[l], out_s), (step, l)
            else:
                assert_out_close(f64(out_m[l]), f64(out_s), w.dtype, f"step {step} layer {l}")
    for l, s in enumerate(singles):
        assert torch.equal(multi.k_caches[l], s.k_cache), l
        assert torch.equal(multi.v_caches[l], s.v_cache), l
        assert torch.equal(multi.q_rots[l, :w.B], s.q_rot[:w.B]), l
    assert multi.device_errors() == 0


def test_layers_match_oracle():
    w = workloads.make_workload("tiny")
    L, steps = 3, 3
    d = dev()
    bt = w.max_blocks_per_seq(extra_tokens=16)
    k0, v0 = workloads.make_caches(w, "cpu")
    dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                              initial_free=w.free_order, device=d, n_layers=L,
                              k_cache=torch.stack([k0] * L).to(d),
                              v_cache=torch.stack([v0] * L).to(d))
    model = BlockAllocatorModel(w.num_blocks, max_seqs=w.B, max_blocks_per_seq=bt,
                                initial_free=w.free_order)
    ids = [dec.join(int(x)) for x in w.seq_lens]
    assert ids == [model.join(int(x)) for x in w.seq_lens]
    caches = [(f64(k0), f64(v0)) for _ in range(L)]
    for step in range(steps):
        q, k, v = _layer_inputs(w, L, step, d)
        out = dec.step(ids, q, k, v).cpu()
        meta = model.prepare_step(ids, bt)
        for l in range(L):
            ref = decode_step(f64(q[l]), f64(k[l]), f64(v[l]), *meta, *caches[l],
                              scale=1.0 / np.sqrt(w.d), base=10000.0, dtype=w.dtype)
            caches[l] = (ref["k_cache"], ref["v_cache"])
            assert_out_close(f64(out[l]), ref["out"], w.dtype, f"step {step} layer {l}")
    assert dec.device_errors() == 0


def test_layers_reject_a_shared_workspace():
    w = workloads.make_workload("tiny")
    d = dev()
    dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B,
                              w.max_blocks_per_seq(), initial_free=w.free_order, device=d,
                              n_layers=2)
    ids = [dec.join(int(x)) for x in w.seq_lens]
    dec.prepare(ids)
    q, k, v = _layer_inputs(w, 2, 0, d)
    a0 = dec.step_args(w.B, q[0], k[0], v[0], layer=0)
    a1 = dec.step_args(w.B, q[1], k[1], v[1], layer=0)   # same workspace as layer 0
    with pytest.raises(binding.PkvError):
        binding.decode_step_layers([a0, a1])


def test_pool_auto_sizing_uses_a_quarter_of_free_memory():
    free, _ = torch.cuda.mem_get_info(dev())
    n = engine.pool_blocks_for_vram(32, 8, 128, "bf16", device=dev())
    per_block = 32 * 2 * 8 * 16 * 128 * 2
    assert n == int(free * 0.25) // per_block
    assert n > 0
