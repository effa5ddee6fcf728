"""The attention call that allocates nothing (pkv_decode_attn_static).

Some callers cannot allocate device memory at all -- code that runs under
another runtime's memory manager, plugins that are handed only their input and
output tensors, paths that must never reach an allocator -- so they cannot
provide the workspace pkv_decode_attn_split needs.  pkv_decode_attn_static takes
its scratch from an array compiled into the library instead.  These tests call
it through the C ABI and compare it with the workspace call and with the float64
oracle.  This file is collected last so that a run stopping at the first failure
has already run every other test; it also passes when run alone in a fresh
process.
"""
import pytest
import torch

from helpers import TOL, assert_out_close, dev, f64, gpu_single_step, oracle_metadata, oracle_rows
from paged_kv_decode_10_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["decode16", "ragged64", "tiny"])
def test_static_scratch_matches_workspace_call_twice(name):
    w = workloads.make_workload(name)
    res = gpu_single_step(w)                 # step through the workspace path
    dec = res["decoder"]
    B = w.B
    ref = torch.empty_like(dec.out[:B])
    binding.decode_attention(dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables,
                             dec.seq_lens, dec.scale, num_parts=dec.num_parts, out=ref)
    torch.cuda.synchronize()
    assert torch.equal(ref.cpu(), res["out"])
    for _ in range(2):                       # two calls in a row share the array
        out = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device=dev())
        binding.decode_attention_static(dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables,
                                        dec.seq_lens, dec.scale, out,
                                        num_parts=dec.num_parts, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        diff = (out.double() - ref.double()).abs().max().item()
        assert diff <= TOL[w.dtype], diff


@pytest.mark.parametrize("name", ["decode16", "tiny"])
def test_static_scratch_matches_the_oracle(name):
    """Every row of the call without a workspace against the float64 oracle, at
    the same tolerances as the workspace path (1e-5 float32, 2e-2 bf16)."""
    w = workloads.make_workload(name)
    res = gpu_single_step(w)
    dec = res["decoder"]
    B = w.B
    out = torch.full_like(dec.out[:B], float("nan"))
    binding.decode_attention_static(dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables,
                                    dec.seq_lens, dec.scale, out, err=dec.err)
    torch.cuda.synchronize()
    assert dec.device_errors() == 0
    caches = workloads.make_caches(w, "cpu")
    tokens = workloads.make_new_tokens(w, 0, "cpu")
    ref = oracle_rows(w, caches, tokens, oracle_metadata(w), range(B))
    got = f64(out)
    for b in range(B):
        assert_out_close(got[b], ref[b]["out"], w.dtype, f"row {b}")


@pytest.mark.parametrize("name,hq,hkv", [("g8", 32, 4), ("g2", 16, 8), ("g1", 8, 8)])
def test_static_default_partition_equals_workspace_default(name, hq, hkv):
    """Left at its default, the call without a workspace picks the same
    partition as pkv_decode_attn_split for the same group size, so the two give
    bit-identical outputs (float32 runs on the CUDA-core consumer, whose
    variants differ by group size)."""
    w = workloads.custom_workload(name, [5, 300, 17, 1200, 0, 64], hq, hkv, 64, "f32", seed=31)
    res = gpu_single_step(w)
    dec = res["decoder"]
    B = w.B
    ref = binding.decode_attention(dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables,
                                   dec.seq_lens, dec.scale)
    out = torch.empty_like(ref)
    binding.decode_attention_static(dec.q_rot[:B], dec.k_cache, dec.v_cache, dec.tables,
                                    dec.seq_lens, dec.scale, out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


def test_static_scratch_alternating_shapes():
    """A call with another layout in between must not leave stale counters."""
    for name in ["decode16", "tiny", "decode16"]:
        w = workloads.make_workload(name)
        res = gpu_single_step(w)
        dec = res["decoder"]
        out = torch.empty_like(dec.out[:w.B])
        binding.decode_attention_static(dec.q_rot[:w.B], dec.k_cache, dec.v_cache, dec.tables,
                                        dec.seq_lens, dec.scale, out)
        torch.cuda.synchronize()
        diff = (out.double().cpu() - res["out"].double()).abs().max().item()
        assert diff <= TOL[w.dtype], (name, diff)


def test_static_scratch_rejects_oversized_calls():
    w = workloads.custom_workload("big", [16] * 4096, 32, 8, 128, "bf16", seed=3)
    d = dev()
    q = torch.zeros(w.B, w.Hq, w.d, dtype=torch.bfloat16, device=d)
    cache = torch.zeros(8, w.Hkv, 16, w.d, dtype=torch.bfloat16, device=d)
    tables = torch.zeros(w.B, 2, dtype=torch.int32, device=d)
    lens = torch.full((w.B,), 17, dtype=torch.int32, device=d)
    with pytest.raises(binding.PkvError) as e:
        binding.decode_attention_static(q, cache, cache, tables, lens, 0.1, torch.empty_like(q))
    assert e.value.code == binding.ERR_UNSUPPORTED
