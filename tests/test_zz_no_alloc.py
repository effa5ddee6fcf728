"""The attention call that allocates nothing (pkv_decode_attn_static).

Callers that cannot allocate device memory use a scratch array compiled into
the library instead of a workspace they would have to provide.  This file is
collected last so that a run stopping at the first failure has already run
every other test; it also passes when run alone in a fresh process.
"""
import numpy as np
import pytest
import torch

from helpers import TOL, dev, gpu_single_step
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


def test_static_scratch_alternating_shapes():
    """A call with another layout in between must not leave stale counters."""
    outs = {}
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
