"""Seeded synthetic workloads for the decode step.

This module only draws inputs: shapes, lengths, pool sizes, the allocator's
initial free order, the churn plan and N(0,1) tensors.  It holds none of the
step's arithmetic (no RoPE, no slot or block-table computation, no attention),
so the CUDA path and the float64 oracle can both be fed from it without sharing
any of the method.

Workloads (lengths are the cached length ``L`` of each row *before* the step;
the step appends one token, so attention reads ``L + 1`` tokens):

``tiny``      B=3, L={5,17,33}, 4 query / 2 KV heads, d=64, float32, a 16-block
              pool whose free order is a seeded permutation.  Also used with a
              right-padded + masked layout.
``decode16``  B=16, L ~ U[128, 2048], 32/8 heads, d=64, bf16.
``ragged64``  B=64, L ~ U[1, 4096], 32/8 heads, d=128, bf16 (long-tail ragged).
``churn256``  B=256, L ~ lognormal(median 2048, sigma 0.5) clipped to
              [512, 8192], 32/8 heads, d=128, bf16; 64 lockstep steps, each
              preceded by 26 rows (10 %) leaving and 26 joining with a prefix
              ~ U[256, 1024].
``long131k``  B=1, L=131072, 32/4 heads, d=128, bf16.

Every non-tiny pool holds ``ceil(1.25 * sum_b ceil((L_b + 1) / 16))`` blocks,
scattered by a seeded permutation of the free list.  Seeds: tiny 0, decode16 1,
ragged64 2, churn256 3, long131k 4.
"""
from dataclasses import dataclass, field
import math

import numpy as np

BLOCK_SIZE = 16


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    dtype: str                      # "f32" or "bf16"
    seq_lens: np.ndarray            # cached length per row before the step
    num_blocks: int
    free_order: np.ndarray          # initial free stack, bottom -> top
    seed: int
    rope_base: float = 10000.0
    steps: int = 1
    churn: list = field(default_factory=list)   # per step: (leave_rows, join_prefixes)

    @property
    def group(self):
        return self.Hq // self.Hkv

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)

    def max_blocks_per_seq(self, extra_tokens=0):
        longest = int(self.seq_lens.max()) + 1 + extra_tokens
        return -(-longest // BLOCK_SIZE)


def _pool_blocks(lens, factor=1.25):
    blocks = sum(-(-(int(x) + 1) // BLOCK_SIZE) for x in lens)
    return int(math.ceil(factor * blocks))


def make_workload(name, seed=None):
    """Build the named workload (see the module docstring)."""
    if name == "tiny":
        seed = 0 if seed is None else seed
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = np.array([5, 17, 33], np.int64)
        nb = 16
        return Workload("tiny", 3, 4, 2, 64, "f32", lens, nb,
                        rng.permutation(nb).astype(np.int32), seed)
    if name == "decode16":
        seed = 1 if seed is None else seed
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = rng.integers(128, 2048, size=16, endpoint=True)
        nb = _pool_blocks(lens)
        return Workload("decode16", 16, 32, 8, 64, "bf16", lens, nb,
                        rng.permutation(nb).astype(np.int32), seed)
    if name == "ragged64":
        seed = 2 if seed is None else seed
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = rng.integers(1, 4096, size=64, endpoint=True)
        nb = _pool_blocks(lens)
        return Workload("ragged64", 64, 32, 8, 128, "bf16", lens, nb,
                        rng.permutation(nb).astype(np.int32), seed)
    if name == "churn256":
        seed = 3 if seed is None else seed
        rng = np.random.Generator(np.random.PCG64(seed))
        B, steps, sigma = 256, 64, 0.5
        raw = np.exp(rng.normal(math.log(2048.0), sigma, size=B))
        lens = np.clip(np.rint(raw), 512, 8192).astype(np.int64)
        nb = _pool_blocks(lens)
        n_move = int(round(0.1 * B))
        churn = []
        for _ in range(steps):
            leave = np.sort(rng.choice(B, size=n_move, replace=False))
            prefixes = rng.integers(256, 1024, size=n_move, endpoint=True)
            churn.append((leave.astype(np.int64), prefixes.astype(np.int64)))
        return Workload("churn256", B, 32, 8, 128, "bf16", lens, nb,
                        rng.permutation(nb).astype(np.int32), seed,
                        steps=steps, churn=churn)
    if name == "long131k":
        seed = 4 if seed is None else seed
        rng = np.random.Generator(np.random.PCG64(seed))
        lens = np.array([131072], np.int64)
        nb = _pool_blocks(lens)
        return Workload("long131k", 1, 32, 4, 128, "bf16", lens, nb,
                        rng.permutation(nb).astype(np.int32), seed)
    raise KeyError(name)


WORKLOAD_NAMES = ("tiny", "decode16", "ragged64", "churn256", "long131k")


def custom_workload(name, lens, Hq, Hkv, d, dtype, seed, pool_factor=1.25,
                    num_blocks=None):
    """A workload with explicit lengths (used by tests for edge cases)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lens = np.asarray(lens, np.int64)
    nb = num_blocks if num_blocks is not None else max(_pool_blocks(lens, pool_factor), 1)
    return Workload(name, len(lens), Hq, Hkv, d, dtype, lens, nb,
                    rng.permutation(nb).astype(np.int32), seed)


def torch_dtype(dtype):
    import torch
    return {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]


def normal(shape, dtype, seed, device="cpu"):
    """N(0,1) draws in float32 from a seeded torch generator, rounded to ``dtype``."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=device)
    return x.to(torch_dtype(dtype))


def make_caches(w, device="cpu", chunk_blocks=4096):
    """K and V pools ``[num_blocks, Hkv, 16, d]`` filled with N(0,1)."""
    import torch
    shape = (w.num_blocks, w.Hkv, BLOCK_SIZE, w.d)
    caches = []
    for which in (0, 1):
        t = torch.empty(shape, dtype=torch_dtype(w.dtype), device=device)
        gen = torch.Generator(device=device)
        gen.manual_seed(int(w.seed) * 7919 + 101 + which)
        for s in range(0, w.num_blocks, chunk_blocks):
            e = min(w.num_blocks, s + chunk_blocks)
            t[s:e] = torch.randn((e - s,) + shape[1:], generator=gen,
                                 dtype=torch.float32, device=device).to(t.dtype)
        caches.append(t)
    return caches[0], caches[1]


def make_new_tokens(w, step=0, device="cpu"):
    """New ``q [B,Hq,d]``, ``k [B,Hkv,d]``, ``v [B,Hkv,d]`` for one step."""
    base = int(w.seed) * 1_000_003 + 17 * int(step)
    q = normal((w.B, w.Hq, w.d), w.dtype, base + 1, device)
    k = normal((w.B, w.Hkv, w.d), w.dtype, base + 2, device)
    v = normal((w.B, w.Hkv, w.d), w.dtype, base + 3, device)
    return q, k, v
