"""The dense right-padded batch that paging replaces, kept as a comparator.

helexa issue 121 batches decode by right-padding every sequence's KV snapshot
to the batch maximum and concatenating the rows (slice 1, ``assemble_batch``),
masking each row's padding gap with an additive ``-inf`` (``batch_decode_mask``)
and putting the lockstep decode columns after the gap; a join or leave
re-batches by slicing every surviving row back to a contiguous snapshot
(slice 3a, ``extract_row``: prefix plus decode columns, gap dropped) and
assembling again.  Keys are stored post-RoPE, so a token's position stays its
true position whatever column it sits in.

``DenseBatch`` does exactly that on the GPU with this library's kernels: the
two copies are ``pkv_dense_assemble`` / ``pkv_dense_extract`` and a decode step
is ``pkv_decode_step`` over the dense rows viewed as a pool (row b's table is
``b*cap/16 + j``) with the gap masked by ``attn_bias``.  Paging makes both
copies unnecessary and reads no gap.
"""
import math

import numpy as np

from . import binding


def snapshot_blocks(n_tokens):
    return -(-int(n_tokens) // binding.BLOCK_SIZE)


class DenseBatch:
    def __init__(self, Hq, Hkv, d, dtype, max_rows, cap, device="cuda", rope_base=10000.0,
                 scale=None, num_parts=None, flags=0):
        import torch
        if cap % binding.BLOCK_SIZE:
            raise ValueError("cap must be a multiple of 16")
        self.torch = torch
        self.device = torch.device(device)
        self.Hq, self.Hkv, self.d, self.dtype = Hq, Hkv, d, dtype
        self.tdtype = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
        self.cap, self.max_rows = cap, max_rows
        self.rope_base = rope_base
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        self.flags = flags
        dev = dict(device=self.device)
        shape = (max_rows * cap // binding.BLOCK_SIZE, Hkv, binding.BLOCK_SIZE, d)
        self.k = torch.zeros(shape, dtype=self.tdtype, **dev)
        self.v = torch.zeros(shape, dtype=self.tdtype, **dev)
        code = binding.F32 if dtype == "f32" else binding.BF16
        self.num_parts = num_parts or binding.default_parts(d, code, flags, Hq, Hkv)
        self.workspace = binding.alloc_workspace(max_rows, Hq, Hkv, d, self.num_parts, self.device)
        self.q_rot = torch.empty((max_rows, Hq, d), dtype=self.tdtype, **dev)
        self.k_rot = torch.empty((max_rows, Hkv, d), dtype=self.tdtype, **dev)
        self.out = torch.empty((max_rows, Hq, d), dtype=self.tdtype, **dev)
        self.err = torch.zeros(1, dtype=torch.int32, **dev)
        self.B = 0
        self.prefix = []
        self.padded_len = 0
        self.steps = 0

    def new_snapshot(self, n_tokens):
        """Empty K and V snapshot buffers for a sequence of ``n_tokens``."""
        shape = (max(snapshot_blocks(n_tokens), 1), self.Hkv, binding.BLOCK_SIZE, self.d)
        t = self.torch
        return (t.zeros(shape, dtype=self.tdtype, device=self.device),
                t.zeros(shape, dtype=self.tdtype, device=self.device))

    # -- rebatch ---------------------------------------------------------------
    def assemble(self, k_snaps, v_snaps, lens, stream=None):
        """Rows = the snapshots (tokens [0, lens[b])), right-padded to max(lens)."""
        torch = self.torch
        lens = [int(x) for x in lens]
        B = len(lens)
        if B > self.max_rows:
            raise ValueError("more rows than the batch holds")
        padded = max(lens) if lens else 0
        if padded + 1 > self.cap:
            raise ValueError("no room for a decode column")
        binding.dense_assemble(k_snaps, v_snaps, lens, padded, self.k, self.v, self.cap, stream)
        self.B, self.prefix, self.padded_len, self.steps = B, lens, padded, 0
        # the gap mask of every row, valid for all later steps (columns past the
        # current length are never read)
        t = np.arange(self.cap)
        pre = np.asarray(lens)[:, None]
        bias = np.where((t[None, :] >= pre) & (t[None, :] < padded), -np.inf, 0.0)
        self.bias = torch.from_numpy(bias.astype(np.float32)).to(self.device)
        nbr = self.cap // binding.BLOCK_SIZE
        self.tables = torch.from_numpy(
            (np.arange(B)[:, None] * nbr + np.arange(nbr)[None, :]).astype(np.int32)).to(self.device)

    def extract(self, rows, k_snaps, v_snaps, stream=None):
        """Snapshots of the listed rows: prefix plus the decode columns so far."""
        binding.dense_extract(self.k, self.v, self.cap, rows, [self.prefix[r] for r in rows],
                              self.padded_len, self.steps, k_snaps, v_snaps, stream)

    def lengths(self):
        """Current length of every row (prefix plus decode columns)."""
        return [p + self.steps for p in self.prefix]

    # -- one lockstep decode step -------------------------------------------
    def step_metadata(self):
        B, P, s = self.B, self.padded_len, self.steps
        nbr = self.cap // binding.BLOCK_SIZE
        if P + s + 1 > self.cap:
            raise ValueError("dense rows are full")
        col = P + s
        positions = np.asarray(self.prefix, np.int64) + s            # true positions
        slots = (np.arange(B) * nbr + col // 16) * 16 + col % 16
        seq_lens = np.full(B, col + 1, np.int32)
        return positions.astype(np.int32), slots.astype(np.int64), seq_lens

    def step_args(self, q, k, v, stream=None):
        torch = self.torch
        pos, slots, lens = self.step_metadata()
        B = self.B
        dev = self.device
        self._meta = [torch.from_numpy(x).to(dev, non_blocking=False) for x in (pos, slots, lens)]
        return binding.make_step_args(
            q, k, v, self.q_rot[:B], self.k_rot[:B], self.k, self.v, self._meta[0],
            self._meta[1], self._meta[2], self.tables, self.scale, self.rope_base,
            self.num_parts, self.workspace, self.out[:B], self.bias, self.flags, self.err)

    def step(self, q, k, v, stream=None):
        """Rotate and append the new tokens at column padded_len + steps, attend
        over each row's prefix and decode columns; returns ``out[:B]``."""
        binding.decode_step_args(self.step_args(q, k, v, stream), stream)
        self.steps += 1
        return self.out[:self.B]

    def device_errors(self):
        val = int(self.err.item())
        self.err.zero_()
        return val
