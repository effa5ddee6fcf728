"""Model of the host block allocator that feeds each decode step.

Test infrastructure only (see the package docstring).

The neurogrid v0.7.0 release describes a block allocator with constant-time
allocation and release, a block table per sequence and 16-token blocks taken on
demand; the v0.8.0 release computes ``kv_len = position + 1``.  The pages fix no policy
beyond that; the policy below is our plainest reading and is what the C++
allocator must reproduce bit for bit:

* The free list is a stack.  It starts as a caller-given order (bottom to top);
  ``pop`` takes the top, ``push`` puts on top.
* ``join(prefix_len)`` takes the smallest free sequence id and pops
  ``ceil(prefix_len / 16)`` blocks, in table order.
* ``leave(seq_id)`` pushes the sequence's blocks in table order (its last block
  ends on top) and frees the id.
* ``prepare_step(seq_ids)`` appends one token to every listed sequence: the new
  token sits at ``position = L`` (the cached length before the step); when
  ``L % 16 == 0`` a block is popped first; ``slot = table[L // 16] * 16 + L % 16``;
  the length becomes ``L + 1``, which is the ``seq_len`` attention reads.
* A request that needs more blocks than are free fails with ``OutOfBlocks`` and
  changes nothing.
* ``seq_slots(seq_id, start, count)`` names where tokens ``[start, start+count)``
  of a sequence live (position ``p``, slot ``table[p // 16] * 16 + p % 16``);
  this is how a joiner's prefix, whose blocks ``join`` popped, is written (the
  "chunked-prefill" path of helexa issue 121's engine, which our reading
  turns into a cache write of the prefix keys and values).
"""
import numpy as np


class OutOfBlocks(Exception):
    pass


class UnknownSequence(Exception):
    pass


class BlockAllocatorModel:
    def __init__(self, num_blocks, block_size=16, max_seqs=1024,
                 max_blocks_per_seq=1 << 20, initial_free=None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.max_seqs = int(max_seqs)
        self.max_blocks_per_seq = int(max_blocks_per_seq)
        if initial_free is None:
            initial_free = range(self.num_blocks)
        self.free = [int(b) for b in initial_free]      # bottom ... top
        if sorted(self.free) != list(range(self.num_blocks)):
            raise ValueError("initial free order must be a permutation")
        self.tables = {}      # seq_id -> list of block ids
        self.lengths = {}     # seq_id -> cached length

    # -- sequence lifecycle -------------------------------------------------
    def _blocks_for(self, n_tokens):
        return -(-int(n_tokens) // self.block_size)

    def join(self, prefix_len):
        need = self._blocks_for(prefix_len)
        free_ids = [i for i in range(self.max_seqs) if i not in self.tables]
        if not free_ids:
            raise ValueError("no free sequence id")
        if need > self.max_blocks_per_seq:
            raise ValueError("prefix longer than a block table")
        if need > len(self.free):
            raise OutOfBlocks(need)
        sid = free_ids[0]
        self.tables[sid] = [self.free.pop() for _ in range(need)]
        self.lengths[sid] = int(prefix_len)
        return sid

    def leave(self, seq_id):
        if seq_id not in self.tables:
            raise UnknownSequence(seq_id)
        for blk in self.tables.pop(seq_id):
            self.free.append(blk)
        del self.lengths[seq_id]

    # -- one decode step ----------------------------------------------------
    def prepare_step(self, seq_ids, bt_stride):
        """Returns ``positions, slot_mapping, seq_lens, block_tables`` as numpy
        arrays (int32, int64, int32, int32 ``[B, bt_stride]`` padded with -1)."""
        seq_ids = [int(s) for s in seq_ids]
        for s in seq_ids:
            if s not in self.tables:
                raise UnknownSequence(s)
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence may appear once per step")
        need = sum(1 for s in seq_ids if self.lengths[s] % self.block_size == 0)
        if need > len(self.free):
            raise OutOfBlocks(need)
        for s in seq_ids:
            if self._blocks_for(self.lengths[s] + 1) > min(bt_stride,
                                                           self.max_blocks_per_seq):
                raise ValueError("block table too narrow")
        B = len(seq_ids)
        positions = np.zeros(B, np.int32)
        slots = np.zeros(B, np.int64)
        seq_lens = np.zeros(B, np.int32)
        tables = np.full((B, bt_stride), -1, np.int32)
        for b, s in enumerate(seq_ids):
            pos = self.lengths[s]
            if pos % self.block_size == 0:
                self.tables[s].append(self.free.pop())
            blk = self.tables[s][pos // self.block_size]
            positions[b] = pos
            slots[b] = blk * self.block_size + pos % self.block_size
            self.lengths[s] = pos + 1
            seq_lens[b] = pos + 1
            tables[b, :len(self.tables[s])] = self.tables[s]
        return positions, slots, seq_lens, tables

    def seq_slots(self, seq_id, start, count):
        """Positions and slots (int32, int64 numpy arrays) of tokens
        ``[start, start+count)`` of a live sequence; they must lie within its
        length."""
        if seq_id not in self.tables:
            raise UnknownSequence(seq_id)
        if start < 0 or count < 0 or start + count > self.lengths[seq_id]:
            raise ValueError("token range outside the sequence")
        table = self.tables[seq_id]
        positions = np.arange(start, start + count, dtype=np.int32)
        slots = np.array([table[p // self.block_size] * self.block_size + p % self.block_size
                          for p in range(start, start + count)], dtype=np.int64)
        return positions, slots

    # -- inspection ---------------------------------------------------------
    def num_free(self):
        return len(self.free)

    def seq_blocks(self, seq_id):
        return list(self.tables[seq_id])

    def seq_len(self, seq_id):
        return self.lengths[seq_id]
