"""One continuous-batching decoder over a paged KV pool: the whole step.

``PagedDecoder`` owns the device KV pool, the host block allocator and the
per-step buffers.  ``step`` runs a0 on the host (allocator: positions,
slot_mapping, seq_lens, block tables, written into one pinned buffer), then
a1-a4 through ``pkv_decode_step`` on one CUDA stream.  With
``metadata="copy"`` the pinned buffer is first copied to the device in one
host-to-device copy; with ``metadata="mapped"`` the kernels read it in place
over the CPU-GPU link and the step has no copy at all.  Nothing is copied back
to the host ("neurogrid releases" v0.8.0: position, seq_len and kv_len live in
GPU buffers; no D2H copies).  ``capture``/``replay_step`` put the (copy and)
kernels of a step in one CUDA graph (v0.8.0: the whole decode replayed as one
graph).

Joins and leaves only edit the allocator's block tables ("neurogrid releases"
v0.7.0: on-demand blocks, O(1) alloc/free); no KV is moved when the batch
changes, which is what replaces the extract/re-assemble rebatch of the helexa
continuous-batching PR.
"""
import math

from . import binding


def _metadata_layout(B, bt_stride):
    """Byte offsets of slot_mapping (int64), positions, seq_lens and block tables
    (int32) in one packed buffer for batch size B, and its size."""
    slots = 0
    pos = 8 * B
    lens = pos + 4 * B
    tables = (lens + 4 * B + 15) // 16 * 16
    return slots, pos, lens, tables, tables + 4 * B * bt_stride


class PagedDecoder:
    def __init__(self, num_blocks, Hq, Hkv, d, dtype, max_seqs, max_blocks_per_seq,
                 initial_free=None, device="cuda", num_parts=None, rope_base=10000.0,
                 scale=None, flags=0, k_cache=None, v_cache=None, metadata="copy"):
        import torch
        if metadata not in ("copy", "mapped"):
            raise ValueError(f"metadata must be 'copy' or 'mapped', not {metadata!r}")
        self.metadata = metadata
        self.torch = torch
        self.device = torch.device(device)
        self.Hq, self.Hkv, self.d = Hq, Hkv, d
        self.dtype = dtype
        self.tdtype = {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]
        self.max_seqs = max_seqs
        self.bt_stride = max_blocks_per_seq
        self.rope_base = rope_base
        self.scale = 1.0 / math.sqrt(d) if scale is None else scale
        self.flags = flags
        shape = (num_blocks, Hkv, binding.BLOCK_SIZE, d)
        self.k_cache = k_cache if k_cache is not None else torch.empty(
            shape, dtype=self.tdtype, device=self.device)
        self.v_cache = v_cache if v_cache is not None else torch.empty(
            shape, dtype=self.tdtype, device=self.device)
        self.num_blocks = num_blocks
        self.alloc = binding.BlockAllocator(num_blocks, max_seqs, max_blocks_per_seq,
                                            initial_free)
        code = binding.F32 if dtype == "f32" else binding.BF16
        self.num_parts = num_parts or binding.default_parts(d, code, flags)
        self.workspace = binding.alloc_workspace(max_seqs, Hq, Hkv, d, self.num_parts,
                                                 self.device)
        dev = dict(device=self.device)
        cap = _metadata_layout(max_seqs, self.bt_stride)[-1]
        self._meta_dev = torch.empty(cap if metadata == "copy" else 0, dtype=torch.uint8, **dev)
        self.q_rot = torch.empty((max_seqs, Hq, d), dtype=self.tdtype, **dev)
        self.k_rot = torch.empty((max_seqs, Hkv, d), dtype=self.tdtype, **dev)
        self.out = torch.empty((max_seqs, Hq, d), dtype=self.tdtype, **dev)
        self.err = torch.zeros(1, dtype=torch.int32, **dev)
        # fixed input buffers for graph replay (the producer of q/k/v writes here)
        self.q_in = torch.empty((max_seqs, Hq, d), dtype=self.tdtype, **dev)
        self.k_in = torch.empty((max_seqs, Hkv, d), dtype=self.tdtype, **dev)
        self.v_in = torch.empty((max_seqs, Hkv, d), dtype=self.tdtype, **dev)
        self._graphs = None
        # two pinned metadata buffers so the host can fill step i+1 while step
        # i's copy (or, mapped, its kernels) still reads the other one
        self._host = [dict(raw=torch.empty(cap, dtype=torch.uint8, pin_memory=True), event=None)
                      for _ in range(2)]
        self._turn = 0
        self._pending = None
        self.last_metadata = None
        self._meta_cur = self._meta_dev if metadata == "copy" else self._host[0]["raw"]
        self._set_device_views(max_seqs)

    # -- packed metadata views ----------------------------------------------
    def _views(self, raw, B):
        torch = self.torch
        o_slots, o_pos, o_lens, o_tab, end = _metadata_layout(B, self.bt_stride)
        return (raw[o_pos:o_pos + 4 * B].view(torch.int32),
                raw[o_slots:o_slots + 8 * B].view(torch.int64),
                raw[o_lens:o_lens + 4 * B].view(torch.int32),
                raw[o_tab:end].view(torch.int32).view(B, self.bt_stride)), end

    def _set_device_views(self, B):
        """positions/slots/seq_lens/tables: the views the kernels read (device
        tensors, or pinned host tensors when mapped)."""
        (self.positions, self.slots, self.seq_lens, self.tables), _ = self._views(
            self._meta_cur, B)

    # -- batch membership ----------------------------------------------------
    def join(self, prefix_len):
        return self.alloc.join(prefix_len)

    def leave(self, seq_id):
        self.alloc.leave(seq_id)

    # -- a0 ----------------------------------------------------------------
    def prepare_host(self, seq_ids):
        """a0 into the pinned buffer that the next copy (or replay) reads."""
        h = self._host[self._turn]
        if h["event"] is not None:
            h["event"].synchronize()
        B = len(seq_ids)
        views, _ = self._views(h["raw"], B)
        npv = tuple(t.numpy() for t in views)
        self.alloc.prepare_step(seq_ids, self.bt_stride, out=npv)
        self.last_metadata = npv
        return npv

    def prepare(self, seq_ids, stream=None):
        """Host allocator step + one async H2D copy of the packed metadata (mapped:
        the kernels of the next ``step_args`` read the pinned buffer itself)."""
        torch = self.torch
        B = len(seq_ids)
        npv = self.prepare_host(seq_ids)
        h = self._host[self._turn]
        self._turn ^= 1
        if self.metadata == "mapped":
            self._meta_cur = h["raw"]
            self._pending = h   # released by the event recorded after the kernels
            self._set_device_views(B)
            return npv
        nbytes = _metadata_layout(B, self.bt_stride)[-1]
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            self._meta_dev[:nbytes].copy_(h["raw"][:nbytes], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s)
        h["event"] = ev
        self._set_device_views(B)
        return npv

    # -- a1..a4 --------------------------------------------------------------
    def step_args(self, B, q, k, v, attn_bias=None):
        self._set_device_views(B)
        return binding.make_step_args(
            q, k, v, self.q_rot[:B], self.k_rot[:B], self.k_cache, self.v_cache,
            self.positions, self.slots, self.seq_lens, self.tables,
            self.scale, self.rope_base, self.num_parts, self.workspace, self.out[:B],
            attn_bias, self.flags, self.err)

    def step(self, seq_ids, q, k, v, attn_bias=None, stream=None):
        """One decode step for the listed sequences; returns ``out[:B]`` (device)."""
        torch = self.torch
        B = len(seq_ids)
        self.prepare(seq_ids, stream)
        binding.decode_step_args(self.step_args(B, q, k, v, attn_bias), stream)
        if self._pending is not None:
            ev = torch.cuda.Event()
            ev.record(stream if stream is not None else torch.cuda.current_stream(self.device))
            self._pending["event"] = ev
            self._pending = None
        return self.out[:B]

    # -- CUDA graph of the whole device step ("neurogrid releases" v0.8.0) ---
    def capture(self, B, attn_bias=None):
        """Captures, for a fixed batch size B, one CUDA graph per pinned
        metadata buffer: its H2D copy (none when mapped) followed by a1..a4
        reading ``q_in/k_in/v_in[:B]``.  ``replay_step`` then costs one graph
        launch."""
        torch = self.torch
        binding.default_parts(self.d, binding.F32 if self.dtype == "f32" else binding.BF16,
                              self.flags)   # sets kernel attributes outside capture
        nbytes = _metadata_layout(B, self.bt_stride)[-1]
        stream = torch.cuda.Stream(self.device)
        stream.wait_stream(torch.cuda.current_stream(self.device))
        graphs, all_args = [], []
        for h in self._host:
            if self.metadata == "mapped":
                self._meta_cur = h["raw"]
            args = self.step_args(B, self.q_in[:B], self.k_in[:B], self.v_in[:B], attn_bias)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                if self.metadata == "copy":
                    self._meta_dev[:nbytes].copy_(h["raw"][:nbytes], non_blocking=True)
                binding.decode_step_args(args, stream)
            graphs.append(g)
            all_args.append(args)
        torch.cuda.current_stream(self.device).wait_stream(stream)
        self._graphs = (B, graphs, all_args)

    def replay_step(self):
        """Launches the captured step for the metadata of the last prepare_host."""
        torch = self.torch
        B, graphs, _ = self._graphs
        turn = self._turn
        self._turn ^= 1
        if self.metadata == "mapped":
            self._meta_cur = self._host[turn]["raw"]
            self._set_device_views(B)
        graphs[turn].replay()
        ev = torch.cuda.Event()
        ev.record(torch.cuda.current_stream(self.device))
        self._host[turn]["event"] = ev
        return self.out[:B]

    def device_errors(self):
        """Reads and clears the device error flag (a D2H copy: not for the hot loop)."""
        val = int(self.err.item())
        self.err.zero_()
        return val
