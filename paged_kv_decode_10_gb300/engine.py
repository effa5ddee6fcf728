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

With ``n_layers > 1`` every layer has its own K/V pool ("neurogrid releases"
v0.7.0: per-layer caches) indexed by the same block tables; a step runs the
layers in order through ``pkv_decode_step_layers`` (each layer's kernels
overlap the previous layer's tail) and one graph holds all of them.  When a
step has long units (``long_units``) the layers are launched with
PKV_LAYERS_MERGE_HELPERS, so that their merges are shared as in a one-layer
step (``layer_merge_helpers`` forces either choice).  ``pool_blocks_for_vram`` sizes the pool from the free device memory (v0.7.0
sizes it from a quarter of the free VRAM).

Joins and leaves only edit the allocator's block tables ("neurogrid releases"
v0.7.0: blocks taken on demand, constant-time allocation and release); no KV
is moved when the batch
changes, which is what replaces the extract/re-assemble rebatch of the helexa
continuous-batching PR.
"""
import math

import numpy as np

from . import binding


def pool_blocks_for_vram(n_layers, Hkv, d, dtype, fraction=0.25, device=None):
    """Blocks that fit in ``fraction`` of the device's free memory, for K and V
    pools of ``n_layers`` layers."""
    import torch
    free, _ = torch.cuda.mem_get_info(device)
    code = binding.F32 if dtype == "f32" else binding.BF16
    return binding.pool_blocks(int(free * fraction), n_layers, Hkv, d, code)


def _metadata_layout(B, bt_stride, plan_parts=0):
    """Byte offsets of slot_mapping (int64), positions, seq_lens, block tables
    (int32) and the partition plan (int32 [plan_parts, PLAN_INTS], 16-byte
    aligned) in one packed buffer for batch size B, and its size."""
    slots = 0
    pos = 8 * B
    lens = pos + 4 * B
    tables = (lens + 4 * B + 15) // 16 * 16
    plan = (tables + 4 * B * bt_stride + 15) // 16 * 16
    return slots, pos, lens, tables, plan, plan + 4 * binding.PLAN_INTS * plan_parts


def long_units(seq_lens, Hkv, d, num_parts, min_parts=8):
    """Whether some (row, KV head) unit of a step with these lengths (after the
    append) spans at least ``min_parts`` parts of the attention partition (a
    unit of n pages when n * num_parts >= min_parts * P, P the position count:
    pages plus the boundary cost of 4 pages at d = 64 and 2 at d = 128 per
    unit).  Such units are merged by helpers in a single-layer call; in a layer
    chain that takes PKV_LAYERS_MERGE_HELPERS."""
    pages = (np.asarray(seq_lens, np.int64) + binding.BLOCK_SIZE - 1) // binding.BLOCK_SIZE
    A = 4 if d <= 64 else 2
    P = Hkv * int(np.sum(np.where(pages > 0, pages + A, 0)))
    return P > 0 and int(pages.max()) * num_parts >= min_parts * P


class PagedDecoder:
    def __init__(self, num_blocks, Hq, Hkv, d, dtype, max_seqs, max_blocks_per_seq,
                 initial_free=None, device="cuda", num_parts=None, rope_base=10000.0,
                 scale=None, flags=0, k_cache=None, v_cache=None, metadata="copy", n_layers=1,
                 plan=True, layer_merge_helpers=None):
        import torch
        if metadata not in ("copy", "mapped"):
            raise ValueError(f"metadata must be 'copy' or 'mapped', not {metadata!r}")
        if n_layers < 1:
            raise ValueError("n_layers must be >= 1")
        self.metadata = metadata
        self.n_layers = n_layers
        # a0 also states the attention partition (pkv_plan_parts), so the
        # kernel starts from it instead of scanning every row length first
        self.planned = bool(plan)
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
        # layer chains: PKV_LAYERS_MERGE_HELPERS when the step has long units
        # (None: decided by each prepare_host from the step's lengths, and a
        # captured graph keeps the decision of the last one before capture)
        self.layer_merge_helpers = layer_merge_helpers
        self._helpers_now = bool(layer_merge_helpers)
        L = n_layers
        shape = (L, num_blocks, Hkv, binding.BLOCK_SIZE, d)
        # caches of every layer: [L, num_blocks, Hkv, 16, d]; a single-layer
        # decoder also accepts (and exposes) [num_blocks, Hkv, 16, d]
        if k_cache is not None and k_cache.dim() == 4:
            k_cache, v_cache = k_cache.unsqueeze(0), v_cache.unsqueeze(0)
        self.k_caches = k_cache if k_cache is not None else torch.empty(
            shape, dtype=self.tdtype, device=self.device)
        self.v_caches = v_cache if v_cache is not None else torch.empty(
            shape, dtype=self.tdtype, device=self.device)
        if tuple(self.k_caches.shape) != shape or tuple(self.v_caches.shape) != shape:
            raise ValueError(f"caches must have shape {shape}")
        self.k_cache, self.v_cache = self.k_caches[0], self.v_caches[0]
        self.num_blocks = num_blocks
        self.alloc = binding.BlockAllocator(num_blocks, max_seqs, max_blocks_per_seq,
                                            initial_free)
        code = binding.F32 if dtype == "f32" else binding.BF16
        self.num_parts = num_parts or binding.default_parts(d, code, flags, Hq, Hkv)
        self.workspace = binding.alloc_workspace(max_seqs, Hq, Hkv, d, self.num_parts,
                                                 self.device)
        # consecutive layers alternate between two workspaces
        self.workspace2 = (binding.alloc_workspace(max_seqs, Hq, Hkv, d, self.num_parts,
                                                   self.device) if L > 1 else None)
        dev = dict(device=self.device)
        self._plan_parts = self.num_parts if self.planned else 0
        cap = _metadata_layout(max_seqs, self.bt_stride, self._plan_parts)[-1]
        self._meta_dev = torch.empty(cap if metadata == "copy" else 0, dtype=torch.uint8, **dev)
        # per-layer buffers [L, max_seqs, H, d]; the unsuffixed names are layer 0
        self.q_rots = torch.empty((L, max_seqs, Hq, d), dtype=self.tdtype, **dev)
        self.k_rots = torch.empty((L, max_seqs, Hkv, d), dtype=self.tdtype, **dev)
        self.outs = torch.empty((L, max_seqs, Hq, d), dtype=self.tdtype, **dev)
        self.err = torch.zeros(1, dtype=torch.int32, **dev)
        # fixed input buffers for graph replay (the producer of q/k/v writes here)
        self.q_ins = torch.empty((L, max_seqs, Hq, d), dtype=self.tdtype, **dev)
        self.k_ins = torch.empty((L, max_seqs, Hkv, d), dtype=self.tdtype, **dev)
        self.v_ins = torch.empty((L, max_seqs, Hkv, d), dtype=self.tdtype, **dev)
        self.q_rot, self.k_rot, self.out = self.q_rots[0], self.k_rots[0], self.outs[0]
        self.q_in, self.k_in, self.v_in = self.q_ins[0], self.k_ins[0], self.v_ins[0]
        self._graphs = None
        # two pinned metadata buffers so the host can fill step i+1 while step
        # i's copy (or, mapped, its kernels) still reads the other one
        self._host = [dict(raw=torch.empty(cap, dtype=torch.uint8, pin_memory=True), event=None,
                           runner=None) for _ in range(2)]
        self._turn = 0
        self._pending = None
        self.last_metadata = None
        self._view_cache = {}
        self._meta_cur = self._meta_dev if metadata == "copy" else self._host[0]["raw"]
        self._set_device_views(max_seqs)

    # -- packed metadata views ----------------------------------------------
    def _views(self, raw, B):
        """Typed views of one packed metadata buffer for batch size B (made once
        per buffer and B: the buffers live as long as the decoder)."""
        key = (raw.data_ptr(), B)
        hit = self._view_cache.get(key)
        if hit is not None:
            return hit
        torch = self.torch
        o_slots, o_pos, o_lens, o_tab, o_plan, end = _metadata_layout(B, self.bt_stride,
                                                                      self._plan_parts)
        views = ((raw[o_pos:o_pos + 4 * B].view(torch.int32),
                  raw[o_slots:o_slots + 8 * B].view(torch.int64),
                  raw[o_lens:o_lens + 4 * B].view(torch.int32),
                  raw[o_tab:o_plan].view(torch.int32)[:B * self.bt_stride].view(B, self.bt_stride),
                  raw[o_plan:end].view(torch.int32).view(-1, binding.PLAN_INTS)
                  if self.planned else None), end)
        self._view_cache[key] = views
        return views

    def _set_device_views(self, B):
        """positions/slots/seq_lens/tables: the views the kernels read (device
        tensors, or pinned host tensors when mapped)."""
        (self.positions, self.slots, self.seq_lens, self.tables, self.plan), _ = self._views(
            self._meta_cur, B)

    # -- batch membership ----------------------------------------------------
    def join(self, prefix_len):
        return self.alloc.join(prefix_len)

    def leave(self, seq_id):
        self.alloc.leave(seq_id)

    # -- a0 ----------------------------------------------------------------
    def wait_host_buffer(self):
        """Blocks until the GPU no longer reads the pinned metadata buffer that
        the next ``prepare_host`` fills (the step two launches back)."""
        h = self._host[self._turn]
        if h["event"] is not None:
            h["event"].synchronize()
            h["event"] = None

    def prepare_host(self, seq_ids):
        """a0 into the pinned buffer that the next copy (or replay) reads."""
        self.wait_host_buffer()
        h = self._host[self._turn]
        B = len(seq_ids)
        run = h["runner"]
        if run is None or run[0] != B:
            views, _ = self._views(h["raw"], B)
            npv = tuple(t.numpy() for t in views[:4])
            ids = np.empty(B, np.int32)
            planner = None
            if self.planned:
                planner = binding.plan_runner(npv[2], npv[3], self.Hkv, self.d, self.num_parts,
                                              views[4].numpy())
            run = h["runner"] = (B, ids, npv, self.alloc.step_runner(ids, self.bt_stride, npv),
                                 planner)
        _, ids, npv, fn, planner = run
        ids[:] = seq_ids
        fn()
        if planner is not None:
            planner()
        if self.n_layers > 1 and self.layer_merge_helpers is None:
            self._helpers_now = long_units(npv[2], self.Hkv, self.d, self.num_parts)
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
        nbytes = _metadata_layout(B, self.bt_stride, self._plan_parts)[-1]
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            self._meta_dev[:nbytes].copy_(h["raw"][:nbytes], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s)
        h["event"] = ev
        self._set_device_views(B)
        return npv

    # -- a1..a4 --------------------------------------------------------------
    def step_args(self, B, q, k, v, attn_bias=None, layer=0, out=None):
        self._set_device_views(B)
        ws = self.workspace if layer % 2 == 0 else self.workspace2
        return binding.make_step_args(
            q, k, v, self.q_rots[layer, :B], self.k_rots[layer, :B], self.k_caches[layer],
            self.v_caches[layer], self.positions, self.slots, self.seq_lens, self.tables,
            self.scale, self.rope_base, self.num_parts, ws,
            self.outs[layer, :B] if out is None else out, attn_bias, self._step_flags(), self.err,
            plan=self.plan)

    def _step_flags(self):
        if self.n_layers > 1 and self._helpers_now:
            return self.flags | binding.LAYERS_MERGE_HELPERS
        return self.flags

    def layer_args(self, B, q, k, v, attn_bias=None):
        """``StepArgs`` of every layer (``q [L,B,Hq,d]``, ``k, v [L,B,Hkv,d]``)."""
        return binding.layer_args_array(
            [self.step_args(B, q[l], k[l], v[l], attn_bias, l) for l in range(self.n_layers)])

    def _launch(self, B, q, k, v, attn_bias, stream):
        if self.n_layers == 1:
            if q.dim() == 4:
                q, k, v = q[0], k[0], v[0]
            binding.decode_step_args(self.step_args(B, q, k, v, attn_bias), stream)
        else:
            binding.decode_step_layers(self.layer_args(B, q, k, v, attn_bias), stream)

    def step(self, seq_ids, q, k, v, attn_bias=None, stream=None):
        """One decode step for the listed sequences; returns ``out[:B]`` (device;
        with several layers, ``outs[:, :B]``).  q/k/v are ``[B,H,d]`` for one
        layer or ``[L,B,H,d]``."""
        torch = self.torch
        B = len(seq_ids)
        self.prepare(seq_ids, stream)
        self._launch(B, q, k, v, attn_bias, stream)
        if self._pending is not None:
            ev = torch.cuda.Event()
            ev.record(stream if stream is not None else torch.cuda.current_stream(self.device))
            self._pending["event"] = ev
            self._pending = None
        return self.out[:B] if self.n_layers == 1 else self.outs[:, :B]

    # -- CUDA graph of the whole device step ("neurogrid releases" v0.8.0) ---
    def capture(self, B, attn_bias=None):
        """Captures, for a fixed batch size B, one CUDA graph per pinned
        metadata buffer: its H2D copy (none when mapped) followed by a1..a4
        reading ``q_in/k_in/v_in[:B]``.  ``replay_step`` then costs one graph
        launch."""
        torch = self.torch
        binding.default_parts(self.d, binding.F32 if self.dtype == "f32" else binding.BF16,
                              self.flags, self.Hq, self.Hkv)   # kernel attributes outside capture
        nbytes = _metadata_layout(B, self.bt_stride, self._plan_parts)[-1]
        stream = torch.cuda.Stream(self.device)
        stream.wait_stream(torch.cuda.current_stream(self.device))
        # a layer chain that picks its merge per step gets both forms, and each
        # replay takes the one its prepare_host chose
        auto = self.n_layers > 1 and self.layer_merge_helpers is None
        decided = self._helpers_now
        graphs, all_args = {}, []
        for helpers in ((False, True) if auto else (decided,)):
            self._helpers_now = helpers
            graphs[helpers] = []
            for h in self._host:
                if self.metadata == "mapped":
                    self._meta_cur = h["raw"]
                if self.n_layers == 1:
                    args = self.step_args(B, self.q_in[:B], self.k_in[:B], self.v_in[:B],
                                          attn_bias)
                else:
                    args = self.layer_args(B, self.q_ins[:, :B], self.k_ins[:, :B],
                                           self.v_ins[:, :B], attn_bias)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    if self.metadata == "copy":
                        self._meta_dev[:nbytes].copy_(h["raw"][:nbytes], non_blocking=True)
                    if self.n_layers == 1:
                        binding.decode_step_args(args, stream)
                    else:
                        binding.decode_step_layers(args, stream)
                graphs[helpers].append(g)
                all_args.append(args)
        self._helpers_now = decided
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
        forms = graphs.get(self._helpers_now)
        (forms if forms is not None else next(iter(graphs.values())))[turn].replay()
        ev = torch.cuda.Event()
        ev.record(torch.cuda.current_stream(self.device))
        self._host[turn]["event"] = ev
        return self.out[:B] if self.n_layers == 1 else self.outs[:, :B]

    # -- end to end from pinned host buffers ------------------------------------
    def capture_host(self, B, attn_bias=None):
        """Captures, for batch size B, one CUDA graph per pinned metadata buffer
        whose kernels read the step's new q/k/v in place from the pinned host
        buffers ``q_host, k_host, v_host`` (over the CPU-GPU link, no staging
        copy) and write the output in place into the pinned ``out_host`` (no
        copy back).  ``host_step`` then costs a0 on the host, one graph launch
        and one wait."""
        torch = self.torch
        if self.n_layers != 1:
            raise ValueError("capture_host is a single-layer step")
        pin = dict(dtype=self.tdtype, pin_memory=True)
        self.q_host = torch.empty((B, self.Hq, self.d), **pin)
        self.k_host = torch.empty((B, self.Hkv, self.d), **pin)
        self.v_host = torch.empty((B, self.Hkv, self.d), **pin)
        self.out_host = torch.empty((B, self.Hq, self.d), **pin)
        binding.default_parts(self.d, binding.F32 if self.dtype == "f32" else binding.BF16,
                              self.flags, self.Hq, self.Hkv)   # kernel attributes outside capture
        nbytes = _metadata_layout(B, self.bt_stride, self._plan_parts)[-1]
        stream = torch.cuda.Stream(self.device)
        stream.wait_stream(torch.cuda.current_stream(self.device))
        graphs, all_args = [], []
        for h in self._host:
            if self.metadata == "mapped":
                self._meta_cur = h["raw"]
            args = self.step_args(B, self.q_host, self.k_host, self.v_host, attn_bias,
                                  out=self.out_host)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                if self.metadata == "copy":
                    self._meta_dev[:nbytes].copy_(h["raw"][:nbytes], non_blocking=True)
                binding.decode_step_args(args, stream)
            graphs.append(g)
            all_args.append(args)
        torch.cuda.current_stream(self.device).wait_stream(stream)
        self._host_graphs = (B, graphs, all_args)

    def host_step(self, seq_ids):
        """One step end to end: the caller has written the step's q/k/v into
        ``q_host/k_host/v_host``; runs a0, replays the captured step and waits;
        returns ``out_host`` (pinned host memory)."""
        torch = self.torch
        B, graphs, _ = self._host_graphs
        if len(seq_ids) != B:
            raise ValueError("batch size differs from the captured one")
        self.prepare_host(seq_ids)
        turn = self._turn
        self._turn ^= 1
        if self.metadata == "mapped":
            self._meta_cur = self._host[turn]["raw"]
            self._set_device_views(B)
        graphs[turn].replay()
        ev = torch.cuda.Event()
        ev.record(torch.cuda.current_stream(self.device))
        self._host[turn]["event"] = ev
        ev.synchronize()
        return self.out_host

    def device_errors(self):
        """Reads and clears the device error flag (a D2H copy: not for the hot loop)."""
        val = int(self.err.item())
        self.err.zero_()
        return val
