"""Benchmark of the continuous-batching decode step over a paged KV cache.

One step = a0 host allocator (positions, slots, seq_lens, block tables, into a
pinned buffer the kernels read in place; ``--metadata copy`` adds an H2D copy
instead) + a1 RoPE + a2 append + a3 split-KV paged attention with a4 (LSE
merge) fused into its epilogue, for every row of the workload, replayed as one
CUDA graph.  Steps are consecutive decode steps (every row grows by one token
per step); churn workloads also move rows out and in between steps.

Default workload: ``churn256`` (B=256, L ~ lognormal(median 2048, sigma 0.5)
clipped to [512, 8192], 32 query / 8 KV heads, d=128, bf16; before every step
26 rows leave and 26 join with prefixes of 256-1024 tokens, whose KV the
prefill kernel writes).  A step reads ~2.4 GB of KV, far more than L2; a
buffer of 4x the L2 size is still read before every timed step (evicting the
KV without dirty write-backs) and only the step itself sits between the CUDA
events.  ``--workload decode16`` (or any other workload name) selects another.

Printed JSON line (rank 0):
  value            whole-job throughput: algorithmic attention bytes of all
                   steps / device time of all steps, GB/s
  steps_per_s      decode steps per second (device time)
  roofline         the attention kernel (a3 + fused a4) timed alone with every
                   input in HBM (the step's block tables, lengths and plan
                   copied to the device): algorithmic bytes per launch / mean
                   launch time against the measured HBM copy peak, with the ncu
                   DRAM bytes of the same kernel source
                   (``profiles/traffic.json``).  Launches that read more than
                   L2 holds are not flushed (a GPU sleep before each keeps the
                   GPU busy while the host enqueues; ``l2`` says which), and
                   ``flushed_launch_us`` gives the same launches after a flush
  rooflines        the same for the workloads named by ``--also`` (default
                   ragged64 and long131k), each set up and timed in this run
  layered          whole L-layer steps (``--layered``, default decode16 x 8,
                   ragged64 x 4, long131k x 4): one graph per step, per-layer time
                   and the layers' attention GB/s
  step_kernels_us  the step's kernels (RoPE/append + attention) without the host
  host_a0_us_per_step  the host allocator per step
  e2e              the same metric through the C ABI's captured host step
                   (a0, inputs read and output written in place in pinned host
                   memory, stream wait), wall clock: for launches that read
                   more than L2, pipelined (a0 of the next step on the host
                   while the GPU runs this one, two buffer sets), with the
                   sequential, flushed loop beside it; otherwise the reverse
  cpu_baseline     the float64 oracle on this host's cores, wall clock, over a
                   sample of the final step's (row, KV head) units
  clocks           nvidia-smi SM clock samples taken inside the timed regions
  prefill, churn_wall_clock  (churn workloads) the joiners' prefix KV writes,
                   and one pass over the churn plan timed by the wall clock
  dense_comparator (``--comparator``) the right-padded batch paging replaces

``--impl reference`` times the float64 oracle (the only reference this method
has) on the host cores for the same workload and metric.
"""
import argparse
import ctypes
import gc
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal (context beside the measured peak)
KERNEL_SOURCES = ["paged_kv_decode_10_gb300/csrc/attention_kernel.cuh",
                  "paged_kv_decode_10_gb300/csrc/attention_mma.cu",
                  "paged_kv_decode_10_gb300/csrc/attention_simt_bf16.cu",
                  "paged_kv_decode_10_gb300/csrc/attention_simt_f32.cu",
                  "paged_kv_decode_10_gb300/csrc/attention.cu",
                  "paged_kv_decode_10_gb300/csrc/common.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="churn256")
    ap.add_argument("--also", default="ragged64,long131k",
                    help="other workloads whose attention kernel is timed alone in the same "
                         "run (comma-separated; empty for none)")
    ap.add_argument("--layered", default="decode16:8,ragged64:4,long131k:4",
                    help="workload:L pairs whose whole L-layer step (one graph, each layer's "
                         "kernels overlapping the previous layer's tail) is timed in the same "
                         "run (comma-separated; empty for none)")
    ap.add_argument("--flags", type=int, default=0, help="1 = CUDA-core attention consumer")
    ap.add_argument("--parts", type=int, default=0, help="attention partition (0 = default)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--comparator", action="store_true",
                    help="also time the dense right-padded batch (assemble/extract rebatch "
                         "and a decode step over the padded rows) on the final state")
    ap.add_argument("--layers", type=int, default=1,
                    help="layers per step, each with its own KV pool under the same block "
                         "tables (one graph per step)")
    ap.add_argument("--metadata", default="mapped", choices=["copy", "mapped"],
                    help="per-step metadata: copied to the device, or read in place from "
                         "pinned host memory")
    ap.add_argument("--launch-check", type=int, default=0, metavar="N",
                    help="only set the workload up and run N launches (the attention kernel "
                         "alone, or with --layers L whole L-layer steps), each after the GPU "
                         "sleep that replaces the L2 flush for inputs larger than L2: the "
                         "command an ncu capture of consecutive unflushed launches runs")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# shared helpers
# ---------------------------------------------------------------------------
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the kernel sources' code: line comments and blank lines are left
    out, so an edit that only touches comments keeps the ncu records valid."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode())
                    h.update(b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(workload, kernel_hash, algorithmic_now):
    """DRAM bytes per launch of the split kernel from the committed ncu summary,
    only if it was taken on the current kernel source.  The capture is an
    earlier launch of the same workload (its rows are a few tokens shorter), so
    its DRAM bytes are scaled by the ratio of algorithmic bytes; returns
    (bytes, note) or (None, reason)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None, "no profiles/traffic.json"
    if not rec or rec.get("kernel_hash") != kernel_hash:
        return None, "no ncu capture of the current kernel source"
    dram, alg = rec.get("dram_bytes_per_launch"), rec.get("algorithmic_bytes_per_launch")
    if not dram or not alg:
        return None, "incomplete capture record"
    return int(round(dram * algorithmic_now / alg)), (
        f"ncu capture of an earlier launch: {dram} DRAM bytes for {alg} algorithmic bytes "
        f"(ratio {dram / alg:.4f}), scaled to this launch")


def aggregate_replicas(local_s, local_bytes, world, device=None):
    """N replicas (one process per GPU, no exchange on the data path): the job's
    time is the slowest rank's, its work the sum of every rank's bytes."""
    if world == 1:
        return local_s, local_bytes
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_s], dtype=torch.float64, device=device)
    b = torch.tensor([float(local_bytes)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def attn_bytes(lens_after, Hq, Hkv, d, elem):
    """Algorithmic bytes of one attention pass (a3+a4): every cached K and V
    element once, q in, out written, block-table entries and seq_lens read."""
    lens_after = np.asarray(lens_after, np.int64)
    kv = int(lens_after.sum()) * Hkv * d * 2 * elem
    qo = 2 * len(lens_after) * Hq * d * elem
    tables = int(((lens_after + 15) // 16).sum()) * 4
    return kv + qo + tables + 4 * len(lens_after)


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, kept for the timed
    regions only: ``window()`` brackets a region, and a sample counts when its
    timestamp falls inside one (or within 20 ms after its end).  nvidia-smi
    writes to a file: no Python thread reads it while GPU work is timed (a
    reader thread taking the interpreter lock between an event and the launch
    it brackets left the GPU idle inside the timing)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []          # (sample time, line)
        self.windows = []

    def start(self):
        """Starts sampling every 10 ms and returns once the first sample is in."""
        import tempfile
        try:
            self.fh = tempfile.NamedTemporaryFile("w+", suffix=".csv")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=self.fh, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        t_end = time.perf_counter() + 5.0
        while os.path.getsize(self.fh.name) == 0 and time.perf_counter() < t_end:
            time.sleep(0.005)

    @staticmethod
    def _parse(line):
        """(sample time in seconds since the epoch, the fields after it)."""
        import datetime
        ts, _, rest = line.partition(",")
        try:
            t = datetime.datetime.strptime(ts.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None, rest.strip()
        return t, rest.strip()

    class _Window:
        def __init__(self, owner):
            self.owner = owner

        def __enter__(self):
            self.t0 = time.time()

        def __exit__(self, *exc):
            self.owner.windows.append((self.t0, time.time() + 0.02))

    def window(self):
        return self._Window(self)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.03)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        with open(self.fh.name) as f:
            self.lines = [self._parse(ln) for ln in f if ln.strip()]
        self.fh.close()
        # a sample without a readable timestamp counts (never drops a throttle)
        inside = [ln for t, ln in self.lines
                  if t is None or any(a <= t <= b for a, b in self.windows)]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in inside:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        timed_s = sum(b - a - 0.02 for a, b in self.windows)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0,
                    "timed_region_s": round(timed_s, 3)}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "timed_region_s": round(timed_s, 3)}


# ---------------------------------------------------------------------------
# oracle on the host (cpu baseline and the reference arm)
# ---------------------------------------------------------------------------
# The sample is a set of (row, KV head) units of one decode step.  Their raw
# inputs (the storage type's bits: q rows of the group, the new k and v, the
# row's K/V pages of that head) sit in one shared-memory block; spawned
# workers, one per host core, each run the float64 oracle's decode step on one
# unit at a time.  A pass over the sample is timed by the wall clock.
_WORKER = None


def _oracle_worker_init(shm_name, spec):
    global _WORKER
    from multiprocessing import shared_memory
    _WORKER = (shared_memory.SharedMemory(name=shm_name), spec)


def _upcast(raw, dtype):
    """Storage-type values (bf16 as its 16-bit pattern, or float32) to float64."""
    if dtype == "bf16":
        return (raw.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return raw.astype(np.float64)


def _oracle_unit_job(i):
    """Runs inside a worker: unit i through the oracle's decode step."""
    from oracle.step import decode_step
    shm, (dtype, G, d, scale, base, table) = _WORKER
    elem = np.uint16 if dtype == "bf16" else np.float32
    buf = np.ndarray((shm.size // np.dtype(elem).itemsize,), dtype=elem, buffer=shm.buf)
    off, n, pos, L = (int(x) for x in table[i])
    page = 16 * d
    q = _upcast(buf[off:off + G * d], dtype).reshape(1, G, d)
    k = _upcast(buf[off + G * d:off + (G + 1) * d], dtype).reshape(1, 1, d)
    v = _upcast(buf[off + (G + 1) * d:off + (G + 2) * d], dtype).reshape(1, 1, d)
    o = off + (G + 2) * d
    kc = _upcast(buf[o:o + n * page], dtype).reshape(n, 1, 16, d)
    vc = _upcast(buf[o + n * page:o + 2 * n * page], dtype).reshape(n, 1, 16, d)
    decode_step(q, k, v, [pos], [pos], [L], np.arange(n)[None, :], kc, vc, scale=scale,
                base=base, dtype=dtype)
    return i


def _raw(t, dtype):
    """A CPU tensor's values as the numpy array the workers read."""
    import torch
    t = t.contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else t.numpy()


class OracleSample:
    """The (row, KV head) units of ``rows`` in one decode step, packed into shared
    memory.  ``pages(b)`` returns the K and V pages ``[n, Hkv, 16, d]`` of row
    b's first n blocks as CPU tensors; ``tokens`` are the step's new q/k/v; ``meta``
    its (positions, slots, seq_lens, block_tables)."""

    def __init__(self, w, rows, tokens, meta, pages):
        from multiprocessing import shared_memory
        self.w, self.rows = w, list(rows)
        pos, _, lens, _ = meta
        G, d = w.group, w.d
        q, k, v = (t.cpu() for t in tokens)
        units, chunks, off = [], [], 0
        for b in self.rows:
            n = -(-int(lens[b]) // 16)
            kp, vp = pages(b, n)
            for g in range(w.Hkv):
                parts = [q[b, g * G:(g + 1) * G], k[b, g], v[b, g], kp[:, g], vp[:, g]]
                flat = [_raw(x, w.dtype).reshape(-1) for x in parts]
                units.append((off, n, int(pos[b]), int(lens[b])))
                chunks.append(flat)
                off += sum(len(x) for x in flat)
        itemsize = 2 if w.dtype == "bf16" else 4
        self.shm = shared_memory.SharedMemory(create=True, size=max(off * itemsize, 16))
        buf = np.ndarray((off,), dtype=np.uint16 if w.dtype == "bf16" else np.float32,
                         buffer=self.shm.buf)
        for (o, _, _, _), flat in zip(units, chunks):
            for x in flat:
                buf[o:o + len(x)] = x
                o += len(x)
        del buf
        self.table = np.array(units, np.int64)
        # longest units first, so the pass does not end on one long unit
        self.order = [int(i) for i in np.argsort(-self.table[:, 1], kind="stable")]
        elem = 2 if w.dtype == "bf16" else 4
        self.nbytes = attn_bytes([lens[b] for b in self.rows], w.Hq, w.Hkv, w.d, elem)

    def pool(self, cores):
        import multiprocessing as mp
        env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
        saved = {k: os.environ.get(k) for k in env_keys}
        for k in env_keys:
            os.environ[k] = "1"
        try:
            spec = (self.w.dtype, self.w.group, self.w.d, self.w.scale, self.w.rope_base,
                    self.table)
            return mp.get_context("spawn").Pool(cores, initializer=_oracle_worker_init,
                                                initargs=(self.shm.name, spec))
        finally:
            for k, val in saved.items():
                if val is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = val

    def run_pass(self, pool):
        """One pass over every unit; returns its wall-clock seconds."""
        t0 = time.perf_counter()
        pool.map(_oracle_unit_job, self.order, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self.shm.close()
        self.shm.unlink()

    def describe(self):
        every = self.rows[1] - self.rows[0] if len(self.rows) > 1 else 1
        return (f"the {len(self.table)} (row, KV head) units of {len(self.rows)} of the "
                f"{self.w.B} rows (every {every}th row from row 0) of one {self.w.name} decode "
                f"step; float64 numpy oracle, one spawned single-threaded worker per host core, "
                f"one unit per task, wall clock")


def sample_rows(w, target_rows=32):
    step = max(1, w.B // target_rows)
    return list(range(0, w.B, step))


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def setup(w, device, parts, flags, steps_total, metadata, n_layers=1):
    import torch
    from paged_kv_decode_10_gb300 import engine, workloads
    # room for the timed steps, the six end-to-end runs (up to 53 steps each)
    # and two wall-clock passes over a churn plan (up to 64 steps each)
    extra_tokens = steps_total + 2 * 64 + 6 * 53 + 64
    bt = w.max_blocks_per_seq(extra_tokens=extra_tokens)
    # The recipe's pool holds 1.25x the blocks of the initial lengths; a long
    # run appends extra_tokens to every row.  Blocks for those go to the bottom
    # of the free stack (in seeded random order): the initial block tables and
    # every block the recipe's pool can give are unchanged, and the extra ones
    # are taken only once it runs dry.  (w is updated in place.)
    extra = w.B * (-(-extra_tokens // 16) + 1)
    rng = np.random.Generator(np.random.PCG64(w.seed + 7))
    more = (w.num_blocks + rng.permutation(extra)).astype(np.int32)
    w.free_order = np.concatenate([more, w.free_order])
    w.num_blocks += extra
    pool_bytes = w.num_blocks * w.Hkv * 16 * w.d * (2 if w.dtype == "bf16" else 4)
    gen_dev = "cpu" if pool_bytes < (1 << 30) else device
    k_cache, v_cache = workloads.make_caches(w, gen_dev)
    if n_layers > 1:
        # every layer's pool starts as a copy of the same synthetic cache
        kd, vd = k_cache.to(device), v_cache.to(device)
        k_dev = kd.unsqueeze(0).expand(n_layers, *kd.shape).contiguous()
        v_dev = vd.unsqueeze(0).expand(n_layers, *vd.shape).contiguous()
        del kd, vd
    else:
        k_dev, v_dev = k_cache.to(device), v_cache.to(device)
    dec = engine.PagedDecoder(w.num_blocks, w.Hq, w.Hkv, w.d, w.dtype, w.B, bt,
                              initial_free=w.free_order, device=device,
                              num_parts=parts or None, flags=flags,
                              k_cache=k_dev, v_cache=v_dev, metadata=metadata,
                              n_layers=n_layers)
    ids = [dec.join(int(L)) for L in w.seq_lens]
    if n_layers == 1:
        tokens = [workloads.make_new_tokens(w, s, device) for s in range(steps_total)]
    else:
        tokens = []
        for s in range(steps_total):
            per = [workloads.make_new_tokens(w, s * n_layers + l, device) for l in range(n_layers)]
            tokens.append(tuple(torch.stack([t[i] for t in per]) for i in range(3)))
    return dec, ids, tokens, (k_cache, v_cache) if gen_dev == "cpu" else None


def resident_metadata(dec, device):
    """The current step's block tables, lengths and plan as device tensors:
    the attention kernel timed alone reads all of its inputs from HBM (the step
    itself may read its metadata in place from pinned host memory)."""
    def dev(t):
        return None if t is None else (t if t.is_cuda else t.to(device))
    return dev(dec.tables), dev(dec.seq_lens), dev(dec.plan)


def launch_prep(nbytes, flush, l2):
    """What runs before each timed launch of a graph that reads ``nbytes``, and
    how the line says so.  Inputs larger than L2 (the timing rules' second
    option) are not flushed: a ~50 us GPU sleep keeps the GPU busy while the
    host enqueues, and the kernel's code, parameters and metadata stay in L2 as
    they do from one step to the next in serving (ncu on consecutive launches
    of ragged64 and long131k: every KV byte still comes from DRAM).  Smaller
    inputs get the L2 flush."""
    import torch
    if nbytes > l2:
        return ((lambda: torch.cuda._sleep(100_000)),
                f"not flushed: inputs of {nbytes / 1e6:.0f} MB per launch > L2 ({l2 / 1e6:.0f} MB);"
                " a GPU sleep of ~50 us before each launch")
    return flush, "flushed before every launch (inputs fit in L2)"


def time_graph_launches(g, K, prep, stream, sampler):
    """K replays of graph g, each after ``prep()`` (an L2 flush, or see
    launch_prep), between CUDA events on ``stream``; returns the milliseconds
    of each."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    with sampler.window():
        for i in range(K):
            prep()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    return [e[0].elapsed_time(e[1]) for e in ev]


def layered_step(name, L, args, device, flush, stream, sampler, peak):
    """The whole step of an L-layer decoder (every layer its own pool under the
    one set of block tables: RoPE/append and attention per layer, each layer's
    kernels programmatic dependents of the previous layer's) as one CUDA graph,
    timed after an L2 flush on the state after a few eager steps (metadata read
    in place, as in the served step).  Per layer: the step time / L, and the
    layers' algorithmic attention bytes / the step time."""
    import torch
    from paged_kv_decode_10_gb300 import workloads
    w = workloads.make_workload(name)
    n_eager = 4
    dec, ids, tokens, _ = setup(w, device, args.parts, args.flags, n_eager, "mapped", L)
    for s in range(n_eager):
        dec.step(ids, *tokens[s])
    B = len(ids)
    q, k, v = tokens[n_eager - 1]
    dec.q_ins[:, :B].copy_(q)
    dec.k_ins[:, :B].copy_(k)
    dec.v_ins[:, :B].copy_(v)
    dec.capture(B)
    torch.cuda.synchronize()
    elem = 2 if w.dtype == "bf16" else 4
    lens = np.array(dec.last_metadata[2])
    # by one layer's bytes: a layer's pool that fits in L2 can keep lines from
    # the previous step (ncu: decode16's last layer read 23 of its 37 MB from DRAM)
    prep, how = launch_prep(attn_bytes(lens, w.Hq, w.Hkv, w.d, elem), flush,
                            torch.cuda.get_device_properties(device).L2_cache_size)
    ms, nbytes = [], 0
    with sampler.window():
        for _ in range(args.steps):
            dec.wait_host_buffer()
            lens = np.array(dec.prepare_host(ids)[2])   # a0: each step appends a token
            nbytes += L * attn_bytes(lens, w.Hq, w.Hkv, w.d, elem)
            prep()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dec.replay_step()
            b.record(stream)
            ms.append((a, b))
        torch.cuda.synchronize()
    assert dec.device_errors() == 0, f"device error flag set during the {name} layered timing"
    total_us = 1e3 * sum(x.elapsed_time(y) for x, y in ms)
    step_us = total_us / len(ms)
    gbs = nbytes / (total_us * 1e-6) / 1e9
    return {"workload": name, "layers": L, "step_us": round(step_us, 3),
            "us_per_layer": round(step_us / L, 3), "attention_gbs": round(gbs, 2),
            "frac": round(gbs / peak, 4), "merge_helpers": bool(dec._helpers_now), "l2": how,
            "step": "one graph: per layer RoPE/append + split-KV attention with fused merge"}


def attention_roofline(name, args, device, flush, stream, sampler, peak):
    """The attention kernel (a3 + fused a4) alone on another workload, in the
    bench's launch configuration: every row joined, a few eager decode steps,
    then K graph launches of the attention call on the final step's state (each
    prepared as launch_prep says, and again each after an L2 flush); also the
    step's kernels (RoPE/append + attention)."""
    import torch
    from paged_kv_decode_10_gb300 import binding, workloads
    w = workloads.make_workload(name)
    n_eager = 4
    dec, ids, tokens, _ = setup(w, device, args.parts, args.flags, n_eager, args.metadata)
    for s in range(n_eager):
        dec.step(ids, *tokens[s])
    torch.cuda.synchronize()
    B = len(ids)
    lens = np.array(dec.last_metadata[2])
    step_args = dec.step_args(B, *tokens[n_eager - 1])   # re-running the last step is idempotent
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    attn_graph, kern_graph = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    tables, lens_d, plan = resident_metadata(dec, device)
    with torch.cuda.graph(attn_graph, stream=cap):
        binding.decode_attention(dec.q_rot[:B], dec.k_cache, dec.v_cache, tables, lens_d,
                                 scale=dec.scale, num_parts=dec.num_parts,
                                 workspace=dec.workspace, out=dec.out[:B], flags=dec.flags,
                                 err=dec.err, stream=cap, plan=plan)
    with torch.cuda.graph(kern_graph, stream=cap):
        binding.decode_step_args(step_args, cap)
    stream.wait_stream(cap)
    elem = 2 if w.dtype == "bf16" else 4
    ab = attn_bytes(lens, w.Hq, w.Hkv, w.d, elem)
    prep, how = launch_prep(ab, flush, torch.cuda.get_device_properties(device).L2_cache_size)
    attn_ms = time_graph_launches(attn_graph, args.steps, prep, stream, sampler)
    kern_ms = time_graph_launches(kern_graph, args.steps, prep, stream, sampler)
    flushed_ms = (attn_ms if prep is flush else
                  time_graph_launches(attn_graph, args.steps, flush, stream, sampler))
    assert dec.device_errors() == 0, f"device error flag set during the {name} timing"
    gbs = ab / (statistics.mean(attn_ms) / 1e3) / 1e9
    traffic, note = profiled_traffic(name, kernel_source_hash(), ab)
    return {"workload": name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d,
            "mean_kv_len": float(np.mean(lens)), "num_parts": dec.num_parts,
            "bound": "hbm", "kernel": "attn_split_kernel (a3 + fused a4), timed alone, metadata in HBM",
            "achieved": round(gbs, 2), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
            "traffic": traffic, "traffic_note": note, "algorithmic_bytes_per_launch": int(ab),
            "mean_launch_us": round(1e3 * statistics.mean(attn_ms), 3),
            "median_launch_us": round(1e3 * statistics.median(attn_ms), 3),
            "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4), "l2": how,
            **flushed_fields(ab, flushed_ms, peak),
            "step_kernels_us": round(1e3 * statistics.mean(kern_ms), 3),
            "steps_per_s": round(1e3 / statistics.mean(kern_ms), 1)}


def flushed_fields(ab, flushed_ms, peak):
    """The same launches each after an L2 flush (for comparison)."""
    us = 1e3 * statistics.mean(flushed_ms)
    return {"flushed_launch_us": round(us, 3), "flushed_frac": round(ab / (us * 1e-6) / 1e9 / peak, 4)}


def launch_check(args):
    """N launches each after a ~50 us GPU sleep and no L2 flush (see
    launch_prep): the attention kernel alone on the state after four eager
    steps, metadata in device memory, or with --layers L whole L-layer steps."""
    import torch
    from paged_kv_decode_10_gb300 import binding, workloads
    device = torch.device("cuda", 0)
    w = workloads.make_workload(args.workload)
    dec, ids, tokens, _ = setup(w, device, args.parts, args.flags, 4, "mapped", args.layers)
    for s in range(4):
        dec.step(ids, *tokens[s])
    B = len(ids)
    if args.layers > 1:
        q, k, v = tokens[3]
        dec.q_ins[:, :B].copy_(q)
        dec.k_ins[:, :B].copy_(k)
        dec.v_ins[:, :B].copy_(v)
        dec.capture(B)
    tables, lens_d, plan = resident_metadata(dec, device)
    for _ in range(args.launch_check):
        if args.layers > 1:
            dec.wait_host_buffer()
            dec.prepare_host(ids)
        torch.cuda._sleep(100_000)
        if args.layers > 1:
            dec.replay_step()
        else:
            binding.decode_attention(dec.q_rot[:B], dec.k_cache, dec.v_cache, tables, lens_d,
                                     scale=dec.scale, num_parts=dec.num_parts,
                                     workspace=dec.workspace, out=dec.out[:B], flags=dec.flags,
                                     err=dec.err, plan=plan)
    torch.cuda.synchronize()
    assert dec.device_errors() == 0
    elem = 2 if w.dtype == "bf16" else 4
    print(json.dumps({"launch_check": args.launch_check, "workload": w.name,
                      "layers": args.layers, "algorithmic_bytes_per_launch": int(attn_bytes(
                          np.array(dec.last_metadata[2]), w.Hq, w.Hkv, w.d, elem))}))


def run_gpu(args, rank, world, want_cpu=False):
    import torch
    from paged_kv_decode_10_gb300 import binding, workloads
    local = int(os.environ.get("LOCAL_RANK", "0"))
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = workloads.make_workload(args.workload)
    W, K, GW = args.warmup, args.steps, 2
    dec, ids, tokens, _ = setup(w, device, args.parts, args.flags, W + GW + K + 1,
                                args.metadata, args.layers)
    assert dec.bt_stride * 16 >= int(w.seq_lens.max()) + W + GW + K + 64
    B = len(ids)
    elem = 2 if w.dtype == "bf16" else 4
    stream = torch.cuda.current_stream(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    # read in full before every timed step: evicts the KV from L2 (without
    # leaving dirty lines to write back) and keeps the GPU busy while the host
    # prepares the next step
    flush_buf = torch.ones(max(4 * l2, 512 << 20) // 8, dtype=torch.int64, device=device)

    def flush():
        if not args.no_flush:
            flush_buf.sum()

    churn_s = []
    prefill_log = []     # (tokens, start event, end event) per churn step
    if w.churn:
        # synthetic raw prefix keys/values of the joiners (the prefill's input)
        max_t = max(int(np.sum(p)) for _, p in w.churn)
        gen = torch.Generator(device=device).manual_seed(1000 + w.seed)
        pre_k = torch.randn((max_t, w.Hkv, w.d), generator=gen, device=device).to(dec.tdtype)
        pre_v = torch.randn((max_t, w.Hkv, w.d), generator=gen, device=device).to(dec.tdtype)
        # two pinned (positions, slots) buffers, so that filling one never waits
        # for the prefill that still reads the other
        pre_bufs = []
        for _ in range(2):
            pos_t = torch.empty(max_t, dtype=torch.int32).pin_memory()
            slot_t = torch.empty(max_t, dtype=torch.int64).pin_memory()
            pre_bufs.append(dict(pos=pos_t, slot=slot_t, np=(pos_t.numpy(), slot_t.numpy()),
                                 done=None))

    def churn(s, timed=True):
        """Continuous batching: before step s >= 1 the planned rows leave and new
        rows join in their places (host allocator; no KV moves), and the joiners'
        prefix KV is written into their new blocks by the prefill kernel
        (pkv_seqs_join's prefix slots + pkv_prefill_kv, timed on its own after an
        L2 flush unless `timed` is off)."""
        if not w.churn or s == 0:
            return
        leave, prefixes = w.churn[(s - 1) % len(w.churn)]
        buf = pre_bufs[s % 2]
        if buf["done"] is not None:
            buf["done"].synchronize()   # the prefill two churns back reads these arrays
        t0 = time.perf_counter()
        dec.alloc.leave_many([ids[row] for row in leave])
        joined = dec.alloc.join_many(prefixes, buf["np"])
        for row, sid in zip(leave, joined):
            ids[row] = int(sid)
        churn_s.append(time.perf_counter() - t0)
        n = int(np.sum(prefixes))
        if timed:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for layer in range(dec.n_layers):
            binding.prefill_kv(pre_k[:n], pre_v[:n], buf["pos"][:n], buf["slot"][:n],
                               dec.k_caches[layer], dec.v_caches[layer], base=dec.rope_base,
                               err=dec.err, stream=stream)
        e1.record(stream)
        buf["done"] = e1
        if timed:
            prefill_log.append((s, n * dec.n_layers, e0, e1))

    # warm-up: eager steps through the C ABI (one pkv_decode_step call each)
    for s in range(W):
        churn(s)
        q, k, v = tokens[s]
        dec.step(ids, q, k, v)
    # the timed step: one CUDA graph (metadata H2D + rope/append + attention)
    dec.capture(B)

    def stage(s):
        q, k, v = tokens[s]
        if args.layers > 1:
            dec.q_ins[:, :B].copy_(q)
            dec.k_ins[:, :B].copy_(k)
            dec.v_ins[:, :B].copy_(v)
        else:
            dec.q_in[:B].copy_(q)
            dec.k_in[:B].copy_(k)
            dec.v_in[:B].copy_(v)

    for s in range(W, W + GW):
        churn(s)
        stage(s)
        dec.prepare_host(ids)
        dec.replay_step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    # K + 1 steps run in the timed loop and the first is not counted: the first
    # step of the loop ran up to 8x slower than the rest, after a full untimed
    # warm-up, for reasons outside the step (a GPU sleep before it did not help)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K + 1)]
    lens_after = []
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_host = 0.0
    with sampler.window():
        for i in range(K + 1):
            churn(W + GW + i)
            stage(W + GW + i)
            dec.wait_host_buffer()   # the replay two steps back still reads it
            t0 = time.perf_counter()
            lens = np.array(dec.prepare_host(ids)[2])
            if i > 0:
                t_host += time.perf_counter() - t0
                lens_after.append(lens)
            flush()   # still running on the GPU when the replay below is enqueued
            evs[i][0].record(stream)
            dec.replay_step()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs[1:]]
    total_s = sum(step_ms) / 1e3

    # The dominant kernel (split-KV attention with its fused merge) timed alone
    # on the final step's state, in the step's launch configuration, and the
    # step's kernels (RoPE/append + attention) without the host side; each is
    # captured once so that no host launch time falls between the events.
    # Re-running the final step is idempotent (the same token re-appended).
    if args.layers > 1:
        step_args = dec.layer_args(B, dec.q_ins[:, :B], dec.k_ins[:, :B], dec.v_ins[:, :B])
    else:
        step_args = dec.step_args(B, dec.q_in[:B], dec.k_in[:B], dec.v_in[:B])
    cap = torch.cuda.Stream(device)
    cap.wait_stream(stream)
    attn_graph, kern_graph = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    tables, lens_d, plan = resident_metadata(dec, device)
    with torch.cuda.graph(attn_graph, stream=cap):
        binding.decode_attention(dec.q_rot[:B], dec.k_cache, dec.v_cache, tables, lens_d,
                                 scale=dec.scale, num_parts=dec.num_parts,
                                 workspace=dec.workspace, out=dec.out[:B], flags=dec.flags,
                                 err=dec.err, stream=cap, plan=plan)
    with torch.cuda.graph(kern_graph, stream=cap):
        if args.layers > 1:
            binding.decode_step_layers(step_args, cap)
        else:
            binding.decode_step_args(step_args, cap)
    stream.wait_stream(cap)

    last_lens = lens_after[-1]
    attn_b = attn_bytes(last_lens, w.Hq, w.Hkv, w.d, elem)
    prep, prep_how = launch_prep(attn_b, flush, l2)

    def time_graph(g, how=None):
        return time_graph_launches(g, K, how or prep, stream, sampler)

    attn_ms = time_graph(attn_graph)
    kern_ms = time_graph(kern_graph)
    flushed_ms = attn_ms if prep is flush else time_graph(attn_graph, flush)

    # the same step with the other metadata placement: copied to the device by
    # a copy node at the head of the graph (or, for a decoder that copies,
    # read in place from the pinned buffer)
    other_ms, other_mode = None, None
    if args.layers == 1:
        from paged_kv_decode_10_gb300 import engine as _engine
        nbytes = _engine._metadata_layout(B, dec.bt_stride, dec._plan_parts)[-1]
        host_raw = dec._host[dec._turn ^ 1]["raw"]    # the buffer of the final step
        if args.metadata == "mapped":
            other_mode = "copy"
            dev_raw = torch.empty(nbytes, dtype=torch.uint8, device=device)
            views = dec._views(dev_raw, B)[0]
        else:
            other_mode = "mapped"
            views = dec._views(host_raw, B)[0]
        oargs = binding.make_step_args(
            dec.q_in[:B], dec.k_in[:B], dec.v_in[:B], dec.q_rot[:B], dec.k_rot[:B], dec.k_cache,
            dec.v_cache, *views[:4], dec.scale, dec.rope_base, dec.num_parts, dec.workspace,
            dec.out[:B], flags=dec.flags, err=dec.err, plan=views[4])
        og = torch.cuda.CUDAGraph()
        cap.wait_stream(stream)
        with torch.cuda.graph(og, stream=cap):
            if other_mode == "copy":
                dev_raw.copy_(host_raw[:nbytes], non_blocking=True)
            binding.decode_step_args(oargs, cap)
        stream.wait_stream(cap)
        other_ms = time_graph(og)

    # the oracle's sample: rows of the final timed step, their pages copied to
    # the host before the state moves on
    sample = None
    if want_cpu:
        meta = [np.array(x) for x in dec.last_metadata]
        last_tok = tokens[W + GW + K]
        if args.layers > 1:
            last_tok = tuple(t[0] for t in last_tok)

        def pages(b, n):
            idx = torch.from_numpy(meta[3][b, :n].astype(np.int64)).to(device)
            return dec.k_cache[idx].cpu(), dec.v_cache[idx].cpu()

        sample = OracleSample(w, sample_rows(w), last_tok, meta, pages)

    # churn plans: passes over the plan timed by the wall clock, host work
    # included, no flush.  The headline pass runs the native serving loop
    # (pkv_server_step: one host call per step does the leaves and joins, the
    # joiners' prefill, input staging, a0, the plan and the graph launch); the
    # pass before it drives the same work from Python, for comparison.
    wall = None
    if w.churn and world == 1 and args.layers == 1:
        n_wall = len(w.churn)
        s0 = W + GW + K + 1
        phase = [0.0] * 4     # churn + prefill enqueue, input staging, a0, graph launch
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n_wall):
            ta = time.perf_counter()
            churn(s0 + i, timed=False)
            tb = time.perf_counter()
            stage((s0 + i) % len(tokens))
            tc = time.perf_counter()
            dec.prepare_host(ids)
            td = time.perf_counter()
            dec.replay_step()
            te = time.perf_counter()
            for j, dt in enumerate((tb - ta, tc - tb, td - tc, te - td)):
                phase[j] += dt
        torch.cuda.synchronize()
        py_s = time.perf_counter() - t0
        us = lambda x: round(1e6 * x / n_wall, 1)
        # the native loop over the next pass of the plan, from the same state
        server = binding.Server(dec, ids, max(int(np.sum(p)) for _, p in w.churn))
        s1 = s0 + n_wall
        runners = []
        for i in range(n_wall):
            leave, prefixes = w.churn[(s1 + i - 1) % len(w.churn)]
            n = int(np.sum(prefixes))
            q, k, v = tokens[(s1 + i) % len(tokens)]
            runners.append(server.step_runner(leave, prefixes, pre_k[:n], pre_v[:n], q, k, v,
                                              stream))
        host_s = 0.0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for run in runners:
            ta = time.perf_counter()
            run()
            host_s += time.perf_counter() - ta
        torch.cuda.synchronize()
        wall_s = time.perf_counter() - t0
        ids[:] = [int(x) for x in server.rows()]
        server.close()
        wall = {"steps": n_wall, "steps_per_s": round(n_wall / wall_s, 1),
                "ms_per_step": round(1e3 * wall_s / n_wall, 4),
                "host_us_per_step": us(host_s),
                "path": "pkv_server_step: leaves and joins, joiners' prefix KV (pkv_prefill_kv), "
                        "input staging, a0 (pkv_prepare_step_cached), plan and one graph launch "
                        "in one host call per step; no L2 flush; the host time includes waits "
                        "for the GPU to release the pinned buffers of the step two back",
                "python_loop": {
                    "ms_per_step": round(1e3 * py_s / n_wall, 4),
                    "host_us_per_step": {"join_leave_prefill": us(phase[0]),
                                         "stage_inputs": us(phase[1]), "a0": us(phase[2]),
                                         "graph_launch": us(phase[3])},
                    "path": "the same steps driven from Python (batched allocator calls, "
                            "pkv_prefill_kv, torch copies, engine a0, graph replay)"}}

    peak, peak_kind = measured_peak()
    rooflines = {}
    for name in [x for x in args.also.split(",") if x and x != w.name]:
        rooflines[name] = attention_roofline(name, args, device, flush, stream, sampler, peak)
    layered = {}
    if args.layers == 1:
        for spec in [x for x in args.layered.split(",") if x]:
            name, L = spec.split(":")
            layered[spec] = layered_step(name, int(L), args, device, flush, stream, sampler,
                                         peak)
    clocks = sampler.stop()

    bytes_steps = [args.layers * attn_bytes(la, w.Hq, w.Hkv, w.d, elem) for la in lens_after]
    kv_only = [args.layers * int(np.asarray(la, np.int64).sum()) * w.Hkv * w.d * 2 * elem
               for la in lens_after]
    total_s, total_bytes = aggregate_replicas(total_s, sum(bytes_steps), world, device)
    value = total_bytes / total_s / 1e9
    attn_gbs = attn_b / (statistics.mean(attn_ms) / 1e3) / 1e9
    assert dec.device_errors() == 0, "device error flag set during the bench"

    khash = kernel_source_hash()
    traffic, traffic_note = profiled_traffic(args.workload, khash,
                                             attn_bytes(last_lens, w.Hq, w.Hkv, w.d, elem))
    result = {
        "metric": "paged decode-attn achieved HBM GB/s (% of GB300 peak); batched decode steps/s",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(total_s * 1e3 / K, 5),
        "ms_per_step_median": round(statistics.median(step_ms), 5),
        "ms_per_step_max": round(max(step_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) q/k/v and KV pool; seeded ragged lengths and "
                "scattered block tables)",
        "config": {"workload": w.name, "layers": args.layers, "B": w.B, "Hq": w.Hq,
                   "Hkv": w.Hkv, "head_dim": w.d,
                   "block_size": 16, "mean_kv_len": float(np.mean(lens_after[0])),
                   "pool_blocks": w.num_blocks, "num_parts": dec.num_parts,
                   "consumer": "simt" if (args.flags & 1 or w.dtype == "f32") else "mma.sync",
                   "step": "one CUDA graph: " + (
                       "metadata H2D copy + " if args.metadata == "copy" else
                       "metadata read in place from pinned host memory + ") + (
                       "one kernel (RoPE, append, split-KV attention, LSE merge)"
                       if args.flags & 4 else
                       "RoPE/append kernel + split-KV attention kernel with fused LSE merge "
                       "(programmatic dependent launch)") + (
                       f", for each of {args.layers} layers (each layer's kernels launched as "
                       "dependents of the previous layer's)" if args.layers > 1 else ""),
                   "l2": "flushed before every timed step" if not args.no_flush else "not flushed",
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "steps_per_s": round(K / (sum(step_ms) / 1e3), 1),
        "attn_gbs": round(attn_gbs, 2),
        "pct_of_peak": round(100 * attn_gbs / peak, 2),
        "kv_bytes_per_step": int(statistics.mean(kv_only)),
        "roofline": {"bound": "hbm", "kernel": "attn_split_kernel (a3 + fused a4), timed alone, metadata in HBM",
                     "achieved": round(attn_gbs, 2), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(attn_gbs / peak, 4),
                     "traffic": traffic, "traffic_note": traffic_note,
                     "algorithmic_bytes_per_launch": int(attn_b),
                     "mean_launch_us": round(1e3 * statistics.mean(attn_ms), 3),
                     "median_launch_us": round(1e3 * statistics.median(attn_ms), 3),
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(attn_gbs / NOMINAL_HBM_GBS, 4),
                     "l2": prep_how, **flushed_fields(attn_b, flushed_ms, peak),
                     "kernel_hash": khash},
        "host_a0_us_per_step": round(1e6 * t_host / K, 2),
        "host_churn_us_per_step": round(1e6 * statistics.mean(churn_s), 2) if churn_s else None,
        "churn_wall_clock": wall,
        "step_kernels_us": round(1e3 * statistics.mean(kern_ms), 3),
        "step_other_metadata": None if other_ms is None else {
            "metadata": other_mode, "step_us": round(1e3 * statistics.mean(other_ms), 3),
            "note": "the final step's graph replayed with its metadata and plan "
                    + ("copied to device memory by a copy node at the head of the graph"
                       if other_mode == "copy" else "read in place from pinned host memory")
                    + ", against step_kernels_us for this run's placement"},
        "prefill": prefill_summary([x[1:] for x in prefill_log if x[0] > W + GW], w, elem,
                                   peak),
        "gpu_launches": K * args.layers * ((1 if args.flags & 4 else 2) +
                                           (1 if args.flags & 2 else 0)),
        "rooflines": rooflines or None,
        "layered": layered or None,
        "clocks": clocks,
    }
    return result, dec, ids, tokens, sample, w


def run_dense_comparator(args, dec, ids, w, peak):
    """The dense right-padded batch that paging replaces, on the same rows and
    lengths as the paged run's final state: the decode step over the padded
    rows (gap masked, read all the same) and one rebatch (every row extracted
    to a snapshot, then assembled again), each timed on the device after an L2
    flush.  Paging's rebatch is a host block-table edit with no device copy."""
    import torch
    from paged_kv_decode_10_gb300 import binding, dense, workloads
    device = dec.device
    B = len(ids)
    elem = 2 if w.dtype == "bf16" else 4
    lens = [dec.alloc.seq_len(s) for s in ids]
    P = max(lens)
    cap = (P + 1 + 15) // 16 * 16
    db = dense.DenseBatch(w.Hq, w.Hkv, w.d, w.dtype, B, cap, device, num_parts=dec.num_parts,
                          flags=dec.flags)
    gen = torch.Generator(device=device).manual_seed(77)
    snaps = []
    for L in lens:
        k, v = db.new_snapshot(L)
        k.normal_(generator=gen)
        v.normal_(generator=gen)
        snaps.append((k, v))
    ks, vs = [s[0] for s in snaps], [s[1] for s in snaps]
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_buf = torch.ones(max(4 * l2, 512 << 20) // 8, dtype=torch.int64, device=device)
    stream = torch.cuda.current_stream(device)
    reps = max(3, min(args.steps, 20))

    def timed(fn):
        ms = []
        for _ in range(reps + 1):
            flush_buf.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        return statistics.mean(ms[1:]) * 1e3

    db.assemble(ks, vs, lens)      # sets up the gap mask and the tables once
    # the timed rebatch is the device copy alone (the mask is rebuilt on the
    # host per rebatch and is not counted)
    assemble_us = timed(lambda: binding.dense_assemble(ks, vs, lens, P, db.k, db.v, cap))
    q, k, v = workloads.make_new_tokens(w, 0, device)
    args_d = db.step_args(q, k, v)
    graph = torch.cuda.CUDAGraph()
    cap_s = torch.cuda.Stream(device)
    cap_s.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap_s):
        binding.decode_step_args(args_d, cap_s)
    stream.wait_stream(cap_s)
    step_us = timed(graph.replay)
    extract_us = timed(lambda: db.extract(list(range(B)), ks, vs))
    assert db.device_errors() == 0
    tok_bytes = w.Hkv * w.d * 2 * elem                     # K and V of one token
    dense_attn = attn_bytes([P + 1] * B, w.Hq, w.Hkv, w.d, elem)
    live = sum(lens)
    rebatch_bytes = 4 * live * tok_bytes + sum(P - L for L in lens) * tok_bytes
    return {"rows": B, "padded_len": P, "live_tokens": live, "padded_tokens": B * P,
            "step_kernels_us": round(step_us, 3),
            "step_attn_bytes": int(dense_attn),
            "step_useful_bytes": int(attn_bytes([L + 1 for L in lens], w.Hq, w.Hkv, w.d, elem)),
            "assemble_us": round(assemble_us, 3), "extract_us": round(extract_us, 3),
            "rebatch_us": round(assemble_us + extract_us, 3),
            # extract reads and writes every live token; assemble does the same and
            # writes the zero gap
            "rebatch_device_bytes": int(rebatch_bytes),
            "rebatch_gbs": round(rebatch_bytes / ((assemble_us + extract_us) * 1e-6) / 1e9, 2),
            "paged_rebatch_device_bytes": 0,
            "note": "dense step = RoPE/append + attention over the padded rows (gap masked); "
                    "rebatch = extract every row + assemble every row (one join/leave event)"}


def prefill_summary(log, w, elem, peak):
    """Joiners' prefix KV writes of a churn run: tokens per call and the
    achieved bandwidth of pkv_prefill_kv (reads raw k and v, writes both into
    the cache, reads positions and slots: 4*Hkv*d*elem + 12 bytes per token)."""
    if not log:
        return None
    toks = [n for n, _, _ in log]
    us = [1e3 * a.elapsed_time(b) for _, a, b in log]
    nbytes = [n * (4 * w.Hkv * w.d * elem + 12) for n in toks]
    gbs = sum(nbytes) / (sum(us) * 1e-6) / 1e9
    med = statistics.median(us)
    gbs_med = statistics.median(b / (t * 1e-6) / 1e9 for b, t in zip(nbytes, us))
    return {"kernel": "prefill_kernel (pkv_prefill_kv)", "calls": len(log),
            "tokens_per_call": round(statistics.mean(toks), 1),
            "us_per_call": round(statistics.mean(us), 3), "achieved_gbs": round(gbs, 2),
            "frac": round(gbs / peak, 4), "us_median": round(med, 3), "us_max": round(max(us), 3),
            "achieved_gbs_median": round(gbs_med, 2), "frac_median": round(gbs_med / peak, 4),
            "l2": "flushed before every call"}


def run_e2e(args, dec, ids, tokens, w):
    """Same metric end to end through the C ABI from pinned host buffers: each
    timed step runs the host allocator (a0) and one launch of the captured host
    step (pkv_step_graph: the kernels read q/k/v and the step metadata in place
    over the CPU-GPU link and write the output in place into host memory -- the
    host-to-device and device-to-host transfers happen inside them), and waits.
    For context the same steps are also timed through pkv_decode_step_host
    without the graph, and with a cudaMemcpyAsync of every input."""
    import torch
    from paged_kv_decode_10_gb300 import binding
    device = dec.device
    B = len(ids)
    elem = 2 if w.dtype == "bf16" else 4
    pinned = [t.cpu().pin_memory() for t in tokens[-1]]
    out_h = torch.empty((B, w.Hq, w.d), dtype=dec.tdtype).pin_memory()
    meta_h = (torch.empty(B, dtype=torch.int32).pin_memory(),
              torch.empty(B, dtype=torch.int64).pin_memory(),
              torch.empty(B, dtype=torch.int32).pin_memory(),
              torch.empty((B, dec.bt_stride), dtype=torch.int32).pin_memory())
    dq, dk, dv = (torch.empty_like(t, device=device) for t in pinned)
    meta_d = [torch.empty_like(m, device=device) for m in meta_h]
    # the host-planned partition, written by the host after a0 like the metadata
    plan_h = torch.empty((dec.num_parts, binding.PLAN_INTS), dtype=torch.int32).pin_memory()
    plan_d = torch.empty_like(plan_h, device=device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_buf = torch.ones(max(2 * l2, 256 << 20) // 8, dtype=torch.int64, device=device)
    h2d = sum(t.numel() * t.element_size() for t in pinned) + \
        sum(t.numel() * t.element_size() for t in meta_h) + plan_h.numel() * 4
    d2h = out_h.numel() * out_h.element_size()
    n = max(3, min(args.steps, 50))

    views = tuple(m.numpy() for m in meta_h)
    # a0 writes the same pinned arrays every step: only the changed table entries
    a0 = dec.alloc.step_runner(ids, dec.bt_stride, views,
                               row_state=np.full(3 * B, -1, np.int32))
    planner = binding.plan_runner(views[2], views[3], w.Hkv, w.d, dec.num_parts, plan_h.numpy())

    def prepare_planned():
        a0()
        planner()
    call = binding.load().pkv_decode_step_host
    launch = binding.load().pkv_step_graph_launch
    stream = binding._stream()

    def timed(step, prepare):
        secs, nbytes = 0.0, 0
        for i in range(n + 3):
            flush_buf.sum()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            prepare()
            step()
            dt = time.perf_counter() - t0
            if i >= 3:
                secs += dt
                nbytes += attn_bytes(views[2], w.Hq, w.Hkv, w.d, elem)
        return nbytes / secs / 1e9, 1e3 * secs / n

    def host_step(io, planned, extra_flags=0):
        a = binding.make_step_args(
            dq, dk, dv, dec.q_rot[:B], dec.k_rot[:B], dec.k_cache, dec.v_cache, *meta_d,
            dec.scale, dec.rope_base, dec.num_parts, dec.workspace, dec.out[:B],
            flags=dec.flags | extra_flags, err=dec.err, plan=plan_d if planned else None)
        refs = (ctypes.byref(a), ctypes.byref(io))
        return (lambda: binding._check(call(refs[0], refs[1], stream))), (a, io)

    def graph_step(planned):
        io = binding.host_io(*pinned, *meta_h, out_h, flags=binding.HOST_IN_PLACE,
                             plan=plan_h if planned else None)
        step, keep = host_step(io, planned)
        g = binding.StepGraph(keep[0], io)
        return (lambda: binding._check(launch(g._h, stream))), g

    def pipelined(planned, extra_flags=0):
        """The captured host step with the host's allocator work (a0 + plan) of
        step i+1 running while the GPU runs step i: two graphs over two sets of
        pinned metadata, plan and output buffers, used in turn.  Per step:
        prepare the next set, enqueue its graph behind the running step, wait
        for the running step (its output is then in host memory).  No L2 flush
        between steps (the GPU is never idle for one): only launches that read
        more than L2 report it as the end-to-end figure."""
        sets = [(meta_h, plan_h, out_h, views, a0, planner)]
        m2 = tuple(torch.empty_like(m).pin_memory() for m in meta_h)
        p2 = torch.empty_like(plan_h).pin_memory()
        o2 = torch.empty_like(out_h).pin_memory()
        v2 = tuple(m.numpy() for m in m2)
        sets.append((m2, p2, o2, v2,
                     dec.alloc.step_runner(ids, dec.bt_stride, v2,
                                           row_state=np.full(3 * B, -1, np.int32)),
                     binding.plan_runner(v2[2], v2[3], w.Hkv, w.d, dec.num_parts, p2.numpy())))
        graphs, preps, lens = [], [], []
        for meta, plan, out, vw, alloc_step, plan_step in sets:
            io = binding.host_io(*pinned, *meta, out, flags=binding.HOST_IN_PLACE,
                                 plan=plan if planned else None)
            a, _ = host_step(io, planned, extra_flags)[1]
            graphs.append(binding.StepGraph(a, io))
            preps.append((lambda s0=alloc_step, s1=plan_step: (s0(), s1()))
                         if planned else alloc_step)
            lens.append(vw[2])
        lib = binding.load()
        enqueue, wait = lib.pkv_step_graph_enqueue, lib.pkv_step_graph_wait
        try:
            flush_buf.sum()
            torch.cuda.synchronize()
            seen = []
            preps[0]()
            binding._check(enqueue(graphs[0]._h, stream))
            for j in range(1, n + 3):          # steps 3 .. n+2 are timed
                if j == 3:
                    t0 = time.perf_counter()
                preps[j % 2]()                 # set j%2: step j-2 was waited for
                binding._check(enqueue(graphs[j % 2]._h, stream))
                binding._check(wait(graphs[(j - 1) % 2]._h))   # step j-1's output
                if j >= 3:
                    seen.append(lens[j % 2].copy())
            binding._check(wait(graphs[(n + 2) % 2]._h))
            secs = time.perf_counter() - t0
        finally:
            for g in graphs:
                g.close()
        nbytes = sum(attn_bytes(x, w.Hq, w.Hkv, w.d, elem) for x in seen)
        return nbytes / secs / 1e9, 1e3 * secs / n

    # the captured host step (pkv_step_graph): one launch per step, with the
    # host-planned partition and without it (the kernel then derives it)
    results = {}
    for planned in (True, False):
        step, g = graph_step(planned)
        results[planned] = timed(step, prepare_planned if planned else a0)
        g.close()
    best = min(results, key=lambda k: results[k][1])
    gbs_pipe, ms_pipe = pipelined(best)
    # the same loop with the whole step in one kernel (PKV_STEP_FUSED): each
    # part rotates its own units' queries and the owners of the rows' last
    # pages append, instead of one RoPE/append kernel reading every q/k/v first
    fused = not (dec.flags & binding.STEP_FUSED) and args.layers == 1
    gbs_fz, ms_fz = pipelined(best, binding.STEP_FUSED) if fused else (None, None)
    io_in_place = binding.host_io(*pinned, *meta_h, out_h, flags=binding.HOST_IN_PLACE,
                                  plan=plan_h if best else None)
    gbs_p, ms_p = timed(host_step(io_in_place, best)[0], prepare_planned if best else a0)
    io_copy = binding.host_io(*pinned, *meta_h, out_h, plan=plan_h if best else None)
    gbs_c, ms_c = timed(host_step(io_copy, best)[0], prepare_planned if best else a0)
    gbs, ms = results[best]
    other = results[not best]
    plan_word = lambda p: "with the host-planned partition" if p else "kernel-derived partition"
    seq_path = ("pkv_step_graph_launch: a0 (+ plan) + one graph (kernels reading the pinned "
                "inputs and writing the pinned output over the CPU-GPU link) + stream wait, "
                "L2 flushed before each step (untimed), " + plan_word(best))
    pipe_path = ("pkv_step_graph_enqueue / pkv_step_graph_wait on two graphs and two pinned "
                 "buffer sets: a0 (+ plan) of step i+1 on the host and its launch queued while "
                 "the GPU runs step i, " + plan_word(best))
    # A launch that reads more than L2 leaves nothing in it for the next step:
    # the pipelined loop (no flush between steps) is then the end-to-end figure.
    fz_path = pipe_path + ", PKV_STEP_FUSED (one kernel per step)"
    fz_faster = fused and ms_fz < ms_pipe
    big = attn_bytes(views[2], w.Hq, w.Hkv, w.d, elem) > l2
    pipe_best = (gbs_fz, ms_fz, fz_path) if fz_faster else (gbs_pipe, ms_pipe, pipe_path)
    pipe_other = (gbs_pipe, ms_pipe, pipe_path) if fz_faster else (gbs_fz, ms_fz, fz_path)
    head = pipe_best if big else (gbs, ms, seq_path)
    tail = (gbs, ms, seq_path) if big else (pipe_best[0], pipe_best[1], pipe_best[2] +
                                            " (no L2 flush between steps: inputs fit in L2)")
    return {"value": round(head[0], 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d - (0 if best else plan_h.numel() * 4)),
            "d2h_bytes_per_step": int(d2h),
            "steps": n, "ms_per_step": round(head[1], 4), "path": head[2],
            "sequential" if big else "pipelined": {
                "value": round(tail[0], 2), "unit": "GB/s", "ms_per_step": round(tail[1], 4),
                "path": tail[2]},
            "pipelined_other_step_form": None if not fused else {
                "value": round(pipe_other[0], 2), "unit": "GB/s",
                "ms_per_step": round(pipe_other[1], 4), "path": pipe_other[2]},
            "other_partition": {"value": round(other[0], 2), "unit": "GB/s",
                                "ms_per_step": round(other[1], 4), "path": plan_word(not best)},
            "without_graph": {"value": round(gbs_p, 2), "unit": "GB/s",
                              "ms_per_step": round(ms_p, 4),
                              "path": "pkv_decode_step_host, PKV_HOST_IN_PLACE"},
            "with_copies": {"value": round(gbs_c, 2), "unit": "GB/s", "ms_per_step": round(ms_c, 4),
                            "path": "pkv_decode_step_host with one cudaMemcpyAsync per input"}}


def cpu_baseline(sample, budget_s):
    """The float64 oracle on this host's cores over the sample, wall clock: one
    untimed pass (worker start-up), then passes until ``budget_s`` is used."""
    cores = host_cores()
    pool = sample.pool(cores)
    try:
        sample.run_pass(pool)
        secs, passes = 0.0, 0
        t_end = time.perf_counter() + budget_s
        while passes < 1 or (time.perf_counter() < t_end and passes < 50):
            secs += sample.run_pass(pool)
            passes += 1
    finally:
        pool.close()
        pool.join()
        sample.close()
    gbs = passes * sample.nbytes / secs / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{passes} timed pass(es) over " + sample.describe(),
            "sample_bytes": int(sample.nbytes),
            "ms_per_pass": round(1e3 * secs / passes, 2)}


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    from oracle.allocator import BlockAllocatorModel
    from paged_kv_decode_10_gb300 import workloads
    if rank != 0:
        return None
    w = workloads.make_workload(args.workload)
    bt = w.max_blocks_per_seq()
    model = BlockAllocatorModel(w.num_blocks, max_seqs=w.B, max_blocks_per_seq=bt,
                                initial_free=w.free_order)
    mids = [model.join(int(L)) for L in w.seq_lens]
    meta = model.prepare_step(mids, bt)
    rows = sample_rows(w)
    tokens = workloads.make_new_tokens(w, 0, "cpu")

    def pages(b, n):   # the sampled rows' pages, drawn N(0,1) row by row
        shape = (n, w.Hkv, 16, w.d)
        return (workloads.normal(shape, w.dtype, w.seed * 7919 + 2 * b + 1),
                workloads.normal(shape, w.dtype, w.seed * 7919 + 2 * b + 2))

    sample = OracleSample(w, rows, tokens, meta, pages)
    cores = host_cores()
    pool = sample.pool(cores)
    try:
        for _ in range(max(1, args.warmup)):
            sample.run_pass(pool)
        secs = sum(sample.run_pass(pool) for _ in range(args.steps))
    finally:
        pool.close()
        pool.join()
        sample.close()
    value = args.steps * sample.nbytes / secs / 1e9
    return {"impl": "reference", "metric": "paged decode-attn achieved HBM GB/s (% of GB300 "
            "peak); batched decode steps/s", "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                       "head_dim": w.d, "block_size": 16},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle",
                             "sample": "each bench step is one pass over " + sample.describe()
                             + " (pages of the sampled rows drawn N(0,1))",
                             "sample_bytes": int(sample.nbytes)},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if world > 1 and rank != 0:
            return
        res = run_reference(args, rank, world)
        print(json.dumps(res), flush=True)
        return
    import torch
    if world > 1:
        torch.distributed.init_process_group(
            backend="nccl", init_method="env://")
    from paged_kv_decode_10_gb300 import build
    build.build()
    if args.launch_check:
        launch_check(args)
        return
    want_cpu = not args.no_cpu and rank == 0 and world == 1
    # no cyclic garbage collection while GPU work is timed: a collection in the
    # host's enqueue path leaves the GPU idle between an event and the work it
    # brackets (single steps of up to ~1 ms were seen)
    gc.collect()
    gc.disable()
    result, dec, ids, tokens, sample, w = run_gpu(args, rank, world, want_cpu)
    if rank == 0:
        if not args.no_e2e and args.layers == 1:
            result["e2e"] = run_e2e(args, dec, ids, tokens, w)
        gc.enable()
        if sample is not None:
            result["cpu_baseline"] = cpu_baseline(sample, args.cpu_seconds)
        if args.comparator and args.layers == 1:
            result["dense_comparator"] = run_dense_comparator(args, dec, ids, w,
                                                              result["roofline"]["peak"])
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
