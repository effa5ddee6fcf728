"""ctypes binding of ``libpkv.so`` (the C ABI declared in ``include/pkv.h``).

Argument marshalling only: torch tensors become device pointers, the current
torch CUDA stream becomes the ``cudaStream_t`` argument, numpy arrays hold the
allocator's host outputs.  Every computation runs in the library's CUDA kernels
or in its C++ allocator; if the library has not been built this module raises
instead of falling back to anything else.
"""
import ctypes
import os

import numpy as np

from . import build as _build

OK, ERR_INVALID_ARG, ERR_OUT_OF_BLOCKS, ERR_UNKNOWN_SEQ, ERR_UNSUPPORTED, ERR_CUDA = range(6)
F32, BF16 = 0, 1
BLOCK_SIZE = 16
DEVERR_BAD_BLOCK, DEVERR_BAD_SLOT, DEVERR_BAD_LEN, DEVERR_TIMEOUT = 1, 2, 4, 8
DEVERR_BAD_PLAN = 16
PLAN_INTS = 24
ATTN_SIMT = 1
ATTN_SEPARATE_MERGE = 2
ATTN_SHORT_WAITS = 8
ATTN_CHECK_PLAN = 16
LAYERS_MERGE_HELPERS = 32
STEP_FUSED = 4

_c_i32 = ctypes.c_int32
_c_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_p_i32 = ctypes.POINTER(ctypes.c_int32)
_p_i64 = ctypes.POINTER(ctypes.c_int64)
_p_f32 = ctypes.POINTER(ctypes.c_float)
_size_t = ctypes.c_size_t


class PkvError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"pkv error {code}: {msg}")
        self.code = code


class OutOfBlocks(PkvError):
    pass


class UnknownSequence(PkvError):
    pass


class StepArgs(ctypes.Structure):
    _fields_ = [
        ("q", _vp), ("k", _vp), ("v", _vp),
        ("q_rot", _vp), ("k_rot", _vp),
        ("k_cache", _vp), ("v_cache", _vp),
        ("num_blocks", _c_i32),
        ("positions", _vp), ("slot_mapping", _vp), ("seq_lens", _vp),
        ("block_tables", _vp), ("bt_stride", _c_i32),
        ("attn_bias", _vp), ("bias_stride", _c_i32),
        ("B", _c_i32), ("Hq", _c_i32), ("Hkv", _c_i32), ("d", _c_i32),
        ("scale", ctypes.c_float), ("rope_base", ctypes.c_float),
        ("dtype", _c_i32), ("flags", _c_i32), ("num_parts", _c_i32),
        ("workspace", _vp), ("workspace_bytes", _size_t),
        ("out", _vp), ("dev_err_flag", _vp), ("plan", _vp),
    ]


class StepHostIO(ctypes.Structure):
    _fields_ = [
        ("q", _vp), ("k", _vp), ("v", _vp),
        ("positions", _vp), ("slot_mapping", _vp), ("seq_lens", _vp),
        ("block_tables", _vp), ("out", _vp), ("flags", _c_i32), ("plan", _vp),
    ]


class ServerDesc(ctypes.Structure):
    _fields_ = [
        ("step", StepArgs), ("alloc", _vp), ("rows", _vp),
        ("meta_host", _vp * 2), ("prefix_host", _vp * 2), ("max_prefix_tokens", _c_i32),
    ]


# name -> (restype, argtypes); every symbol declared in include/pkv.h
SIGNATURES = {
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_abi_version": (ctypes.c_int, []),
    "pkv_alloc_create": (ctypes.c_int, [_c_i32, _c_i32, _c_i32, _c_i32, _p_i32,
                                        ctypes.POINTER(_vp)]),
    "pkv_alloc_destroy": (None, [_vp]),
    "pkv_seq_join": (ctypes.c_int, [_vp, _c_i32, _p_i32]),
    "pkv_seq_leave": (ctypes.c_int, [_vp, _c_i32]),
    "pkv_seqs_join": (ctypes.c_int, [_vp, _p_i32, _c_i32, _p_i32, _p_i32, _p_i64]),
    "pkv_seqs_leave": (ctypes.c_int, [_vp, _p_i32, _c_i32]),
    "pkv_prepare_step": (ctypes.c_int, [_vp, _p_i32, _c_i32, _p_i32, _p_i64, _p_i32, _p_i32,
                                        _c_i32]),
    "pkv_prepare_step_cached": (ctypes.c_int, [_vp, _p_i32, _c_i32, _p_i32, _p_i64, _p_i32,
                                               _p_i32, _c_i32, _p_i32]),
    "pkv_seq_len": (ctypes.c_int, [_vp, _c_i32, _p_i32]),
    "pkv_seq_blocks": (ctypes.c_int, [_vp, _c_i32, _p_i32, _c_i32, _p_i32]),
    "pkv_seq_slots": (ctypes.c_int, [_vp, _c_i32, _c_i32, _c_i32, _p_i32, _p_i64]),
    "pkv_num_free": (ctypes.c_int, [_vp, _p_i32]),
    "pkv_pool_blocks": (ctypes.c_int, [ctypes.c_uint64, _c_i32, _c_i32, _c_i32, _c_i32, _p_i32]),
    "pkv_alloc_dump": (ctypes.c_int, [_vp, _p_i32, _c_i32, _p_i32]),
    "pkv_rope": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _c_i32, _c_i32, _c_i32, _c_i32,
                                ctypes.c_float, _c_i32, _vp]),
    "pkv_rope_append": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_i32,
                                       _c_i32, _c_i32, _c_i32, _c_i32, ctypes.c_float, _c_i32,
                                       _vp, _vp]),
    "pkv_append": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _c_i32, _c_i32, _c_i32, _c_i32,
                                  _c_i32, _vp, _vp]),
    "pkv_prefill_kv": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_i32, _c_i32, _c_i32,
                                      _c_i32, ctypes.c_float, _c_i32, _vp, _vp]),
    "pkv_attn_default_parts": (ctypes.c_int, [_c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _p_i32]),
    "pkv_attn_workspace_bytes": (ctypes.c_int, [_c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                                ctypes.POINTER(_size_t)]),
    "pkv_decode_attn_split": (ctypes.c_int, [_vp, _vp, _vp, _c_i32, _vp, _c_i32, _vp, _vp,
                                             _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                             ctypes.c_float, _c_i32, _vp, _size_t, _vp, _c_i32,
                                             _c_i32, _vp, _vp]),
    "pkv_decode_attn_static": (ctypes.c_int, [_vp, _vp, _vp, _c_i32, _vp, _c_i32, _vp, _vp,
                                              _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                              ctypes.c_float, _c_i32, _vp, _c_i32, _c_i32, _vp,
                                              _vp]),
    "pkv_plan_parts": (ctypes.c_int, [_p_i32, _c_i32, _c_i32, _c_i32, _p_i32, _c_i32, _c_i32,
                                      _c_i32, _p_i32]),
    "pkv_decode_attn_planned": (ctypes.c_int, [_vp, _vp, _vp, _c_i32, _vp, _c_i32, _vp, _vp,
                                               _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                               ctypes.c_float, _c_i32, _vp, _vp, _size_t, _vp,
                                               _c_i32, _c_i32, _vp, _vp]),
    "pkv_lse_merge": (ctypes.c_int, [_vp, _size_t, _vp, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32,
                                     _c_i32, _c_i32, _vp, _c_i32, _vp]),
    "pkv_decode_step": (ctypes.c_int, [ctypes.POINTER(StepArgs), _vp]),
    "pkv_mapped_pointer": (ctypes.c_int, [_vp, ctypes.POINTER(_vp)]),
    "pkv_decode_step_layers": (ctypes.c_int, [ctypes.POINTER(StepArgs), _c_i32, _vp]),
    "pkv_dense_assemble": (ctypes.c_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _p_i32,
                                          _c_i32, _c_i32, _vp, _vp, _c_i32, _c_i32, _c_i32,
                                          _c_i32, _vp]),
    "pkv_dense_extract": (ctypes.c_int, [_vp, _vp, _c_i32, _p_i32, _p_i32, _c_i32, _c_i32,
                                         _c_i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp),
                                         _c_i32, _c_i32, _c_i32, _vp]),
    "pkv_decode_step_host": (ctypes.c_int, [ctypes.POINTER(StepArgs),
                                            ctypes.POINTER(StepHostIO), _vp]),
    "pkv_step_graph_create": (ctypes.c_int, [ctypes.POINTER(StepArgs),
                                             ctypes.POINTER(StepHostIO), ctypes.POINTER(_vp)]),
    "pkv_step_graph_launch": (ctypes.c_int, [_vp, _vp]),
    "pkv_step_graph_enqueue": (ctypes.c_int, [_vp, _vp]),
    "pkv_step_graph_wait": (ctypes.c_int, [_vp]),
    "pkv_step_graph_destroy": (None, [_vp]),
    "pkv_server_meta_bytes": (_size_t, [_c_i32, _c_i32, _c_i32]),
    "pkv_server_prefix_bytes": (_size_t, [_c_i32]),
    "pkv_server_create": (ctypes.c_int, [ctypes.POINTER(ServerDesc), ctypes.POINTER(_vp)]),
    "pkv_server_step": (ctypes.c_int, [_vp, _p_i32, _p_i32, _c_i32, _vp, _vp, _vp, _vp, _vp,
                                       _vp]),
    "pkv_server_rows": (ctypes.c_int, [_vp, _p_i32]),
    "pkv_server_destroy": (None, [_vp]),
}

_LIB = None
ABI_VERSION = 5   # pkv_abi_version() of the library this binding describes


def library_path():
    return _build.LIB


def load():
    """Load the built library (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library {path} is missing: build it with "
            "`python -m paged_kv_decode_10_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.pkv_abi_version() != ABI_VERSION:
        raise RuntimeError(f"{path} has ABI version {lib.pkv_abi_version()}, this binding "
                           f"expects {ABI_VERSION}: rebuild it")
    _LIB = lib
    return lib


def _check(rc):
    if rc == OK:
        return
    msg = load().pkv_last_error().decode(errors="replace")
    if rc == ERR_OUT_OF_BLOCKS:
        raise OutOfBlocks(rc, msg)
    if rc == ERR_UNKNOWN_SEQ:
        raise UnknownSequence(rc, msg)
    raise PkvError(rc, msg)


# --------------------------------------------------------------------------
# host allocator
# --------------------------------------------------------------------------
_NP_OF = {ctypes.c_int32: np.int32, ctypes.c_int64: np.int64}


def _np_ptr(a, ctype, min_len=0):
    """Pointer to a numpy array the library reads or fills: the dtype must be
    the C type's, the array C-contiguous and at least ``min_len`` long (the C
    side writes through the pointer without knowing the array)."""
    if not isinstance(a, np.ndarray) or a.dtype != _NP_OF[ctype]:
        raise PkvError(ERR_INVALID_ARG, f"expected a numpy {np.dtype(_NP_OF[ctype])} array, "
                                        f"got {getattr(a, 'dtype', type(a))}")
    if not a.flags.c_contiguous or a.size < min_len:
        raise PkvError(ERR_INVALID_ARG, f"array must be C-contiguous with >= {min_len} entries")
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class BlockAllocator:
    """Host block allocator (C++); policy in ``include/pkv.h``."""

    def __init__(self, num_blocks, max_seqs, max_blocks_per_seq, initial_free=None):
        lib = load()
        handle = _vp()
        init = None
        if initial_free is not None:
            self._init = np.ascontiguousarray(initial_free, dtype=np.int32)
            init = _np_ptr(self._init, ctypes.c_int32)
        _check(lib.pkv_alloc_create(num_blocks, BLOCK_SIZE, max_seqs, max_blocks_per_seq, init,
                                    ctypes.byref(handle)))
        self._h = handle
        self._lib = lib
        self.num_blocks = num_blocks

    def close(self):
        if self._h:
            self._lib.pkv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def join(self, prefix_len):
        sid = ctypes.c_int32()
        _check(self._lib.pkv_seq_join(self._h, int(prefix_len), ctypes.byref(sid)))
        return sid.value

    def leave(self, seq_id):
        _check(self._lib.pkv_seq_leave(self._h, int(seq_id)))

    def join_many(self, prefix_lens, slots_out=None):
        """Joins one sequence per prefix length in one call (``pkv_seqs_join``);
        returns their ids.  ``slots_out = (positions, slot_mapping)``, arrays of at
        least sum(prefix_lens) entries, also receives every joiner's prefix
        positions and cache slots, packed in order."""
        lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
        ids = np.empty(len(lens), np.int32)
        pos = slots = None
        if slots_out is not None:
            n = int(lens.astype(np.int64).sum())
            pos = _np_ptr(slots_out[0], ctypes.c_int32, n)
            slots = _np_ptr(slots_out[1], ctypes.c_int64, n)
        _check(self._lib.pkv_seqs_join(self._h, _np_ptr(lens, ctypes.c_int32), len(lens),
                                       _np_ptr(ids, ctypes.c_int32), pos, slots))
        return ids

    def leave_many(self, seq_ids):
        """Retires the listed sequences in one call (``pkv_seqs_leave``)."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        _check(self._lib.pkv_seqs_leave(self._h, _np_ptr(ids, ctypes.c_int32), len(ids)))

    def prepare_step(self, seq_ids, bt_stride, out=None):
        """Returns ``positions, slot_mapping, seq_lens, block_tables`` (numpy).
        ``out`` may supply preallocated (e.g. pinned) arrays to fill."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        B = len(ids)
        if out is None:
            out = (np.empty(B, np.int32), np.empty(B, np.int64), np.empty(B, np.int32),
                   np.empty((B, bt_stride), np.int32))
        pos, slots, lens, tables = out
        _check(self._lib.pkv_prepare_step(self._h, _np_ptr(ids, ctypes.c_int32), B,
                                          _np_ptr(pos, ctypes.c_int32, B),
                                          _np_ptr(slots, ctypes.c_int64, B),
                                          _np_ptr(lens, ctypes.c_int32, B),
                                          _np_ptr(tables, ctypes.c_int32, B * int(bt_stride)),
                                          int(bt_stride)))
        return pos, slots, lens, tables

    def step_runner(self, seq_ids, bt_stride, out, row_state=None):
        """A no-argument callable that runs ``prepare_step`` for these sequence ids
        into the arrays ``out`` (positions, slot_mapping, seq_lens, block_tables),
        with every pointer converted once (a serving loop calls it every step).
        With ``row_state`` (int32 [B*3], -1 before the first call) it runs
        ``prepare_step_cached``: ``out`` must then be the same arrays every call."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        pos, slots, lens, tables = out
        h, B, bt = self._h, len(ids), int(bt_stride)
        ptrs = (_np_ptr(ids, ctypes.c_int32), _np_ptr(pos, ctypes.c_int32, B),
                _np_ptr(slots, ctypes.c_int64, B), _np_ptr(lens, ctypes.c_int32, B),
                _np_ptr(tables, ctypes.c_int32, B * bt))
        if row_state is None:
            fn, extra = self._lib.pkv_prepare_step, ()
        else:
            fn, extra = self._lib.pkv_prepare_step_cached, (_np_ptr(row_state, ctypes.c_int32,
                                                                    3 * B),)
        keep = (ids, out, row_state)
        args = (h, ptrs[0], B, ptrs[1], ptrs[2], ptrs[3], ptrs[4], bt) + extra

        def run():
            _check(fn(*args))
            return keep[1]
        return run

    def prepare_step_cached(self, seq_ids, bt_stride, out, row_state):
        """``pkv_prepare_step_cached`` into ``out`` (positions, slot_mapping,
        seq_lens, block_tables) with the caller-kept ``row_state`` (int32 [B*3])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        B = len(ids)
        pos, slots, lens, tables = out
        _check(self._lib.pkv_prepare_step_cached(
            self._h, _np_ptr(ids, ctypes.c_int32), B, _np_ptr(pos, ctypes.c_int32, B),
            _np_ptr(slots, ctypes.c_int64, B), _np_ptr(lens, ctypes.c_int32, B),
            _np_ptr(tables, ctypes.c_int32, B * int(bt_stride)), int(bt_stride),
            _np_ptr(row_state, ctypes.c_int32, 3 * B)))
        return out

    def seq_len(self, seq_id):
        n = ctypes.c_int32()
        _check(self._lib.pkv_seq_len(self._h, int(seq_id), ctypes.byref(n)))
        return n.value

    def seq_blocks(self, seq_id):
        n = ctypes.c_int32()
        _check(self._lib.pkv_seq_blocks(self._h, int(seq_id), None, 0, ctypes.byref(n)))
        buf = np.empty(n.value, np.int32)
        _check(self._lib.pkv_seq_blocks(self._h, int(seq_id), _np_ptr(buf, ctypes.c_int32),
                                        n.value, ctypes.byref(n)))
        return buf.tolist()

    def seq_slots(self, seq_id, start, count, out=None):
        """Positions and cache slots of tokens [start, start+count) of a live
        sequence (``pkv_seq_slots``); ``out`` may supply the two arrays."""
        if out is None:
            out = (np.empty(count, np.int32), np.empty(count, np.int64))
        pos, slots = out
        _check(self._lib.pkv_seq_slots(self._h, int(seq_id), int(start), int(count),
                                       _np_ptr(pos, ctypes.c_int32, int(count)),
                                       _np_ptr(slots, ctypes.c_int64, int(count))))
        return pos, slots

    def num_free(self):
        n = ctypes.c_int32()
        _check(self._lib.pkv_num_free(self._h, ctypes.byref(n)))
        return n.value

    def free_stack(self):
        n = ctypes.c_int32()
        _check(self._lib.pkv_alloc_dump(self._h, None, 0, ctypes.byref(n)))
        buf = np.empty(n.value, np.int32)
        _check(self._lib.pkv_alloc_dump(self._h, _np_ptr(buf, ctypes.c_int32), n.value,
                                        ctypes.byref(n)))
        return buf.tolist()


# --------------------------------------------------------------------------
# device calls (torch tensors in, torch tensors out)
# --------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise PkvError(ERR_UNSUPPORTED, f"dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise PkvError(ERR_INVALID_ARG, "tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise PkvError(ERR_INVALID_ARG, "tensor must be contiguous")
    return _vp(t.data_ptr())


def mapped_pointer(t):
    """Device-side address of a contiguous pinned CPU tensor (``pkv_mapped_pointer``)."""
    if t.is_cuda or not t.is_pinned():
        raise PkvError(ERR_INVALID_ARG, "tensor must be in pinned host memory")
    if not t.is_contiguous():
        raise PkvError(ERR_INVALID_ARG, "tensor must be contiguous")
    out = _vp()
    _check(load().pkv_mapped_pointer(_vp(t.data_ptr()), ctypes.byref(out)))
    return out


def _meta_ptr(t):
    """Step metadata may be a device tensor or a pinned host tensor the kernels
    read in place."""
    if t is not None and not t.is_cuda:
        return mapped_pointer(t)
    return _ptr(t)


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return _vp(s.cuda_stream)


def rope(q, k, positions, base=10000.0, q_out=None, k_out=None, stream=None):
    """a1: rotate-half RoPE of ``q [B,Hq,d]`` and ``k [B,Hkv,d]`` at ``positions [B]`` (int32)."""
    torch = _torch()
    q_out = torch.empty_like(q) if q_out is None else q_out
    k_out = torch.empty_like(k) if k_out is None else k_out
    B, Hq, d = q.shape
    _check(load().pkv_rope(_ptr(q), _ptr(k), _ptr(q_out), _ptr(k_out), _meta_ptr(positions), B, Hq,
                           k.shape[1], d, float(base), dtype_code(q), _stream(stream)))
    return q_out, k_out


def rope_append(q, k, v, positions, slot_mapping, k_cache, v_cache, base=10000.0, q_out=None,
                k_out=None, err=None, stream=None):
    """a1 + a2 fused: rotate q/k and write the rotated k and raw v into the cache slots."""
    torch = _torch()
    q_out = torch.empty_like(q) if q_out is None else q_out
    k_out = torch.empty_like(k) if k_out is None else k_out
    B, Hq, d = q.shape
    _check(load().pkv_rope_append(_ptr(q), _ptr(k), _ptr(v), _ptr(q_out), _ptr(k_out),
                                  _meta_ptr(positions), _meta_ptr(slot_mapping), _ptr(k_cache),
                                  _ptr(v_cache), B, Hq, k.shape[1], d, k_cache.shape[0],
                                  float(base), dtype_code(q), _ptr(err), _stream(stream)))
    return q_out, k_out


def prefill_kv(k, v, positions, slot_mapping, k_cache, v_cache, base=10000.0, err=None,
               stream=None):
    """Prefix KV of joining sequences: rotate ``k [T,Hkv,d]`` at ``positions [T]``
    and write it and ``v`` into ``slot_mapping [T]`` of the caches."""
    T, Hkv, d = k.shape
    _check(load().pkv_prefill_kv(_ptr(k), _ptr(v), _meta_ptr(positions),
                                 _meta_ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), T, Hkv,
                                 d, k_cache.shape[0], float(base), dtype_code(k), _ptr(err),
                                 _stream(stream)))


def append(k_rot, v, slot_mapping, k_cache, v_cache, err=None, stream=None):
    """a2: write ``k_rot``/``v`` ``[B,Hkv,d]`` into cache slots ``slot_mapping [B]`` (int64)."""
    B, Hkv, d = k_rot.shape
    _check(load().pkv_append(_ptr(k_rot), _ptr(v), _meta_ptr(slot_mapping), _ptr(k_cache),
                             _ptr(v_cache), B, Hkv, d, k_cache.shape[0], dtype_code(k_rot),
                             _ptr(err), _stream(stream)))


def default_parts(d, dtype, flags=0, Hq=32, Hkv=8):
    n = ctypes.c_int32()
    _check(load().pkv_attn_default_parts(d, Hq, Hkv, dtype, flags, ctypes.byref(n)))
    return n.value


def workspace_bytes(B, Hq, Hkv, d, num_parts):
    n = _size_t()
    _check(load().pkv_attn_workspace_bytes(B, Hq, Hkv, d, num_parts, ctypes.byref(n)))
    return n.value


def alloc_workspace(B, Hq, Hkv, d, num_parts, device=None):
    torch = _torch()
    nbytes = workspace_bytes(B, Hq, Hkv, d, num_parts)
    # zero-filled once: the fused merge's counters start (and stay) at zero
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device or "cuda")


def decode_attn_split(q_rot, k_cache, v_cache, block_tables, seq_lens, scale, num_parts,
                      workspace, out, attn_bias=None, flags=0, err=None, stream=None):
    """a3: split-KV paged GQA attention (fills ``out`` for single-part units and
    the workspace partials for the rest)."""
    B, Hq, d = q_rot.shape
    Hkv = k_cache.shape[1]
    bias_stride = attn_bias.shape[1] if attn_bias is not None else 0
    _check(load().pkv_decode_attn_split(
        _ptr(q_rot), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _meta_ptr(block_tables),
        block_tables.shape[1], _meta_ptr(seq_lens), _ptr(attn_bias), bias_stride, B, Hq, Hkv, d,
        float(scale), int(num_parts), _ptr(workspace), workspace.numel(), _ptr(out),
        dtype_code(q_rot), int(flags), _ptr(err), _stream(stream)))


def plan_parts(seq_lens, Hkv, d, block_tables, num_parts, bias_stride=0, out=None):
    """Host-planned partition (``pkv_plan_parts``) of numpy step metadata:
    ``seq_lens int32 [B]``, ``block_tables int32 [B, bt_stride]``; returns (or
    fills) ``int32 [num_parts, PLAN_INTS]``."""
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    B = len(lens)
    if tables.ndim != 2 or tables.shape[0] != B:
        raise PkvError(ERR_INVALID_ARG, "block_tables must be [B, bt_stride]")
    if out is None:
        out = np.empty((num_parts, PLAN_INTS), np.int32)
    _check(load().pkv_plan_parts(_np_ptr(lens, ctypes.c_int32), B, int(Hkv), int(d),
                                 _np_ptr(tables, ctypes.c_int32), tables.shape[1],
                                 int(bias_stride), int(num_parts),
                                 _np_ptr(out, ctypes.c_int32, num_parts * PLAN_INTS)))
    return out


def plan_runner(seq_lens, block_tables, Hkv, d, num_parts, out, bias_stride=0):
    """A no-argument callable running ``pkv_plan_parts`` on these (fixed)
    numpy arrays into ``out`` with every pointer converted once, for a loop
    that re-plans every step after a0 rewrote the arrays in place."""
    fn = load().pkv_plan_parts
    B, bt = len(seq_lens), block_tables.shape[1]
    ptrs = (_np_ptr(seq_lens, ctypes.c_int32, B), _np_ptr(block_tables, ctypes.c_int32, B * bt),
            _np_ptr(out, ctypes.c_int32, num_parts * PLAN_INTS))
    args = (ptrs[0], B, int(Hkv), int(d), ptrs[1], bt, int(bias_stride), int(num_parts), ptrs[2])
    keep = (seq_lens, block_tables, out)

    def run():
        _check(fn(*args))
        return keep[2]
    return run


def decode_attn_planned(q_rot, k_cache, v_cache, block_tables, seq_lens, scale, num_parts, plan,
                        workspace, out, attn_bias=None, flags=0, err=None, stream=None):
    """a3 with a host-planned partition (``plan``: device or pinned int32
    ``[num_parts, PLAN_INTS]`` tensor from ``plan_parts``)."""
    B, Hq, d = q_rot.shape
    Hkv = k_cache.shape[1]
    bias_stride = attn_bias.shape[1] if attn_bias is not None else 0
    _check(load().pkv_decode_attn_planned(
        _ptr(q_rot), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _meta_ptr(block_tables),
        block_tables.shape[1], _meta_ptr(seq_lens), _ptr(attn_bias), bias_stride, B, Hq, Hkv, d,
        float(scale), int(num_parts), _meta_ptr(plan), _ptr(workspace), workspace.numel(),
        _ptr(out), dtype_code(q_rot), int(flags), _ptr(err), _stream(stream)))


def decode_attention_static(q_rot, k_cache, v_cache, block_tables, seq_lens, scale, out,
                            num_parts=0, attn_bias=None, flags=0, err=None, stream=None):
    """a3 + fused a4 with the library's built-in scratch array instead of a
    workspace, for callers that cannot allocate device memory (see
    ``pkv_decode_attn_static`` in ``include/pkv.h``)."""
    B, Hq, d = q_rot.shape
    Hkv = k_cache.shape[1]
    bias_stride = attn_bias.shape[1] if attn_bias is not None else 0
    _check(load().pkv_decode_attn_static(
        _ptr(q_rot), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _meta_ptr(block_tables),
        block_tables.shape[1], _meta_ptr(seq_lens), _ptr(attn_bias), bias_stride, B, Hq, Hkv, d,
        float(scale), int(num_parts), _ptr(out), dtype_code(q_rot), int(flags), _ptr(err),
        _stream(stream)))
    return out


def lse_merge(workspace, seq_lens, bt_stride, B, Hq, Hkv, d, num_parts, out, bias_stride=0,
              stream=None):
    """a4: LSE merge of the split partials into ``out``."""
    _check(load().pkv_lse_merge(_ptr(workspace), workspace.numel(), _meta_ptr(seq_lens),
                                int(bt_stride), int(bias_stride), B, Hq, Hkv, d, int(num_parts),
                                _ptr(out), dtype_code(out), _stream(stream)))


def decode_attention(q_rot, k_cache, v_cache, block_tables, seq_lens, scale, num_parts=None,
                     workspace=None, out=None, attn_bias=None, flags=0, err=None, stream=None,
                     plan=None):
    """a3 + a4: returns ``out [B,Hq,d]`` (with ``plan``, through the host-planned
    partition; ``num_parts`` must then be the plan's)."""
    torch = _torch()
    B, Hq, d = q_rot.shape
    Hkv = k_cache.shape[1]
    if num_parts is None:
        num_parts = default_parts(d, dtype_code(q_rot), flags, Hq, Hkv)
    if workspace is None:
        workspace = alloc_workspace(B, Hq, Hkv, d, num_parts, q_rot.device)
    if out is None:
        out = torch.empty_like(q_rot)
    if plan is not None:
        decode_attn_planned(q_rot, k_cache, v_cache, block_tables, seq_lens, scale, num_parts,
                            plan, workspace, out, attn_bias, flags, err, stream)
    else:
        decode_attn_split(q_rot, k_cache, v_cache, block_tables, seq_lens, scale, num_parts,
                          workspace, out, attn_bias, flags, err, stream)
    if flags & ATTN_SEPARATE_MERGE:
        lse_merge(workspace, seq_lens, block_tables.shape[1], B, Hq, Hkv, d, num_parts, out,
                  attn_bias.shape[1] if attn_bias is not None else 0, stream)
    return out


def make_step_args(q, k, v, q_rot, k_rot, k_cache, v_cache, positions, slot_mapping, seq_lens,
                   block_tables, scale, rope_base, num_parts, workspace, out, attn_bias=None,
                   flags=0, err=None, plan=None):
    """Fills the ``pkv_step_args`` struct.  All tensors are on the device except
    that q, k, v, positions, slot_mapping, seq_lens and block_tables may be pinned
    host tensors, which the kernels then read in place, and out may be a pinned
    host tensor, which the kernels then write in place."""
    a = StepArgs()
    a.q, a.k, a.v = _meta_ptr(q), _meta_ptr(k), _meta_ptr(v)
    a.q_rot, a.k_rot = _ptr(q_rot), _ptr(k_rot)
    a.k_cache, a.v_cache = _ptr(k_cache), _ptr(v_cache)
    a.num_blocks = k_cache.shape[0]
    a.positions, a.slot_mapping = _meta_ptr(positions), _meta_ptr(slot_mapping)
    a.seq_lens = _meta_ptr(seq_lens)
    a.block_tables, a.bt_stride = _meta_ptr(block_tables), block_tables.shape[1]
    a.attn_bias = _ptr(attn_bias)
    a.bias_stride = attn_bias.shape[1] if attn_bias is not None else 0
    a.B, a.Hq, a.d = q.shape
    a.Hkv = k.shape[1]
    a.scale, a.rope_base = float(scale), float(rope_base)
    a.dtype, a.flags, a.num_parts = dtype_code(q), int(flags), int(num_parts)
    a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel()
    a.out = _meta_ptr(out)
    a.dev_err_flag = _ptr(err)
    a.plan = _meta_ptr(plan)
    return a


def decode_step_args(args, stream=None):
    """Runs a1 -> a4 from a prepared ``StepArgs``."""
    _check(load().pkv_decode_step(ctypes.byref(args), _stream(stream)))


def layer_args_array(layers):
    """A ctypes array of ``StepArgs``, one per layer, for ``decode_step_layers``."""
    arr = (StepArgs * len(layers))()
    for i, a in enumerate(layers):
        arr[i] = a
    return arr


def decode_step_layers(layers, stream=None):
    """One decode step through every layer (``pkv_decode_step_layers``);
    ``layers`` is a list of ``StepArgs`` or an array from ``layer_args_array``."""
    arr = layers if isinstance(layers, ctypes.Array) else layer_args_array(layers)
    _check(load().pkv_decode_step_layers(arr, len(arr), _stream(stream)))


def _ptr_array(tensors):
    arr = (_vp * max(len(tensors), 1))()
    for i, t in enumerate(tensors):
        arr[i] = _ptr(t)
    return arr


def dense_assemble(k_snaps, v_snaps, lens, padded_len, k_dense, v_dense, cap, stream=None):
    """Right-padded dense batch from per-sequence snapshots (``pkv_dense_assemble``).
    Snapshots and the dense caches use the block layout ``[blocks, Hkv, 16, d]``;
    the dense batch has ``cap`` tokens per row."""
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    if not len(k_snaps) == len(v_snaps) == len(lens):
        raise PkvError(ERR_INVALID_ARG, "one K and one V snapshot per length")
    Hkv, d = k_dense.shape[1], k_dense.shape[3]
    _check(load().pkv_dense_assemble(_ptr_array(k_snaps), _ptr_array(v_snaps),
                                     _np_ptr(lens, ctypes.c_int32), len(lens), int(padded_len),
                                     _ptr(k_dense), _ptr(v_dense), int(cap), Hkv, d,
                                     dtype_code(k_dense), _stream(stream)))


def dense_extract(k_dense, v_dense, cap, rows, prefix_lens, padded_len, steps, k_snaps, v_snaps,
                  stream=None):
    """Rows of a dense batch back into snapshots: prefix plus decode columns
    (``pkv_dense_extract``)."""
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    prefix_lens = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    if not len(prefix_lens) == len(k_snaps) == len(v_snaps) == len(rows):
        raise PkvError(ERR_INVALID_ARG, "one prefix length and K/V snapshot per row")
    Hkv, d = k_dense.shape[1], k_dense.shape[3]
    _check(load().pkv_dense_extract(_ptr(k_dense), _ptr(v_dense), int(cap),
                                    _np_ptr(rows, ctypes.c_int32),
                                    _np_ptr(prefix_lens, ctypes.c_int32), len(rows),
                                    int(padded_len), int(steps), _ptr_array(k_snaps),
                                    _ptr_array(v_snaps), Hkv, d, dtype_code(k_dense),
                                    _stream(stream)))


def pool_blocks(budget_bytes, n_layers, Hkv, d, dtype):
    """Blocks of a K/V pool for ``n_layers`` layers that fit in ``budget_bytes``."""
    n = ctypes.c_int32()
    _check(load().pkv_pool_blocks(int(budget_bytes), int(n_layers), int(Hkv), int(d),
                                  int(dtype), ctypes.byref(n)))
    return n.value


def decode_step_host(args, host_io, stream=None):
    """End-to-end step from host buffers (see ``pkv_decode_step_host``)."""
    _check(load().pkv_decode_step_host(ctypes.byref(args), ctypes.byref(host_io),
                                       _stream(stream)))


HOST_IN_PLACE = 1


class StepGraph:
    """``pkv_step_graph``: the host step for fixed buffers captured once;
    ``launch()`` runs one step and waits for its output in host memory."""

    def __init__(self, args, io):
        self._lib = load()
        self._keep = (args, io)
        h = _vp()
        _check(self._lib.pkv_step_graph_create(ctypes.byref(args), ctypes.byref(io),
                                               ctypes.byref(h)))
        self._h = h

    def launch(self, stream=None):
        _check(self._lib.pkv_step_graph_launch(self._h, _stream(stream)))

    def enqueue(self, stream=None):
        """The launch without the wait (``wait`` waits for the last one)."""
        _check(self._lib.pkv_step_graph_enqueue(self._h, _stream(stream)))

    def wait(self):
        """Waits for this graph's last ``enqueue`` (its output is then set)."""
        _check(self._lib.pkv_step_graph_wait(self._h))

    def close(self):
        if self._h:
            self._lib.pkv_step_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def host_io(q, k, v, positions, slot_mapping, seq_lens, block_tables, out, flags=0, plan=None):
    """``pkv_step_host_io`` over host (CPU, ideally pinned; pinned for
    ``HOST_IN_PLACE``) torch tensors."""
    io = StepHostIO()
    io.flags = int(flags)
    for name, t in (("q", q), ("k", k), ("v", v), ("positions", positions),
                    ("slot_mapping", slot_mapping), ("seq_lens", seq_lens),
                    ("block_tables", block_tables), ("out", out), ("plan", plan)):
        if t is None and name == "plan":
            continue
        if t.is_cuda or not t.is_contiguous():
            raise PkvError(ERR_INVALID_ARG, f"{name} must be a contiguous host tensor")
        setattr(io, name, _vp(t.data_ptr()))
    return io


class Server:
    """The native serving loop (``pkv_server``) over a single-layer
    ``engine.PagedDecoder``'s device buffers for the sequences ``rows`` (one
    per row); joins and leaves then go through ``step``.  Holds the pinned host
    buffers the server needs."""

    def __init__(self, dec, rows, max_prefix_tokens):
        torch = _torch()
        lib = load()
        B = len(rows)
        self.B, self._lib = B, lib
        nb = lib.pkv_server_meta_bytes(B, dec.bt_stride, dec.num_parts)
        pb = lib.pkv_server_prefix_bytes(int(max_prefix_tokens))
        self.meta = [torch.empty(nb, dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.prefix = [torch.empty(max(pb, 16), dtype=torch.uint8).pin_memory() for _ in range(2)]
        self.rows_in = np.ascontiguousarray(rows, dtype=np.int32)
        step = make_step_args(dec.q_in[:B], dec.k_in[:B], dec.v_in[:B], dec.q_rot[:B],
                              dec.k_rot[:B], dec.k_cache, dec.v_cache, dec.positions[:B],
                              dec.slots[:B], dec.seq_lens[:B], dec.tables[:B], dec.scale,
                              dec.rope_base, dec.num_parts, dec.workspace, dec.out[:B],
                              flags=dec.flags, err=dec.err)
        self.desc = ServerDesc()
        self.desc.step = step
        self.desc.alloc = dec.alloc._h
        self.desc.rows = self.rows_in.ctypes.data_as(_vp)
        for t in range(2):
            self.desc.meta_host[t] = _vp(self.meta[t].data_ptr())
            self.desc.prefix_host[t] = _vp(self.prefix[t].data_ptr())
        self.desc.max_prefix_tokens = int(max_prefix_tokens)
        h = _vp()
        _check(lib.pkv_server_create(ctypes.byref(self.desc), ctypes.byref(h)))
        self._h = h

    def step(self, leave_rows, prefix_lens, prefix_k=None, prefix_v=None, q=None, k=None,
             v=None, stream=None):
        """One step (see ``pkv_server_step``); leave_rows and prefix_lens are
        int32 numpy arrays of the same length."""
        lr = np.ascontiguousarray(leave_rows, dtype=np.int32)
        pl = np.ascontiguousarray(prefix_lens, dtype=np.int32)
        if len(lr) != len(pl):
            raise PkvError(ERR_INVALID_ARG, "one prefix length per leaving row")
        _check(self._lib.pkv_server_step(
            self._h, _np_ptr(lr, ctypes.c_int32), _np_ptr(pl, ctypes.c_int32), len(lr),
            _ptr(prefix_k), _ptr(prefix_v), _ptr(q), _ptr(k), _ptr(v), _stream(stream)))

    def step_runner(self, leave_rows, prefix_lens, prefix_k=None, prefix_v=None, q=None, k=None,
                    v=None, stream=None):
        """A no-argument callable running this step with every argument
        converted once (a loop that replays a planned schedule)."""
        lr = np.ascontiguousarray(leave_rows, dtype=np.int32)
        pl = np.ascontiguousarray(prefix_lens, dtype=np.int32)
        if len(lr) != len(pl):
            raise PkvError(ERR_INVALID_ARG, "one prefix length per leaving row")
        args = (self._h, _np_ptr(lr, ctypes.c_int32), _np_ptr(pl, ctypes.c_int32), len(lr),
                _ptr(prefix_k), _ptr(prefix_v), _ptr(q), _ptr(k), _ptr(v), _stream(stream))
        fn, keep = self._lib.pkv_server_step, (lr, pl, prefix_k, prefix_v, q, k, v)

        def run():
            _check(fn(*args))
            return keep
        return run

    def rows(self):
        out = np.empty(self.B, np.int32)
        _check(self._lib.pkv_server_rows(self._h, _np_ptr(out, ctypes.c_int32, self.B)))
        return out

    def close(self):
        if self._h:
            self._lib.pkv_server_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
