/*
 * pkv.h -- C ABI of the paged-KV continuous-batching decode step (GB300, sm_103a).
 *
 * One decode step appends one token to every row of a batch and attends over
 * each row's cached keys/values.  It has four device parts and one host part:
 *
 *   a0  host block allocator: positions, slot_mapping, seq_lens, block tables
 *   a1  pkv_rope               rotate-half RoPE of the new q and k at per-row positions
 *   a2  pkv_append             write rotated k and raw v into the cache slot
 *   a3  pkv_decode_attn_split  grouped-query attention through block tables,
 *                              split over a page-balanced partition, online softmax
 *   a4  pkv_lse_merge          log-sum-exp merge of the split partials
 *
 * Sources: "neurogrid releases" v0.7.0 (paged KV cache in fixed 16-token blocks,
 * O(1) block allocator with per-sequence block tables, paged attention with GQA),
 * v0.6.0 (flash decode: online softmax over KV tiles), v0.8.0 (kv_len =
 * position + 1 computed on the GPU, zero device-to-host copies, every kernel on
 * one caller stream); helexa issue 121 "continuous batching -- batched decode +
 * engine", slice 1 (per-row RoPE positions, rotate-half, keys stored post-RoPE,
 * additive (B,1,1,S) mask over each row's padding gap); "cortex-engine writeup",
 * block-sparse attention kernel (a row with zero softmax denominator outputs
 * zeros instead of NaN).
 *
 * Conventions
 *  - Every call returns PKV_OK (0) or a PKV_ERR_* code; pkv_last_error()
 *    returns a message for the calling thread's last failure.
 *  - The library never allocates device memory.  The caller owns every device
 *    buffer and the CUDA stream.  Device calls are asynchronous on `stream`
 *    (a cudaStream_t passed as void*, NULL = legacy default stream), make no
 *    device-to-host copy (the host-step calls at the end of this header are
 *    the exception: they return the result in host memory) and check
 *    cudaGetLastError after each launch.
 *  - Every tensor is dense and row-major in the layout stated.  dtype is
 *    PKV_F32 or PKV_BF16 and applies to q, k, v, the caches and the output.
 *  - dev_err_flag (nullable, device int32): kernels that meet an out-of-range
 *    block id, slot or length atomically OR a PKV_DEVERR_* bit into it and skip
 *    that access instead of faulting.  The caller clears it.
 *  - The allocator is host-only and not thread-safe: one owner per allocator.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG 1   /* null pointer, bad size, bad stride, duplicate row */
#define PKV_ERR_OUT_OF_BLOCKS 2 /* the free list cannot satisfy the request; nothing changed */
#define PKV_ERR_UNKNOWN_SEQ 3   /* sequence id not live */
#define PKV_ERR_UNSUPPORTED 4   /* dtype, head_dim, group size or block size not built */
#define PKV_ERR_CUDA 5          /* a CUDA runtime/driver call failed; see pkv_last_error */

#define PKV_F32 0
#define PKV_BF16 1

#define PKV_BLOCK_SIZE 16       /* tokens per KV block ("neurogrid releases" v0.7.0) */

/* bits OR-ed into dev_err_flag */
#define PKV_DEVERR_BAD_BLOCK 1  /* a block table entry outside [0, num_blocks) */
#define PKV_DEVERR_BAD_SLOT 2   /* a slot outside [0, num_blocks * 16) */
#define PKV_DEVERR_BAD_LEN 4    /* seq_len < 0, or longer than bt_stride*16 or bias_stride */
#define PKV_DEVERR_TIMEOUT 8    /* an internal pipeline wait gave up (never expected) */
#define PKV_DEVERR_BAD_PLAN 16  /* PKV_ATTN_CHECK_PLAN: the plan disagrees with the metadata */

/* flags for the attention calls */
#define PKV_ATTN_SIMT 1         /* use the CUDA-core consumer instead of mma.sync (bf16 only;
                                   f32 always uses CUDA cores) */
#define PKV_ATTN_SEPARATE_MERGE 2 /* leave the split partials for pkv_lse_merge instead of
                                     merging them in the split kernel's epilogue */
#define PKV_STEP_FUSED 4          /* pkv_decode_step: run a1+a2 inside the attention kernel
                                     (one launch per step) instead of as their own kernel */
#define PKV_ATTN_SHORT_WAITS 8    /* diagnostic: every wait inside the attention kernel gives
                                     up after ~64 SM clocks instead of ~1 s, so the timeout
                                     path can be exercised (PKV_DEVERR_TIMEOUT is set, the
                                     output is incomplete, every copy the kernel issued still
                                     lands before it exits); the workspace must be zero-filled
                                     again before its next use */
#define PKV_ATTN_CHECK_PLAN 16    /* with a plan: also derive the partition from the metadata
                                     in the kernel, set PKV_DEVERR_BAD_PLAN where the plan
                                     disagrees and use the derived one there */
#define PKV_LAYERS_MERGE_HELPERS 32 /* pkv_decode_step_layers: launch each layer's attention
                                     kernel cooperatively, so that the merge of a unit split
                                     over many parts is shared by its last parts as in a
                                     single-layer call (otherwise its last part merges it
                                     alone).  Worth it for long rows; the next layer's
                                     attention kernel then starts only once the previous one
                                     has left the GPU.  Ignored by the other calls. */

/* Message for the calling thread's last failed call ("" if none). */
const char *pkv_last_error(void);
/* ABI version of this header (bumped on any signature change). */
int pkv_abi_version(void);

/* ======================================================================== */
/* a0: host block allocator                                                  */
/* ======================================================================== */
/*
 * Policy ("neurogrid releases" v0.7.0: constant-time block allocation and
 * release, one block table per sequence; v0.8.0: kv_len = position + 1):
 *  - The free list is a stack, seeded bottom-to-top with `initial_free` (a
 *    permutation of 0..num_blocks-1; NULL = 0,1,2,...).  Pop takes the top.
 *  - join pops ceil(prefix_len/16) blocks in table order and takes the
 *    smallest free sequence id; leave pushes the sequence's blocks in table
 *    order and frees its id.
 *  - prepare_step appends one token to each listed sequence: position = L
 *    (cached length before the step); if L % 16 == 0 a block is popped first;
 *    slot = table[L/16]*16 + L%16; the length becomes L+1.
 *  - A request that cannot be met returns PKV_ERR_OUT_OF_BLOCKS and changes
 *    nothing.  Each pop/push is O(1).
 */
typedef struct pkv_alloc pkv_alloc;

/* block_size must be 16.  max_blocks_per_seq bounds each block table.
 * On success *out owns the allocator (free with pkv_alloc_destroy). */
int pkv_alloc_create(int32_t num_blocks, int32_t block_size, int32_t max_seqs,
                     int32_t max_blocks_per_seq, const int32_t *initial_free,
                     pkv_alloc **out);
void pkv_alloc_destroy(pkv_alloc *a);

/* A new sequence whose first prefix_len tokens are already in its blocks
 * (their contents are written by the caller, e.g. by a prefill). */
int pkv_seq_join(pkv_alloc *a, int32_t prefix_len, int32_t *seq_id);
int pkv_seq_leave(pkv_alloc *a, int32_t seq_id);

/* Several joins in one call (one host call per step for a serving loop that
 * admits many sequences): the same as pkv_seq_join(prefix_lens[i]) for i = 0..n-1
 * in order, into seq_ids[i].  If positions and slot_mapping are given they receive,
 * packed one sequence after another, the positions and cache slots of every
 * joiner's prefix tokens [0, prefix_lens[i]) (sum(prefix_lens) entries, as
 * pkv_seq_slots gives them): the input of pkv_prefill_kv.  All or nothing: if
 * the sequence ids, the pool or a table cannot take every joiner, nothing
 * changes (PKV_ERR_OUT_OF_BLOCKS when the pool is short). */
int pkv_seqs_join(pkv_alloc *a, const int32_t *prefix_lens, int32_t n, int32_t *seq_ids,
                  int32_t *positions, int64_t *slot_mapping);
/* Several leaves in one call: pkv_seq_leave(seq_ids[i]) for i = 0..n-1 in order.
 * All or nothing: every id must be live and listed once, else nothing changes. */
int pkv_seqs_leave(pkv_alloc *a, const int32_t *seq_ids, int32_t n);

/*
 * Host part of one decode step for the B listed (distinct, live) sequences.
 * Outputs (host arrays, row b = seq_ids[b]):
 *   positions[B]      int32  position of the new token (= cached length before)
 *   slot_mapping[B]   int64  cache slot of the new token
 *   seq_lens[B]       int32  length after the append (what attention reads)
 *   block_tables[B*bt_stride] int32, row-major, padded with -1
 * Atomic: on any error nothing changes.
 */
int pkv_prepare_step(pkv_alloc *a, const int32_t *seq_ids, int32_t B,
                     int32_t *positions, int64_t *slot_mapping, int32_t *seq_lens,
                     int32_t *block_tables, int32_t bt_stride);
/* The same step, for a block_tables buffer that is rewritten step after step:
 * row_state (int32 [B*3], all -1 before the first call on a fresh buffer, then
 * kept by the caller with that buffer) records which sequence, join and table
 * length each row of the buffer holds, and only the entries that differ are
 * written (a row whose sequence stayed gets just its new blocks; a row that
 * changed sequence is rewritten and its stale entries set to -1).  The buffer
 * then holds exactly what pkv_prepare_step would have written.  Every output
 * and all allocator state are the same as pkv_prepare_step's. */
int pkv_prepare_step_cached(pkv_alloc *a, const int32_t *seq_ids, int32_t B,
                            int32_t *positions, int64_t *slot_mapping, int32_t *seq_lens,
                            int32_t *block_tables, int32_t bt_stride, int32_t *row_state);

int pkv_seq_len(const pkv_alloc *a, int32_t seq_id, int32_t *len);
/* Copies up to cap block ids of the sequence's table into out; *n = table length. */
int pkv_seq_blocks(const pkv_alloc *a, int32_t seq_id, int32_t *out, int32_t cap,
                   int32_t *n);
/* Positions and cache slots of tokens [start, start+count) of a live sequence
 * (already covered by its blocks: start+count <= its length), for writing a
 * prefix chunk with pkv_prefill_kv.  positions[i] = start+i,
 * slot_mapping[i] = table[p/16]*16 + p%16.  PKV_ERR_INVALID_ARG if the range
 * is negative or beyond the length; nothing is changed. */
int pkv_seq_slots(const pkv_alloc *a, int32_t seq_id, int32_t start, int32_t count,
                  int32_t *positions, int64_t *slot_mapping);
int pkv_num_free(const pkv_alloc *a, int32_t *n);
/* Pool auto-sizing ("neurogrid releases" v0.7.0: the pool is sized from the
 * VRAM budget): the number of 16-token blocks whose K and V, for every KV head
 * and every one of n_layers layers, fit in budget_bytes (floor; host only). */
int pkv_pool_blocks(uint64_t budget_bytes, int32_t n_layers, int32_t Hkv, int32_t d,
                    int32_t dtype, int32_t *num_blocks);
/* Copies the free stack bottom-to-top (up to cap entries); *n = its size. */
int pkv_alloc_dump(const pkv_alloc *a, int32_t *free_stack, int32_t cap, int32_t *n);

/* Device calls.  Tensors are device memory, except that the integer index
 * arrays (positions, slot_mapping, seq_lens, block_tables) -- and the new q, k,
 * v of pkv_decode_step -- may instead be page-locked host memory at its mapped
 * address (pkv_mapped_pointer): the kernels then read them in place over the
 * CPU-GPU link, and the host must not rewrite them until those kernels have
 * finished.  All calls are asynchronous
 * on `stream` (a cudaStream_t; NULL = the legacy default stream). */

/* ======================================================================== */
/* a1: RoPE (helexa issue 121, slice 1: batch_cos_sin at per-row positions,   */
/*     rotate-half apply)                                                    */
/* ======================================================================== */
/*
 * q [B,Hq,d], k [B,Hkv,d] -> q_out [B,Hq,d], k_out [B,Hkv,d] (device, dtype).
 * For pair i < d/2 at position p = positions[b]:
 *   theta = p * base^(-2i/d)
 *   out[i]     = x[i] cos(theta) - x[i+d/2] sin(theta)
 *   out[i+d/2] = x[i+d/2] cos(theta) + x[i] sin(theta)
 * theta is formed modulo 2*pi exactly (64-bit fixed-point turns from a
 * double-precision host table), then rotated in float32 and rounded once to
 * dtype.  In-place (q_out == q) is allowed.
 * d even, 2 <= d <= 256.
 */
int pkv_rope(const void *q, const void *k, void *q_out, void *k_out,
             const int32_t *positions, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
             float base, int32_t dtype, void *stream);

/* ======================================================================== */
/* a2: append ("neurogrid releases" v0.7.0: fixed 16-token blocks)           */
/* ======================================================================== */
/*
 * k_cache, v_cache: [num_blocks, Hkv, 16, d] (device, dtype).
 * For each row b with slot = slot_mapping[b] >= 0:
 *   k_cache[slot/16, h, slot%16, :] = k_rot[b, h, :]
 *   v_cache[slot/16, h, slot%16, :] = v[b, h, :]
 * A negative slot appends nothing (padding row).  A slot >= num_blocks*16 sets
 * PKV_DEVERR_BAD_SLOT and is skipped.  d*sizeof(dtype) must be a multiple of 16.
 */
int pkv_append(const void *k_rot, const void *v, const int64_t *slot_mapping,
               void *k_cache, void *v_cache, int32_t B, int32_t Hkv, int32_t d,
               int32_t num_blocks, int32_t dtype, int32_t *dev_err_flag, void *stream);

/*
 * a1 + a2 fused: one launch that rotates q and k as pkv_rope does and writes
 * the rotated key and the raw value into the cache slot as pkv_append does
 * (k_out still receives the rotated key).  Same argument rules as the two calls.
 */
int pkv_rope_append(const void *q, const void *k, const void *v, void *q_out, void *k_out,
                    const int32_t *positions, const int64_t *slot_mapping, void *k_cache,
                    void *v_cache, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                    int32_t num_blocks, float base, int32_t dtype, int32_t *dev_err_flag,
                    void *stream);

/*
 * Prefix KV of joining sequences (chunked prefill's cache write): T tokens,
 * each with its raw key k[t, Hkv, d], value v[t, Hkv, d], position
 * positions[t] and cache slot slot_mapping[t] (pkv_seq_slots gives both for a
 * chunk of one sequence; chunks of several sequences may be concatenated).
 * The key is rotated at its position exactly as pkv_rope_append rotates a
 * decode token (bit-identical rows), then both are written to the slot.
 * Same argument rules as pkv_rope_append; there is no query and no rotated-key
 * output.  Writes nothing but the T slots; a negative slot writes nothing.
 */
int pkv_prefill_kv(const void *k, const void *v, const int32_t *positions,
                   const int64_t *slot_mapping, void *k_cache, void *v_cache, int32_t T,
                   int32_t Hkv, int32_t d, int32_t num_blocks, float base, int32_t dtype,
                   int32_t *dev_err_flag, void *stream);

/* ======================================================================== */
/* a3 + a4: split-KV paged GQA decode attention and its LSE merge            */
/* ("neurogrid releases" v0.7.0 paged attention with GQA, v0.6.0 flash       */
/*  decode; "cortex-engine writeup" zero-denominator guard)                  */
/* ======================================================================== */
/*
 * Row b attends over its first seq_lens[b] tokens (the token appended in this
 * step included).  Token t of row b is row t%16 of block
 * block_tables[b*bt_stride + t/16].  Query head h uses KV head h / (Hq/Hkv).
 *   s_t   = (q_rot[b,h] . k_t) * scale + attn_bias[b*bias_stride + t]
 *   out   = sum_t softmax(s)_t v_t            (float32 accumulation)
 * attn_bias (device float32, nullable) is additive; -inf excludes a token (the
 * value at an excluded token must still be finite).  A row with no tokens, or
 * whose tokens are all excluded, outputs zeros.
 *
 * Partition: the (row, KV head) units, in row-major order, are laid end to
 * end as positions: a unit of n pages takes n + A positions, the first A
 * without a page (A, the cost of a unit boundary in pages: 4 at d = 64, 2 at
 * d = 128).  With P positions in all, part c of num_parts owns positions
 * [floor(c*P/num_parts), floor((c+1)*P/num_parts)) and the pages in them, and
 * runs as one CTA, so parts balance pages plus unit boundaries.  A unit whose
 * pages lie in one part is written to `out` directly.  Every other
 * unit leaves one float32 (o, lse) partial per part it touches in `workspace`;
 * the LSE merge (M = max lse; out = sum exp(lse_s - M) o_s / sum exp(lse_s - M))
 * then combines them.  By default the merge runs in the epilogue of
 * pkv_decode_attn_split, so `out` is complete when the call's kernel ends:
 * the last H parts of a unit to finish each merge a slice of its output
 * columns (H <= 32, at least 8 float4 columns each).  H > 1 only when the
 * grid fits on the GPU at once (num_parts <= the resident CTAs, which the
 * default partition always does): the kernel is then launched cooperatively,
 * so the helpers may wait for each other; otherwise the last part to finish
 * merges the unit alone.  With PKV_ATTN_SEPARATE_MERGE the
 * split kernel stops at the partials and pkv_lse_merge must follow with the
 * same arguments.  pkv_lse_merge may also be called after a fused call: it
 * recomputes the same merge from the partials left in the workspace.
 *
 * Workspace: pkv_attn_workspace_bytes(...) bytes, 256-byte aligned, owned by
 * the caller, ZERO-FILLED ONCE after allocation (it holds the fused merge's
 * per-unit counters, which every call leaves at zero).  Calls that share a
 * workspace must not overlap on the GPU.
 *
 * Supported: dtype PKV_BF16 or PKV_F32; d in {64, 128}; Hq/Hkv in {1,2,4,8};
 * B <= 65536.  q_rot [B,Hq,d] (16-byte aligned); out [B,Hq,d] (device, dtype,
 * 16-byte aligned).
 * num_parts <= 0 selects pkv_attn_default_parts(d, Hq, Hkv, dtype, flags) for the
 * current device (every SM holding as many CTAs as fit: the kernel variant,
 * and so the count, depends on the head dimension, the group size Hq/Hkv, the
 * dtype and PKV_ATTN_SIMT); at most 4096 parts.
 */
int pkv_attn_default_parts(int32_t d, int32_t Hq, int32_t Hkv, int32_t dtype, int32_t flags,
                           int32_t *num_parts);
int pkv_attn_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                             int32_t num_parts, size_t *bytes);

int pkv_decode_attn_split(const void *q_rot, const void *k_cache, const void *v_cache,
                          int32_t num_blocks, const int32_t *block_tables,
                          int32_t bt_stride, const int32_t *seq_lens,
                          const float *attn_bias, int32_t bias_stride, int32_t B,
                          int32_t Hq, int32_t Hkv, int32_t d, float scale,
                          int32_t num_parts, void *workspace, size_t workspace_bytes,
                          void *out, int32_t dtype, int32_t flags,
                          int32_t *dev_err_flag, void *stream);

/*
 * Attention without a caller-provided workspace.  This call has no
 * counterpart in the pages the method comes from; it exists for callers that
 * cannot allocate device memory (code running under another runtime's memory
 * manager, plugins that are handed only their input and output tensors, or
 * paths that must never reach an allocator).  It computes the same result as
 * pkv_decode_attn_split followed by its fused merge (same arguments, minus
 * the workspace) and takes its scratch from a 16 MiB array compiled into this
 * library; calls needing more scratch than that fail with
 * PKV_ERR_UNSUPPORTED.  It performs no device allocation or free.
 *  - Every GPU that loads the library holds the 16 MiB array until the
 *    process exits.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - All calls share the one array, which keeps the previous call's contents;
 *    each call clears the bytes it uses first (an asynchronous memset on
 *    `stream`).  Calls that overlap on the GPU (other streams, other host
 *    threads) race on the array and give wrong results: serialise them.
 *  - PKV_ATTN_SEPARATE_MERGE is rejected (the merge always runs in-kernel).
 */
int pkv_decode_attn_static(const void *q_rot, const void *k_cache, const void *v_cache,
                           int32_t num_blocks, const int32_t *block_tables, int32_t bt_stride,
                           const int32_t *seq_lens, const float *attn_bias, int32_t bias_stride,
                           int32_t B, int32_t Hq, int32_t Hkv, int32_t d, float scale,
                           int32_t num_parts, void *out, int32_t dtype, int32_t flags,
                           int32_t *dev_err_flag, void *stream);

/*
 * Host-planned partition.  Without a plan, every CTA of the attention kernel
 * first reads all row lengths (to find where its part starts) and then the
 * block ids of its first pages: two dependent reads before its first page
 * load, each a round trip over the CPU-GPU link when the step's metadata is
 * read in place from host memory.  The host that prepared the metadata (a0)
 * can state the same partition instead: pkv_plan_parts writes one record of
 * PKV_PLAN_INTS int32 per part, and the kernel then makes one read before it
 * loads pages.  Record c (part c of num_parts):
 *   [0] first row b0 of the part (-1: the part owns no position)
 *   [1] positions of the rows before b0, per KV head (sum of n_b + A over
 *       rows b < b0 with n_b > 0 pages; A = 4 at d = 64, 2 at d = 128)
 *   [2] seq_lens[b0], [3] seq_lens[b0 + 1] (0 past the last row)
 *   [4], [5] P, the total position count (int64, low word first)
 *   [6], [7] zero
 *   [8 + i], i < 16: block id of page j0 + i of the part's first unit segment
 *       (j0 its first page there); entries past the segment's last page are
 *       not written (and not read)
 * The plan is a pure function of (seq_lens, block tables, B, Hkv, d,
 * bt_stride, bias_stride, num_parts): it must come from the very metadata the
 * kernel reads, and be rebuilt whenever that changes.  PKV_ATTN_CHECK_PLAN
 * makes the kernel verify it.  Host-only; plan is [num_parts * PKV_PLAN_INTS].
 */
#define PKV_PLAN_INTS 24
int pkv_plan_parts(const int32_t *seq_lens, int32_t B, int32_t Hkv, int32_t d,
                   const int32_t *block_tables, int32_t bt_stride, int32_t bias_stride,
                   int32_t num_parts, int32_t *plan);

/* pkv_decode_attn_split with a plan from pkv_plan_parts (device or mapped
 * pointer; num_parts must be the plan's).  Same results, bit for bit.  Without
 * PKV_ATTN_CHECK_PLAN and without attn_bias the launch runs a smaller build of
 * the kernel (no row-length scan, plan check or bias code), which is faster:
 * the plan is the fast path. */
int pkv_decode_attn_planned(const void *q_rot, const void *k_cache, const void *v_cache,
                            int32_t num_blocks, const int32_t *block_tables,
                            int32_t bt_stride, const int32_t *seq_lens,
                            const float *attn_bias, int32_t bias_stride, int32_t B,
                            int32_t Hq, int32_t Hkv, int32_t d, float scale,
                            int32_t num_parts, const int32_t *plan, void *workspace,
                            size_t workspace_bytes, void *out, int32_t dtype, int32_t flags,
                            int32_t *dev_err_flag, void *stream);

/* bt_stride and bias_stride (0 when no bias was given) are the values passed to
 * pkv_decode_attn_split: they decide which rows are valid, exactly as there. */
int pkv_lse_merge(const void *workspace, size_t workspace_bytes, const int32_t *seq_lens,
                  int32_t bt_stride, int32_t bias_stride, int32_t B, int32_t Hq,
                  int32_t Hkv, int32_t d, int32_t num_parts, void *out, int32_t dtype,
                  void *stream);

/* ======================================================================== */
/* the whole device step: a1 -> a2 -> a3 -> a4 on one stream                */
/* ======================================================================== */
typedef struct pkv_step_args {
  const void *q, *k, *v;             /* new tokens: [B,Hq,d], [B,Hkv,d], [B,Hkv,d] */
  void *q_rot, *k_rot;               /* RoPE outputs (device scratch owned by the caller) */
  void *k_cache, *v_cache;           /* [num_blocks,Hkv,16,d] */
  int32_t num_blocks;
  const int32_t *positions;          /* [B] */
  const int64_t *slot_mapping;       /* [B] */
  const int32_t *seq_lens;           /* [B] lengths after the append */
  const int32_t *block_tables;       /* [B*bt_stride] */
  int32_t bt_stride;
  const float *attn_bias;            /* nullable, [B*bias_stride] */
  int32_t bias_stride;
  int32_t B, Hq, Hkv, d;
  float scale, rope_base;
  int32_t dtype, flags, num_parts;
  void *workspace;                   /* pkv_attn_workspace_bytes(...) bytes */
  size_t workspace_bytes;
  void *out;                         /* [B,Hq,d] */
  int32_t *dev_err_flag;             /* nullable */
  const int32_t *plan;               /* nullable: pkv_plan_parts of this step's metadata
                                        for num_parts parts (num_parts must then be > 0) */
} pkv_step_args;

/* All pointers in *args are device pointers or host memory the GPU can reach
 * (pinned / mapped: q, k, v, positions, slot_mapping, seq_lens and block_tables
 * may live there so that a step needs no host-to-device copy -- the kernels read
 * them in place -- and out so that it needs no copy back; give the mapped
 * address, pkv_mapped_pointer); asynchronous on stream.
 * Runs pkv_rope_append, then pkv_decode_attn_split launched as a programmatic
 * dependent (its prologue overlaps the RoPE kernel), and pkv_lse_merge when
 * flags has PKV_ATTN_SEPARATE_MERGE.  With PKV_STEP_FUSED the whole step is
 * one kernel instead: the attention kernel also rotates q and k and appends
 * the rotated key and the value (the part that owns a row's last page writes
 * that row's slot before it loads the page; rows with seq_len 0 are not
 * appended).  Both forms give bit-identical results.  q_rot/k_rot receive the
 * rotated q and k.  Each row's slot must be its position seq_len-1 in its own
 * blocks, as pkv_prepare_step produces. */
int pkv_decode_step(const pkv_step_args *args, void *stream);

/*
 * A decode step through n_layers layers, each with its own caches
 * ("neurogrid releases" v0.7.0: per-layer caches; the block tables, slots,
 * positions and lengths are the same for every layer, so layers[l] differ in
 * q, k, v, q_rot, k_rot, k_cache, v_cache, out and workspace).  Layer l runs
 * after layer l-1 on `stream`: its RoPE/append kernel is launched as a
 * programmatic dependent of layer l-1's attention kernel (its angles are
 * formed early; its q/k/v reads and cache writes wait for that kernel), and
 * its attention kernel as a dependent of its RoPE/append kernel, so each
 * layer's start overlaps the previous layer's tail.  Consecutive layers must
 * not share a workspace (two alternating workspaces suffice).
 * PKV_STEP_FUSED is rejected.  Stops at the first failing layer.  The layers'
 * attention kernels are not launched cooperatively unless a layer's flags have
 * PKV_LAYERS_MERGE_HELPERS, so by default each unit's merge is done by its last
 * part alone (the next layer's kernels may then start on SMs the previous layer
 * has freed); with it, each layer merges like pkv_decode_step (bit-identical to
 * one single-layer step per layer).
 */
int pkv_decode_step_layers(const pkv_step_args *layers, int32_t n_layers, void *stream);

/*
 * The dense right-padded batch that paging replaces, kept as a comparator
 * (helexa issue 121: slice 1 assemble_batch, slice 3a extract_row).  All KV
 * buffers use the block layout [blocks, Hkv, 16, d] (dtype): a snapshot is one
 * sequence's tokens [0, len) in ceil(len/16) blocks; a dense batch of B rows
 * and cap tokens per row (cap a multiple of 16) is B*cap/16 blocks, row b owning
 * blocks [b*cap/16, (b+1)*cap/16), so the attention call reads it as a pool
 * with block table row b = b*cap/16 + j and an additive -inf bias on the gap.
 * k_snaps, v_snaps: host arrays of device pointers.  Buffers must be large
 * enough for the tokens named; nothing else is checked on the device.
 * Hkv * d * sizeof(dtype) must be at most 16 KB.
 *
 * pkv_dense_assemble: dense row b = snapshot b's tokens [0, lens[b]) followed by
 * zeros up to padded_len (lens[b] <= padded_len <= cap); tokens from
 * padded_len on are left for the decode columns.
 * pkv_dense_extract: for each i, snapshot i = dense row rows[i]'s prefix
 * [0, prefix_lens[i]) followed by its decode columns [padded_len,
 * padded_len + steps) (the gap is dropped).
 */
int pkv_dense_assemble(const void *const *k_snaps, const void *const *v_snaps,
                       const int32_t *lens, int32_t B, int32_t padded_len, void *k_dense,
                       void *v_dense, int32_t cap, int32_t Hkv, int32_t d, int32_t dtype,
                       void *stream);
int pkv_dense_extract(const void *k_dense, const void *v_dense, int32_t cap,
                      const int32_t *rows, const int32_t *prefix_lens, int32_t n_rows,
                      int32_t padded_len, int32_t steps, void *const *k_snaps,
                      void *const *v_snaps, int32_t Hkv, int32_t d, int32_t dtype,
                      void *stream);

/* The address under which kernels read the page-locked host buffer at
 * host_ptr (allocated pinned, or registered with the mapped flag), so that the
 * per-step metadata of pkv_decode_step can stay in host memory and be read by
 * the kernels over the CPU-GPU link instead of being copied first.  The buffer
 * must not change until the kernels that read it have finished.  Returns
 * PKV_ERR_INVALID_ARG for a NULL pointer and PKV_ERR_CUDA when the memory is
 * not mapped for the current device. */
int pkv_mapped_pointer(const void *host_ptr, void **device_ptr);

/* Host-side buffers for pkv_decode_step_host (pinned memory recommended). */
#define PKV_HOST_IN_PLACE 1   /* pkv_step_host_io.flags: the kernels read the host
                                 inputs and write the host output in place
                                 instead of going through device copies */

typedef struct pkv_step_host_io {
  const void *q, *k, *v;             /* [B,Hq,d], [B,Hkv,d], [B,Hkv,d] */
  const int32_t *positions;
  const int64_t *slot_mapping;
  const int32_t *seq_lens;
  const int32_t *block_tables;       /* [B*bt_stride] */
  void *out;                         /* [B,Hq,d] */
  int32_t flags;                     /* 0 or PKV_HOST_IN_PLACE */
  const int32_t *plan;               /* nullable: the step's plan (pkv_plan_parts), read in
                                        place or copied to dev->plan like the metadata */
} pkv_step_host_io;

/*
 * End-to-end step from host memory: copies the host inputs into the device
 * buffers named by *dev (q, k, v, positions, slot_mapping, seq_lens,
 * block_tables), runs pkv_decode_step, copies dev->out back to host->out and
 * waits for the stream.  Returns after the result is in host memory.  With
 * PKV_HOST_IN_PLACE the inputs and host->out must be page-locked host memory;
 * the step's kernels read the inputs and write the result over the CPU-GPU
 * link at their mapped addresses (no staging or result copies; dev's input
 * pointers and dev->out are not used).  The mapped address of each host buffer is looked up once per
 * device and remembered (a buffer freed and re-registered at the same address
 * must keep its mapping).
 */
int pkv_decode_step_host(const pkv_step_args *dev, const pkv_step_host_io *host,
                         void *stream);

/*
 * The work of pkv_decode_step_host(dev, host) -- staging copies or in-place
 * reads per host->flags, the step's kernels, the copy of the output back --
 * captured once as a CUDA graph for these exact buffers (their addresses are
 * fixed in it: each launch reads whatever the host last wrote there, typically
 * pkv_prepare_step's outputs and the new q/k/v).  A serving loop then pays one
 * graph launch per step instead of every launch and copy.  *out owns the graph
 * (free with pkv_step_graph_destroy).  Nothing runs at creation.
 */
typedef struct pkv_step_graph pkv_step_graph;
int pkv_step_graph_create(const pkv_step_args *dev, const pkv_step_host_io *host,
                          pkv_step_graph **out);
/* Launches the captured step on stream and waits for it (host->out is then set). */
int pkv_step_graph_launch(pkv_step_graph *g, void *stream);
/*
 * The same launch without the wait, and the wait on its own.  Each graph
 * records its own completion event after every enqueue, so a loop over two
 * graphs (two sets of host buffers) keeps the GPU busy: prepare step i into
 * set i%2 (a0, the plan, the new q/k/v), enqueue its graph, then wait for the
 * graph of step i-1 and read its output while the GPU runs step i.  Host
 * buffers a queued or running launch reads or writes must not be touched until
 * pkv_step_graph_wait has returned for that graph.  The graphs of one loop
 * share the device buffers of dev (scratch, caches), so they go on one stream.
 * Errors: PKV_ERR_INVALID_ARG for a NULL graph; PKV_ERR_CUDA if the launch or
 * the event record fails (the message names the call).
 */
int pkv_step_graph_enqueue(pkv_step_graph *g, void *stream);
/* Waits (blocking the calling thread) for the last pkv_step_graph_enqueue of
 * g; host->out then holds that step's output.  Returns at once if g was never
 * enqueued.  Errors: PKV_ERR_INVALID_ARG for a NULL graph; PKV_ERR_CUDA if the
 * step failed on the device (a sticky CUDA error: the context is then lost). */
int pkv_step_graph_wait(pkv_step_graph *g);
/* Frees the graph and its event (NULL is ignored); no launch of g may be in
 * flight. */
void pkv_step_graph_destroy(pkv_step_graph *g);

/* ======================================================================== */
/* native serving loop: continuous batching, one host call per step          */
/* ======================================================================== */
/*
 * The continuous-batching loop of helexa issue 121, slice 3b (admit joiners,
 * prefill them, rebatch, decode every live sequence in lockstep) over the
 * paged cache of "neurogrid releases" v0.7.0 (joining or leaving edits block
 * tables only; no KV moves), the step replayed as one CUDA graph that reads
 * the host-written metadata in place (v0.8.0).  A joiner takes over the row of
 * a sequence that left, so the batch keeps its B rows and two captured graphs
 * (one per pinned metadata buffer, used alternately) serve every step.
 *
 * The caller owns every buffer and keeps each alive and in place for the
 * server's lifetime (the server allocates no device memory):
 *  - step: pkv_decode_step's device buffers and sizes for B rows.  step.q,
 *    step.k, step.v are the graph's input buffers.  Its metadata and plan
 *    pointers are ignored (the server points them into meta_host); num_parts
 *    must be > 0; attn_bias must be NULL.
 *  - alloc: the block allocator; rows[b] (B entries) are live sequences of it,
 *    which the server then manages (joins and leaves go through the server).
 *  - meta_host[2]: page-locked host buffers of pkv_server_meta_bytes(B,
 *    bt_stride, num_parts) bytes, 16-byte aligned (positions, slots, lengths,
 *    block tables and the partition plan of a step).
 *  - prefix_host[2]: page-locked host buffers of
 *    pkv_server_prefix_bytes(max_prefix_tokens) bytes (joiners' prefix
 *    positions and slots), or NULL when max_prefix_tokens is 0.
 * Creation captures the two graphs; nothing runs.
 */
typedef struct pkv_server pkv_server;
typedef struct pkv_server_desc {
  pkv_step_args step;
  pkv_alloc *alloc;
  const int32_t *rows;               /* [step.B] live sequence ids, one per row */
  void *meta_host[2];
  void *prefix_host[2];
  int32_t max_prefix_tokens;         /* most prefix tokens joining in one step */
} pkv_server_desc;
size_t pkv_server_meta_bytes(int32_t B, int32_t bt_stride, int32_t num_parts);
size_t pkv_server_prefix_bytes(int32_t max_prefix_tokens);
int pkv_server_create(const pkv_server_desc *desc, pkv_server **out);
/*
 * One step, enqueued on stream.  The sequences of rows leave_rows[0..n-1]
 * retire and n joiners take those rows, joiner i with a prefix of
 * prefix_lens[i] tokens whose raw keys and values are prefix_k, prefix_v
 * (device, [sum(prefix_lens), Hkv, d], joiner after joiner): they are rotated
 * at their positions and written into the joiners' blocks (pkv_prefill_kv).
 * Then every row decodes one token: q, k, v (device, [B,Hq,d], [B,Hkv,d],
 * [B,Hkv,d]; NULL or the step's own input buffers: nothing to copy) are copied
 * into the step's input buffers, a0 (pkv_prepare_step_cached) and the plan
 * (pkv_plan_parts) are written into a metadata buffer, and the captured step
 * is launched: the result is in step.out when the stream gets there.  The
 * call waits only for the step two calls back, which used the same host
 * buffers.  Argument errors change nothing; a failure after the leaves (the
 * pool cannot take the joiners: PKV_ERR_OUT_OF_BLOCKS) leaves the server
 * unusable, and every later step returns PKV_ERR_INVALID_ARG.
 */
int pkv_server_step(pkv_server *s, const int32_t *leave_rows, const int32_t *prefix_lens,
                    int32_t n, const void *prefix_k, const void *prefix_v, const void *q,
                    const void *k, const void *v, void *stream);
/* The sequence id of every row ([B]). */
int pkv_server_rows(const pkv_server *s, int32_t *rows);
/* Frees the server (not the caller's buffers or allocator); call after its
 * last step has finished on the GPU. */
void pkv_server_destroy(pkv_server *s);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
