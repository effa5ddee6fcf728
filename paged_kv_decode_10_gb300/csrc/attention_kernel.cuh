// a3: split-KV paged grouped-query decode attention (sm_103a).
//
// What it computes ("neurogrid releases" v0.7.0: paged attention reading K/V
// through block_table indirection with GQA; v0.6.0: flash decode, online
// softmax over KV tiles without materialising the score matrix;
// "cortex-engine writeup", block-sparse attention: zero denominator -> zero
// output):  out[b,h] = sum_t softmax_t(q[b,h].k_t * scale + bias[b,t]) v_t over
// the first seq_lens[b] tokens of row b, with query head h reading KV head
// h / G.
//
// How it runs on GB300:
//  * Work list.  The (row, KV head) units, row-major, are laid end to end as
//    positions: a unit of n pages takes n + A positions (A = seg_cost, the
//    cost of a unit boundary in pages).  CTA c (one per part, grid =
//    num_parts) owns positions [c*P/C, (c+1)*P/C) and the pages in them, so
//    every CTA gets the same pages-plus-boundaries work whatever the length
//    mix.  The host may state each CTA's start in a plan record (first row,
//    its offset and length, the first block ids); otherwise the prologue
//    derives it from a scan of the row lengths.  A unit split across CTAs
//    leaves one (o, lse) partial per CTA, merged in the epilogue by the last
//    CTA to finish it, or for long splits by the last H CTAs (merge helpers,
//    one column slice each, under a cooperative launch), or by the LSE merge
//    kernel; a unit inside one CTA is written to the output directly.
//  * Producer warp.  Walks the CTA's unit segments, hands each to the
//    consumers through a shared-memory slot (a header and the unit's query
//    rows, bulk-copied), reads block ids 32 at a time (the next segment's
//    ahead) and issues 2-D TMA tensor loads (128-byte swizzle, L2
//    evict-first) of each 16-token K and V page into a ring of NS stages, each
//    guarded by a full/empty mbarrier pair.  Every K/V byte is read from HBM
//    once, because a CTA holds all G query heads of its KV head.
//  * Consumer warps.  Page x of the range goes to consumer warp x % NW.  Each
//    warp keeps its own online-softmax state (running max m, sum l,
//    accumulator) for the G heads and, at the end of each unit segment, the
//    warps combine their states through shared memory.
//      - MMA consumer (bf16): S^T = K Q^T and O^T += V^T P^T with
//        mma.sync.m16n8k16 (16 tokens x 8 head columns, f32 accumulate);
//        K/V fragments come from ldmatrix (.trans for V) on the swizzled
//        stage, P^T from movmatrix.  Head columns beyond G hold zero queries.
//      - SIMT consumer (bf16 / f32): each lane owns d/32 dimensions; the G
//        partial dot products of a token are reduce-scattered across the warp
//        so each lane ends with one head's score; P goes through a small
//        shared buffer for the P.V update.
//  * Softmax runs in base 2 (scores pre-multiplied by log2 e); partial lse
//    values in the workspace are base-2.
#pragma once
#include <cuda.h>

#include "common.cuh"

namespace pkv {

struct AttnParams {
  const void *q;            // [B, Hq, D] rotated queries
  const int32_t *block_tables;
  const int32_t *seq_lens;
  const float *bias;        // nullable [B, bias_stride]
  float *o_part;            // [(U + C), G, D]
  float *lse_part;          // [(U + C), G]
  int32_t *meta;            // [U, 2]: first part, number of parts spanned; then P (int64)
  int32_t *counters;        // [U] parts of a split unit that have written their partial
  int32_t *done;            // [U] merge helpers of a unit that are done (both kept at 0)
  void *out;                // [B, Hq, D]
  const int32_t *plan;      // nullable: [C, PKV_PLAN_INTS] host-planned partition (pkv_plan_parts)
  int check_plan;           // also derive the partition here and flag a plan that disagrees
  int32_t *err;
  int bt_stride, bias_stride;
  int B, Hq, Hkv, G;
  int num_blocks, num_parts;
  int fuse_merge;           // 1: the parts of a unit merge it (a4 in the epilogue)
  int max_helpers;          // parts that may share one unit's merge (1 unless co-resident)
  int seg_cost;             // pages of work a unit boundary is worth to the partition
  float scale_log2;         // softmax scale * log2(e)
  long long wait_limit;     // SM clocks after which a pipeline or merge wait gives up
  // whole-step kernels only (a1 + a2 fused in): the step's new tokens, where
  // they go, and where their rotated copies are reported
  const void *q_new, *k_new, *v_new;   // [B,Hq,D], [B,Hkv,D], [B,Hkv,D]
  const int32_t *positions;            // [B] RoPE positions
  const int64_t *slots;                // [B] cache slots of the new tokens
  void *k_cache_w, *v_cache_w;         // the caches, written at the slots
  void *q_rot_out, *k_rot_out;         // [B,Hq,D], [B,Hkv,D]
  long long num_slots;                 // num_blocks * 16
  unsigned long long turns[128];       // RoPE fixed-point turns (fill_rope_turns)
};

constexpr float kLog2e = 1.4426950408889634f;
constexpr long long kWaitLimitCycles = 1ll << 31;   // about one second
// block ids a plan record carries (the first chunk of a part's pages)
constexpr int kPlanIds = PKV_PLAN_INTS - 8;
// a merge helper takes at least this many float4 columns of a unit's output
constexpr int kHelperMinCols = 8;
constexpr int kMaxHelpers = 32;
// units split over fewer parts are merged by their last part alone (its loads
// of all partials fit in one round trip; helpers would only add a wait)
constexpr int kHelperMinSplit = 8;

// Pages of a row of length L, or 0 for an invalid length (which also sets *bad).
__device__ __forceinline__ int pages_of_len(int L, int bt_stride, bool has_bias, int bias_stride,
                                            bool *bad) {
  const bool ok = L >= 0 && L <= bt_stride * kBlockTokens && (!has_bias || L <= bias_stride);
  *bad = !ok;
  return ok ? (L + kBlockTokens - 1) / kBlockTokens : 0;
}
__device__ __forceinline__ int row_pages(const int32_t *seq_lens, int b, int bt_stride,
                                         bool has_bias, int bias_stride, bool *bad) {
  return pages_of_len(seq_lens[b], bt_stride, has_bias, bias_stride, bad);
}

// floor(a / b) for a >= 0, b > 0 (the compiler's 64-bit division measured
// faster here than float-estimate variants).
__device__ __forceinline__ long long div_floor(long long a, long long b) { return a / b; }

// Part that owns global page x: the largest c with floor(c*P/C) <= x, i.e.
// with c*P < (x+1)*C.
__device__ __forceinline__ int part_of(long long x, long long P, int C) {
  return static_cast<int>(div_floor((x + 1) * C - 1, P));
}

// A part owns no page when C > P and its page range is empty.
__device__ __forceinline__ bool part_empty(long long c, long long P, int C) {
  return div_floor(P * c, C) == div_floor(P * (c + 1), C);
}

// The same, kept out of line: callers test C > P first, and the 64-bit
// divisions must not be evaluated speculatively on the common path.
static __device__ __noinline__ bool part_empty_slow(long long c, long long P, int C) {
  return part_empty(c, P, C);
}

// Parts c0 .. c0+n-1 that own at least one page (all of them when C <= P).
// The counting loops only run when C > P and are kept out of line so that the
// common path stays short (the epilogue's code is fetched cold).
static __device__ __noinline__ int count_real_parts(int c0, int n, long long P, int C) {
  int r = 0;
  for (int s = 0; s < n; ++s) r += !part_empty(c0 + s, P, C);
  return r;
}
__device__ __forceinline__ int real_parts(int c0, int n, long long P, int C) {
  return C <= P ? n : count_real_parts(c0, n, P, C);
}

// a4, the LSE merge of one float4 column (head h, dims 4*d4 .. 4*d4+3) over the
// partials i < n stored at slots slot0 + i*stride (skip(i): no partial there).
// A partial is (o_s normalised, base-2 lse_s):
//   out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M),  M = max_s lse_s,
// and the merged lse is M + log2(sum_s 2^(lse_s - M)).  Nothing unmasked
// anywhere -> zeros and lse = -inf.  Loads bypass L1: other CTAs of this grid
// wrote the partials.
template <typename Skip>
__device__ __forceinline__ float4 merge_column(const float *o, const float *lse, size_t slot0,
                                               int n, int stride, int G, int D, int h, int d4,
                                               Skip skip, float *lse_out) {
  float M = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (!skip(i)) M = fmaxf(M, __ldcg(lse + (slot0 + static_cast<size_t>(i) * stride) * G + h));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (M != -INFINITY) {
    for (int i = 0; i < n; ++i) {
      if (skip(i)) continue;
      const size_t s = slot0 + static_cast<size_t>(i) * stride;
      const float w = ex2(__ldcg(lse + s * G + h) - M);
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(o + (s * G + h) * D) + d4);
      den += w;
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
  }
  if (den > 0.f) {
    const float r = 1.f / den;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
    *lse_out = M + log2f(den);
  } else {
    *lse_out = -INFINITY;
  }
  return acc;
}

template <typename T>
__device__ __forceinline__ void store4(T *dst, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float *dst, float4 v) {
  *reinterpret_cast<float4 *>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *dst, float4 v) {
  uint2 w;
  w.x = pack_bf16(v.x, v.y);
  w.y = pack_bf16(v.z, v.w);
  *reinterpret_cast<uint2 *>(dst) = w;
}

// The fused a4.  Every part of a unit split over n parts writes its (o, lse)
// partial and adds one to the unit's counter.  The last H parts to arrive are
// the unit's merge helpers: helper r waits until the counter reaches n, then
// merges float4 columns [r*NC/H, (r+1)*NC/H) of the unit's output (NC = G*D/4)
// over all n partials.  With H > 1 the merge of a long unit is spread over H
// CTAs and each thread issues the loads of its few partials at once, so it
// costs about one L2 round trip after the last partial lands.  Helpers wait on
// other CTAs of the grid, so H > 1 only when the launch makes every CTA
// co-resident (a cooperative launch); otherwise H = 1, the last part alone.
__device__ __forceinline__ int merge_helpers(int n, int ncols, int max_helpers) {
  return max(1, min(n, min(max_helpers, ncols / kHelperMinCols)));
}

// Online combination of partials (base-2 lse) into (M, den, acc): acc and den
// are sums of 2^(lse_s - M) o_s and 2^(lse_s - M).
struct MergeAcc {
  float M, den;
  float4 acc;
};

template <int K>
__device__ __forceinline__ void merge_acc_add(MergeAcc &a, const float (&l)[K],
                                              const float4 (&v)[K]) {
  float m = a.M;
#pragma unroll
  for (int u = 0; u < K; ++u) m = fmaxf(m, l[u]);
  if (m == -INFINITY) return;
  const float r = ex2(a.M - m);   // 0 while nothing was accumulated
  a.den *= r;
  a.acc.x *= r;
  a.acc.y *= r;
  a.acc.z *= r;
  a.acc.w *= r;
#pragma unroll
  for (int u = 0; u < K; ++u) {
    const float w = ex2(l[u] - m);
    if (w != 0.f) {
      a.den += w;
      a.acc.x = fmaf(w, v[u].x, a.acc.x);
      a.acc.y = fmaf(w, v[u].y, a.acc.y);
      a.acc.z = fmaf(w, v[u].z, a.acc.z);
      a.acc.w = fmaf(w, v[u].w, a.acc.w);
    }
  }
  a.M = m;
}

// Partials i = j, j + R, j + 2R, ... < nseg of unit u_idx (part cf + i, slot
// u_idx + cf + i; parts that own no page have none), float4 column `col`.
// The loads of up to 8 partials go out together.  Loads bypass L1: other CTAs
// of this grid wrote the partials.
__device__ __forceinline__ MergeAcc merge_partials(const float *o, const float *lse, int u_idx,
                                                   int cf, int nseg, int j, int R, int col,
                                                   int G, int D, long long P, int C) {
  const int h = col / (D / 4), d4 = col - h * (D / 4);
  MergeAcc a{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  constexpr int K = 8;
  for (int i0 = j; i0 < nseg; i0 += K * R) {
    float l[K];
    float4 v[K];
#pragma unroll
    for (int t = 0; t < K; ++t) {
      const int i = i0 + t * R;
      const bool on = i < nseg && !(C > P && part_empty_slow(cf + i, P, C));
      const size_t slot = static_cast<size_t>(u_idx) + cf + i;
      l[t] = on ? __ldcg(lse + slot * G + h) : -INFINITY;
      v[t] = on ? __ldcg(reinterpret_cast<const float4 *>(o + (slot * G + h) * D) + d4)
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    merge_acc_add<K>(a, l, v);
  }
  return a;
}

template <typename T>
__device__ __forceinline__ void merge_store(T *out_rows, int col, int D, const MergeAcc &a) {
  const int h = col / (D / 4), d4 = col - h * (D / 4);
  float4 o = a.acc;
  if (a.den > 0.f) {
    const float inv = __frcp_rn(a.den);
    o.x *= inv;
    o.y *= inv;
    o.z *= inv;
    o.w *= inv;
  } else {
    o = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  store4<T>(out_rows + h * D + 4 * d4, o);
}

// Helper r of H: columns [r*NC/H, (r+1)*NC/H) of unit u_idx (parts cf ..
// cf+nseg-1) merged into out_rows [G, D] by the NTHR consumer threads.  When
// the slice has fewer columns than threads, R = NTHR / cols threads share a
// column (each takes every R-th partial) and combine through `scratch`
// (NTHR * 6 floats of shared memory; all NTHR threads must call this).
template <typename T, int NTHR>
__device__ __forceinline__ void merge_slice(const AttnParams &p, int u_idx, int cf, int nseg,
                                            long long P, int C, int r, int H, int D, T *out_rows,
                                            float *scratch, int tid) {
  const int NC = p.G * (D / 4);
  const int col0 = r * NC / H, cols = (r + 1) * NC / H - col0;
  const int R = max(1, NTHR / cols);
  if (R == 1) {
    for (int c = tid; c < cols; c += NTHR)
      merge_store<T>(out_rows, col0 + c, D,
                     merge_partials(p.o_part, p.lse_part, u_idx, cf, nseg, 0, 1, col0 + c, p.G, D,
                                    P, C));
    return;
  }
  MergeAcc a{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  if (tid < cols * R)
    a = merge_partials(p.o_part, p.lse_part, u_idx, cf, nseg, tid / cols, R, col0 + tid % cols,
                       p.G, D, P, C);
  float *e = scratch + tid * 6;
  e[0] = a.M;
  e[1] = a.den;
  e[2] = a.acc.x;
  e[3] = a.acc.y;
  e[4] = a.acc.z;
  e[5] = a.acc.w;
  asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
  if (tid < cols) {
    // combine the R subset results: rescale each to the largest M
    float m = -INFINITY;
    for (int q = 0; q < R; ++q) m = fmaxf(m, scratch[(tid + q * cols) * 6]);
    MergeAcc t{m, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
    if (m != -INFINITY) {
      for (int q = 0; q < R; ++q) {
        const float *f = scratch + (tid + q * cols) * 6;
        const float w = ex2(f[0] - m);   // 0 for a subset that saw nothing
        t.den = fmaf(w, f[1], t.den);
        t.acc.x = fmaf(w, f[2], t.acc.x);
        t.acc.y = fmaf(w, f[3], t.acc.y);
        t.acc.z = fmaf(w, f[4], t.acc.z);
        t.acc.w = fmaf(w, f[5], t.acc.w);
      }
    }
    merge_store<T>(out_rows, col0 + tid, D, t);
  }
}

// Waits until *counter >= target (acquire); gives up after ~limit SM clocks.
__device__ __forceinline__ bool wait_count(const int32_t *counter, int target, long long limit) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
  if (v >= target) return true;
  const long long t0 = clock64();
  for (;;) {
    __nanosleep(32);
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    if (v >= target) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// Release / acquire at GPU scope around the merge counters (the partials that
// other threads of this CTA wrote before a CTA barrier are covered: fences are
// cumulative).
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ int atom_add_relaxed_gpu(int32_t *p, int v) {
  int old;
  asm volatile("atom.relaxed.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void fence_sc_cta() { asm volatile("fence.sc.cta;" ::: "memory"); }

// Waits (bounded) for the last phase armed on every ring stage and segment
// slot, the only phases that can still have a copy in flight.
template <int NS, int SLOTS>
__device__ __noinline__ void drain_copies(uint64_t *full, uint64_t *segfull, const int *stage_pg,
                                          const int *slot_seg, int lane) {
  for (int s = lane; s < NS; s += 32)
    if (stage_pg[s] >= 0)
      mbar_wait_bounded(&full[s], static_cast<uint32_t>(stage_pg[s] / NS) & 1u, kWaitLimitCycles);
  for (int s = lane; s < SLOTS; s += 32)
    if (slot_seg[s] >= 0)
      mbar_wait_bounded(&segfull[s], static_cast<uint32_t>(slot_seg[s] / SLOTS) & 1u,
                        kWaitLimitCycles);
}

// A consumer thread gives up: it records the abort and, if the producer warp
// has already finished (and so will not drain), drains the copies itself.
template <int NS, int SLOTS>
__device__ __noinline__ void consumer_abort(volatile int *misc, uint64_t *full, uint64_t *segfull,
                                            const int *stage_pg, const int *slot_seg) {
  misc[2] = 1;
  fence_sc_cta();
  if (misc[3] != 0) drain_copies<NS, SLOTS>(full, segfull, stage_pg, slot_seg, 0);
}

struct UnitCursor {
  int b, g, n;      // row, KV head, pages per unit of this row
  long long off;    // first global page of unit (b, g)
};

// Compile-time geometry of one kernel variant.
template <typename T, int D, int NW, int NS>
struct Geo {
  static constexpr int kElem = sizeof(T);
  static constexpr int kSubCols = 128 / kElem;                 // elements per 128-B row
  static constexpr int kSubs = D * kElem / 128;                // 128-B sub-tiles per token row
  static constexpr int kSubBytes = kBlockTokens * 128;         // one sub-tile of a page
  static constexpr int kTileBytes = kBlockTokens * D * kElem;  // one K (or V) page
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kThreads = (NW + 1) * 32;
  static constexpr int kHeadsPad = 8;
  // shared-memory carve-up (after 1024-byte alignment of the base)
  static constexpr int kOffRedAcc = NS * kStageBytes;
  static constexpr int kOffRedM = kOffRedAcc + NW * kHeadsPad * D * 4;
  static constexpr int kOffRedL = kOffRedM + NW * kHeadsPad * 4;
  static constexpr int kOffPBuf = kOffRedL + NW * kHeadsPad * 4;
  static constexpr int kOffABuf = kOffPBuf + NW * kBlockTokens * kHeadsPad * 4;
  static constexpr int kOffBars = kOffABuf + NW * kHeadsPad * 4;      // 8-aligned
  static constexpr int kOffBad = kOffBars + 2 * NS * 8;
  static constexpr int kOffScan = kOffBad + NS * 4;
  static constexpr int kOffMisc = kOffScan + (kThreads / 32) * 4;   // 16 ints
  // segment slots: the producer hands each unit segment to the consumers as a
  // 64-byte header (row, KV head, pages, length, page range, first page; FUSE:
  // the row's position) and the unit's query rows (up to 8 heads): rotated
  // rows bulk-copied from global memory, or (FUSE) the raw rows it loaded
  static constexpr int kSegSlots = 4;
  static constexpr int kSegQBytes = 8 * D * kElem;
  static constexpr int kSegBytes = 64 + kSegQBytes;
  // per ring stage and per segment slot: the last page / segment the producer
  // arrived on it for (its pending phase, which an aborting CTA drains)
  static constexpr int kOffPg = kOffMisc + 64;
  static constexpr int kOffSeg = (kOffPg + (NS + kSegSlots) * 4 + 127) / 128 * 128;
  static constexpr int kOffSegBars = kOffSeg + kSegSlots * kSegBytes;
  // row lengths of the first kLensCache rows, as the prologue read them
  static constexpr int kLensCache = 256;
  static constexpr int kOffLens = kOffSegBars + 2 * kSegSlots * 8;
  // whole-step kernels: the RoPE turn table, copied from the parameters once
  // (threads index it by pair, which the parameter bank would serialise)
  static constexpr int kOffTurns = kOffLens + kLensCache * 4;
  static constexpr int kSmemBytes = kOffTurns + (D / 2) * 8 + 1024;   // + alignment slack
  static_assert(kSubs >= 1 && D * kElem % 128 == 0, "row must be whole 128-B lines");
  static_assert(NS % NW == 0, "a stage must always feed the same consumer warp");
};

// Byte offset inside a page tile of (token row, 16-byte chunk j16) under the
// 128-byte TMA swizzle: chunk index XOR (row % 8) inside each 128-B line.
__device__ __forceinline__ uint32_t swz(int row, int j16) {
  return static_cast<uint32_t>((j16 >> 3) * (kBlockTokens * 128) + row * 128 +
                               (((j16 & 7) ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------------------
// consumers
// ---------------------------------------------------------------------------
template <int D>
struct MmaState {
  uint32_t qb[D / 16][2];
  float acc[D / 16][4];
  float m[2], l[2];
};

template <typename T, int D>
__device__ __forceinline__ void mma_begin(MmaState<D> &s, const AttnParams &p, int b, int g,
                                          int lane) {
  const int r = lane >> 2, c = lane & 3;
  const bool real = r < p.G;
  const __nv_bfloat16 *qrow = static_cast<const __nv_bfloat16 *>(p.q) +
                              (static_cast<size_t>(b) * p.Hq + g * p.G + (real ? r : 0)) * D;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * c);
    s.qb[ks][0] = real ? w[0] : 0u;
    s.qb[ks][1] = real ? w[4] : 0u;
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) s.acc[mt][e] = 0.f;
  s.m[0] = s.m[1] = -INFINITY;
  s.l[0] = s.l[1] = 0.f;
}

// One 16-token page: tokens t0 .. t0+15 of which the first `valid` count.
template <int D>
__device__ __forceinline__ void mma_page(MmaState<D> &s, const AttnParams &p, uint32_t ktile,
                                         uint32_t vtile, int valid, int b, int t0, int lane,
                                         bool may_bias) {
  const int r = lane >> 2, c = lane & 3;
  const int mq = lane >> 3;
  const int krow = (lane & 7) + (mq & 1) * 8, kj = mq >> 1;
  const int vrow = (lane & 7) + (mq >> 1) * 8, vj = mq & 1;
  // S^T[token, head] = sum_d K[token, d] Q[head, d]; two accumulators shorten the chain.
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4(ktile + swz(krow, ks * 2 + kj), a0, a1, a2, a3);
    if (ks & 1)
      mma_bf16_16816(sb, a0, a1, a2, a3, s.qb[ks][0], s.qb[ks][1]);
    else
      mma_bf16_16816(sa, a0, a1, a2, a3, s.qb[ks][0], s.qb[ks][1]);
  }
  float sc[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) sc[e] = (sa[e] + sb[e]) * p.scale_log2;
  // sc[0]: (token r, head 2c)  sc[1]: (r, 2c+1)  sc[2]: (r+8, 2c)  sc[3]: (r+8, 2c+1)
  if (may_bias && p.bias) {
    const float *bias = p.bias + static_cast<size_t>(b) * p.bias_stride + t0;
    if (r < valid) {
      const float x = bias[r] * kLog2e;
      sc[0] += x;
      sc[1] += x;
    }
    if (r + 8 < valid) {
      const float x = bias[r + 8] * kLog2e;
      sc[2] += x;
      sc[3] += x;
    }
  }
  if (r >= valid) sc[0] = sc[1] = -INFINITY;
  if (r + 8 >= valid) sc[2] = sc[3] = -INFINITY;
  float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const float mn0 = fmaxf(s.m[0], mx0), mn1 = fmaxf(s.m[1], mx1);
  const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
  const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
  const float al0 = ex2(s.m[0] - mu0), al1 = ex2(s.m[1] - mu1);
  s.m[0] = mn0;
  s.m[1] = mn1;
  const uint32_t p01 = pack_bf16(ex2(sc[0] - mu0), ex2(sc[1] - mu1));
  const uint32_t p23 = pack_bf16(ex2(sc[2] - mu0), ex2(sc[3] - mu1));
  // the normaliser sums the same bf16-rounded weights the P.V product uses
  s.l[0] = s.l[0] * al0 + bf16_lo(p01) + bf16_lo(p23);
  s.l[1] = s.l[1] * al1 + bf16_hi(p01) + bf16_hi(p23);
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    s.acc[mt][0] *= al0;
    s.acc[mt][1] *= al1;
    s.acc[mt][2] *= al0;
    s.acc[mt][3] *= al1;
  }
  const uint32_t b0 = movmatrix_trans(p01);   // P^T rows: tokens 2c, 2c+1; column: head r
  const uint32_t b1 = movmatrix_trans(p23);   // tokens 2c+8, 2c+9
  // Tokens past `valid` may hold stale cache contents; zero their V lanes so
  // 0 * (non-finite) never reaches the accumulator.
  uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
  if (valid < kBlockTokens) {
    mlo = (2 * c < valid ? 0x0000ffffu : 0u) | (2 * c + 1 < valid ? 0xffff0000u : 0u);
    mhi = (2 * c + 8 < valid ? 0x0000ffffu : 0u) | (2 * c + 9 < valid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    uint32_t a0, a1, a2, a3;
    ldsm_x4_trans(vtile + swz(vrow, mt * 2 + vj), a0, a1, a2, a3);
    mma_bf16_16816(s.acc[mt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, b0, b1);
  }
}

// Writes the warp's state to the reduction buffers (heads padded to 8).
template <int D>
__device__ __forceinline__ void mma_stash(MmaState<D> &s, float *red_acc, float *red_m,
                                          float *red_l, int lane) {
  const int r = lane >> 2, c = lane & 3;
  float l0 = s.l[0], l1 = s.l[1];
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o);
  }
  if (r == 0) {
    red_m[2 * c] = s.m[0];
    red_m[2 * c + 1] = s.m[1];
    red_l[2 * c] = l0;
    red_l[2 * c + 1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int d0 = mt * 16 + r;
    red_acc[(2 * c) * D + d0] = s.acc[mt][0];
    red_acc[(2 * c + 1) * D + d0] = s.acc[mt][1];
    red_acc[(2 * c) * D + d0 + 8] = s.acc[mt][2];
    red_acc[(2 * c + 1) * D + d0 + 8] = s.acc[mt][3];
  }
}

// ---- SIMT consumer ----------------------------------------------------------
// Sum over the warp of v[h] for h = lane / (32/G): reduce-scatter halves the
// set of heads at each butterfly step, then the remaining lanes of a head add.
template <int G>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int lane) {
#pragma unroll
  for (int n = G, o = 16; n > 1; n >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float x = v[0];
#pragma unroll
  for (int o = 16 / G; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T, int D, int G>
struct SimtState {
  static constexpr int DPL = D / 32;
  float qf[G][DPL];
  float acc[G][DPL];
  float m, l;
};

// Loads the lane's DPL consecutive elements of token row `row` from a tile.
template <typename T, int DPL>
__device__ __forceinline__ void simt_load_row(const char *tile, int row, int lane,
                                              float (&x)[DPL]) {
  const int byte = lane * DPL * static_cast<int>(sizeof(T));
  const char *ptr = tile + swz(row, byte >> 4) + (byte & 15);
  if constexpr (sizeof(T) == 2) {
    if constexpr (DPL == 4) {
      const uint2 w = *reinterpret_cast<const uint2 *>(ptr);
      x[0] = bf16_lo(w.x);
      x[1] = bf16_hi(w.x);
      x[2] = bf16_lo(w.y);
      x[3] = bf16_hi(w.y);
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t *>(ptr);
      x[0] = bf16_lo(w);
      x[1] = bf16_hi(w);
    }
  } else {
    if constexpr (DPL == 4) {
      const float4 w = *reinterpret_cast<const float4 *>(ptr);
      x[0] = w.x;
      x[1] = w.y;
      x[2] = w.z;
      x[3] = w.w;
    } else {
      const float2 w = *reinterpret_cast<const float2 *>(ptr);
      x[0] = w.x;
      x[1] = w.y;
    }
  }
}

// ---- whole-step kernels: a1 + a2 inside the attention kernel ---------------
// Rotated queries of unit (b, g), built by the consumer threads in place in
// shared memory qs [G][D]: the producer put the raw rows and the row's
// position there ahead of the segment (loaded one segment early), so this
// costs no global round trip, only the angles and one barrier.  Storage type
// T, rounded once as pkv_rope does; the part that owns the unit's first page
// also reports the rotated rows in q_rot_out.
template <typename T, int D, int NTHR>
__device__ __forceinline__ void fused_rotate_q(const AttnParams &p, const unsigned long long *turns,
                                               int b, int g, uint32_t pos, bool report, T *qs,
                                               int tid) {
  constexpr int half = D / 2;
  constexpr int KM = (8 * half + NTHR - 1) / NTHR;   // pairs per thread (G <= 8)
  const int npairs = p.G * half;
  T *qo = static_cast<T *>(p.q_rot_out) + (static_cast<size_t>(b) * p.Hq + g * p.G) * D;
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    const int e = tid + k * NTHR;
    if (e < npairs) {
      const int h = e / half, i = e - h * half;
      float c, s, y1, y2;
      rope_cossin(pos, turns[i], &c, &s);
      rope_rotate(to_f32(qs[h * D + i]), to_f32(qs[h * D + half + i]), c, s, &y1, &y2);
      const T t1 = from_f32<T>(y1), t2 = from_f32<T>(y2);
      qs[h * D + i] = t1;
      qs[h * D + half + i] = t2;
      if (report) {
        qo[h * D + i] = t1;
        qo[h * D + half + i] = t2;
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NTHR) : "memory");
}

// The new token of unit (b, g), appended by the 32 lanes of the producer warp
// of the part that owns the unit's last page -- the only part that reads that
// page.  fetch() loads everything at the start of the segment; put() (called
// just before the batch that loads the last page) rotates the key, writes key
// and value into the cache slot (and the key into k_rot_out) and fences the
// generic-proxy stores ahead of the page's TMA (async-proxy) load.
template <typename T, int D>
struct FusedAppend {
  static constexpr int KP = (D / 2 + 31) / 32;   // pairs per lane
  static constexpr int KV = (D + 31) / 32;       // values per lane
  T x1[KP], x2[KP], v[KV];   // as loaded: converted only when put() needs them
  long long slot;
  uint32_t pos;

  __device__ __forceinline__ void fetch(const AttnParams &p, int b, int g, int lane) {
    constexpr int half = D / 2;
    slot = p.slots[b];
    pos = static_cast<uint32_t>(p.positions[b]);
    const T *kn = static_cast<const T *>(p.k_new) + (static_cast<size_t>(b) * p.Hkv + g) * D;
    const T *vn = static_cast<const T *>(p.v_new) + (static_cast<size_t>(b) * p.Hkv + g) * D;
#pragma unroll
    for (int k = 0; k < KP; ++k) {
      const int i = lane + 32 * k;
      if (i < half) {
        x1[k] = kn[i];
        x2[k] = kn[half + i];
      }
    }
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int i = lane + 32 * k;
      if (i < D) v[k] = vn[i];
    }
  }

  __device__ __forceinline__ void put(const AttnParams &p, const unsigned long long *turns, int b,
                                      int g, int lane) {
    constexpr int half = D / 2;
    if (slot >= p.num_slots) {
      if (lane == 0) set_dev_err(p.err, PKV_DEVERR_BAD_SLOT);
    } else if (slot >= 0) {
      const long long blk = slot / kBlockTokens;
      const size_t row =
          (static_cast<size_t>(blk * p.Hkv + g) * kBlockTokens + (slot - blk * kBlockTokens)) * D;
      T *kc = static_cast<T *>(p.k_cache_w) + row;
      T *vc = static_cast<T *>(p.v_cache_w) + row;
      T *ko = static_cast<T *>(p.k_rot_out) + (static_cast<size_t>(b) * p.Hkv + g) * D;
#pragma unroll
      for (int k = 0; k < KP; ++k) {
        const int i = lane + 32 * k;
        if (i < half) {
          float c, s, y1, y2;
          rope_cossin(pos, turns[i], &c, &s);
          rope_rotate(to_f32(x1[k]), to_f32(x2[k]), c, s, &y1, &y2);
          const T t1 = from_f32<T>(y1), t2 = from_f32<T>(y2);
          kc[i] = t1;
          kc[half + i] = t2;
          ko[i] = t1;
          ko[half + i] = t2;
        }
      }
#pragma unroll
      for (int k = 0; k < KV; ++k) {
        const int i = lane + 32 * k;
        if (i < D) vc[i] = v[k];
      }
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncwarp();
  }
};

template <int D>
__device__ __forceinline__ void mma_begin_smem(MmaState<D> &s, const __nv_bfloat16 *qs, int G,
                                               int lane) {
  const int r = lane >> 2, c = lane & 3;
  const bool real = r < G;
  const __nv_bfloat16 *qrow = qs + (real ? r : 0) * D;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 2 * c);
    s.qb[ks][0] = real ? w[0] : 0u;
    s.qb[ks][1] = real ? w[4] : 0u;
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) s.acc[mt][e] = 0.f;
  s.m[0] = s.m[1] = -INFINITY;
  s.l[0] = s.l[1] = 0.f;
}

template <typename T, int D, int G>
__device__ __forceinline__ void simt_begin_smem(SimtState<T, D, G> &s, const T *qs, int Greal,
                                                float scale_log2, int lane) {
  constexpr int DPL = D / 32;
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      s.qf[h][e] = h < Greal ? to_f32(qs[h * D + lane * DPL + e]) * scale_log2 : 0.f;
      s.acc[h][e] = 0.f;
    }
  s.m = -INFINITY;
  s.l = 0.f;
}

template <typename T, int D, int G>
__device__ __forceinline__ void simt_begin(SimtState<T, D, G> &s, const AttnParams &p, int b,
                                           int g, int lane) {
  constexpr int DPL = D / 32;
  const T *q = static_cast<const T *>(p.q) + (static_cast<size_t>(b) * p.Hq + g * p.G) * D;
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      s.qf[h][e] = h < p.G ? to_f32(q[h * D + lane * DPL + e]) * p.scale_log2 : 0.f;
      s.acc[h][e] = 0.f;
    }
  s.m = -INFINITY;
  s.l = 0.f;
}

template <typename T, int D, int G>
__device__ __forceinline__ void simt_page(SimtState<T, D, G> &s, const AttnParams &p,
                                          const char *ktile, const char *vtile, int valid, int b,
                                          int t0, int lane, float *pbuf, float *abuf,
                                          bool may_bias) {
  constexpr int DPL = D / 32;
  constexpr int LPH = 32 / G;
  float sc[kBlockTokens];
#pragma unroll
  for (int i = 0; i < kBlockTokens; ++i) {
    float k[DPL];
    simt_load_row<T, DPL>(ktile, i, lane, k);
    float part[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) a = fmaf(s.qf[h][e], k[e], a);
      part[h] = a;
    }
    sc[i] = reduce_scatter<G>(part, lane);
  }
  const float *bias =
      may_bias && p.bias ? p.bias + static_cast<size_t>(b) * p.bias_stride + t0 : nullptr;
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < kBlockTokens; ++i) {
    if (i < valid) {
      if (bias) sc[i] += bias[i] * kLog2e;
    } else {
      sc[i] = -INFINITY;
    }
    mx = fmaxf(mx, sc[i]);
  }
  const float mn = fmaxf(s.m, mx);
  const float mu = mn == -INFINITY ? 0.f : mn;
  const float alpha = ex2(s.m - mu);
  s.m = mn;
  float psum = 0.f;
  const int hl = lane / LPH;
  const bool writer = (lane % LPH) == 0;
#pragma unroll
  for (int i = 0; i < kBlockTokens; ++i) {
    const float pi = ex2(sc[i] - mu);
    psum += pi;
    if (writer) pbuf[i * 8 + hl] = pi;
  }
  s.l = s.l * alpha + psum;
  if (writer) abuf[hl] = alpha;
  __syncwarp();
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float a = abuf[h];
#pragma unroll
    for (int e = 0; e < DPL; ++e) s.acc[h][e] *= a;
  }
  for (int i = 0; i < valid; ++i) {
    float v[DPL];
    simt_load_row<T, DPL>(vtile, i, lane, v);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float ph = pbuf[i * 8 + h];
#pragma unroll
      for (int e = 0; e < DPL; ++e) s.acc[h][e] = fmaf(ph, v[e], s.acc[h][e]);
    }
  }
  __syncwarp();
}

template <typename T, int D, int G>
__device__ __forceinline__ void simt_stash(SimtState<T, D, G> &s, float *red_acc, float *red_m,
                                           float *red_l, int lane) {
  constexpr int DPL = D / 32;
  constexpr int LPH = 32 / G;
  if (lane % LPH == 0) {
    red_m[lane / LPH] = s.m;
    red_l[lane / LPH] = s.l;
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < DPL; ++e) red_acc[h * D + lane * DPL + e] = s.acc[h][e];
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// KIND 0: MMA consumer (T must be bf16, G <= 8 at run time).
// KIND 1: SIMT consumer with compile-time group G.
// FUSE: whole-step kernel -- also rotates the step's q/k and appends k/v
// (a1 + a2), so a decode step is one launch.
// PLAN: the launch has a plan that is not checked and no attention bias
// (p.plan != nullptr, !p.check_plan, p.bias == nullptr): the row-length scan,
// the plan check and the bias are compiled out, and the smaller kernel runs
// faster (its instructions come cold at both ends of every CTA).
template <typename T, int D, int NW, int NS, int KIND, int G, bool FUSE, bool PLAN>
__global__ void __launch_bounds__((NW + 1) * 32, KIND == 0 ? 2 : 1)
    attn_split_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v,
                      const __grid_constant__ AttnParams p) {
  using Q = Geo<T, D, NW, NS>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float *red_acc = reinterpret_cast<float *>(smem + Q::kOffRedAcc);
  float *red_m = reinterpret_cast<float *>(smem + Q::kOffRedM);
  float *red_l = reinterpret_cast<float *>(smem + Q::kOffRedL);
  float *pbuf_all = reinterpret_cast<float *>(smem + Q::kOffPBuf);
  float *abuf_all = reinterpret_cast<float *>(smem + Q::kOffABuf);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Q::kOffBars);
  uint64_t *empty = full + NS;
  uint64_t *segfull = reinterpret_cast<uint64_t *>(smem + Q::kOffSegBars);
  uint64_t *segempty = segfull + Q::kSegSlots;
  volatile int *stage_bad = reinterpret_cast<volatile int *>(smem + Q::kOffBad);
  int *scan = reinterpret_cast<int *>(smem + Q::kOffScan);
  int *lens_s = reinterpret_cast<int *>(smem + Q::kOffLens);
  unsigned long long *turns_s = reinterpret_cast<unsigned long long *>(smem + Q::kOffTurns);
  volatile int *misc = reinterpret_cast<volatile int *>(smem + Q::kOffMisc);  // b0, rowoff0, abort
  int *stage_pg = reinterpret_cast<int *>(smem + Q::kOffPg);   // [NS], then [kSegSlots]
  int *slot_seg = stage_pg + NS;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int C = p.num_parts;
  const bool has_bias = !PLAN && p.bias != nullptr;
  // a kernel launched after this one as a programmatic dependent (the next
  // layer's RoPE/append) may start now; it waits for this grid before it reads
  // anything this grid produces
  if (!FUSE) pdl_launch_dependents();

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < Q::kSegSlots; ++s) {
      mbar_init(&segfull[s], 1);
      mbar_init(&segempty[s], NW);   // one arrival per consumer warp
    }
    misc[0] = -1;
    misc[1] = 0;
    misc[2] = 0;   // a wait gave up: stop
    misc[3] = 0;   // the producer warp has issued its last copy
    for (int s = 0; s < NS + Q::kSegSlots; ++s) stage_pg[s] = -1;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == NW && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }
  if constexpr (FUSE) {   // read after the block-wide barrier below
    for (int i = tid; i < D / 2; i += Q::kThreads) turns_s[i] = p.turns[i];
  }

  // The partition balances pages plus seg_cost per unit: a unit of n pages
  // spans n + seg_cost positions, the first seg_cost of them holding no page
  // (a part that starts a unit pays for the boundary with fewer pages).
  const int A = p.seg_cost;
  auto upos = [A](int n) { return n > 0 ? n + A : 0; };
  const int nthreads = Q::kThreads;
  // ---- host-planned partition: this part's record (one read; its block ids
  // let the producer issue the first TMA loads without a block-table read) ----
  const bool planned = PLAN || p.plan != nullptr;
  const int32_t *rec = planned ? p.plan + static_cast<size_t>(blockIdx.x) * PKV_PLAN_INTS : nullptr;
  int4 rec_h = make_int4(-1, 0, 0, 0), rec_p = make_int4(0, 0, 0, 0);
  int plan_ids = -1;
  if (planned) {
    rec_h = __ldcg(reinterpret_cast<const int4 *>(rec));       // row, row offset, L, next L
    rec_p = __ldcg(reinterpret_cast<const int4 *>(rec) + 1);   // P (int64)
    // the producer's first block ids go out in the same round trip
    if (warp == NW && lane < kPlanIds) plan_ids = __ldcg(rec + 8 + lane);
  }
  // ---- otherwise (or to check the plan): page counts of all rows,
  // per-thread chunk sums, block-wide scan ----
  const bool scanned = !PLAN && (!planned || p.check_plan);
  long long P_dev = 0;
  if (scanned) {
    const int chunk = (p.B + nthreads - 1) / nthreads;
    const int r0 = min(p.B, tid * chunk), r1 = min(p.B, r0 + chunk);
    int mysum = 0;
    for (int b = r0; b < r1; ++b) {
      bool bad;
      const int len = p.seq_lens[b];
      if (b < Q::kLensCache) lens_s[b] = len;   // kept for the row search and the producer
      mysum += upos(pages_of_len(len, p.bt_stride, has_bias, p.bias_stride, &bad));
      if (bad && blockIdx.x == 0) set_dev_err(p.err, PKV_DEVERR_BAD_LEN);
    }
    int incl = mysum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < nthreads / 32; ++w) {
      const int t = scan[w];
      if (w < warp) before += t;
      total += t;
    }
    const long long excl = before + incl - mysum;
    P_dev = static_cast<long long>(total) * p.Hkv;
    const long long s0 = div_floor(P_dev * blockIdx.x, C);
    if (s0 < div_floor(P_dev * (blockIdx.x + 1), C) && mysum > 0 && s0 >= excl * p.Hkv &&
        s0 < (excl + mysum) * p.Hkv) {
      long long acc = excl;
      for (int b = r0; b < r1; ++b) {
        bool bad;
        const int len = b < Q::kLensCache ? lens_s[b] : p.seq_lens[b];   // own rows: written above
        const int n = upos(pages_of_len(len, p.bt_stride, has_bias, p.bias_stride, &bad));
        if (s0 < (acc + n) * p.Hkv) {
          misc[0] = b;
          misc[1] = static_cast<int>(acc);
          break;
        }
        acc += n;
      }
    }
    // rows with no token (or an invalid length) output zeros; part c clears
    // rows c, c + C, ...
    for (int b = blockIdx.x; b < p.B; b += C) {   // (after the barrier above: lens_s is complete)
      bool bad;
      const int len = b < Q::kLensCache ? lens_s[b] : p.seq_lens[b];
      if (pages_of_len(len, p.bt_stride, has_bias, p.bias_stride, &bad) == 0) {
        T *o = static_cast<T *>(p.out) + static_cast<size_t>(b) * p.Hq * D;
        for (int e = tid; e < p.Hq * D; e += nthreads) o[e] = from_f32<T>(0.f);
      }
    }
  }
  const long long P_plan =
      static_cast<long long>(static_cast<uint32_t>(rec_p.x)) | (static_cast<long long>(rec_p.y) << 32);
  __syncthreads();
  // with a plan, the producer starts from it; checked plans must agree with
  // the partition derived here (otherwise that one is used, and flagged)
  bool use_plan = planned;
  if (!PLAN && planned && p.check_plan) {
    bool same = P_plan == P_dev;
    if (same && div_floor(P_dev * blockIdx.x, C) < div_floor(P_dev * (blockIdx.x + 1), C)) {
      const int b = misc[0];
      same = b >= 0 && b == rec_h.x && misc[1] == rec_h.y && rec_h.z == p.seq_lens[b] &&
             (b + 1 >= p.B || rec_h.w == p.seq_lens[b + 1]);
    }
    if (!same) {
      use_plan = false;
      if (tid == 0) set_dev_err(p.err, PKV_DEVERR_BAD_PLAN);
    }
  }
  const long long P = use_plan ? P_plan : P_dev;
  const long long start = div_floor(P * blockIdx.x, C);
  const long long end = div_floor(P * (blockIdx.x + 1), C);
  if (blockIdx.x == 0 && tid == 0) {
    // total position count, for the merge to tell empty parts (C > P) from real ones
    p.meta[2 * p.B * p.Hkv] = static_cast<int32_t>(P & 0xffffffffll);
    p.meta[2 * p.B * p.Hkv + 1] = static_cast<int32_t>(P >> 32);
  }
  // rows with no token: without the scan, the consumer warps clear them (off
  // the producer's path)
  if (!scanned && warp < NW) {
    for (int b = blockIdx.x; b < p.B; b += C) {
      bool bad;
      if (pages_of_len(p.seq_lens[b], p.bt_stride, has_bias, p.bias_stride, &bad) == 0) {
        T *o = static_cast<T *>(p.out) + static_cast<size_t>(b) * p.Hq * D;
        for (int e = tid; e < p.Hq * D; e += NW * 32) o[e] = from_f32<T>(0.f);
      }
      if (bad && tid == 0) set_dev_err(p.err, PKV_DEVERR_BAD_LEN);
    }
  }
  if (start >= end) return;
  if (use_plan && rec_h.x >= p.B) {   // a record naming no row: never read outside seq_lens
    if (tid == 0) set_dev_err(p.err, PKV_DEVERR_BAD_PLAN);
    return;
  }
  const int first_row = use_plan ? rec_h.x : misc[0];
  if (first_row < 0) {   // no owner of `start` (never expected)
    if (tid == 0) set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
    return;
  }

  if (warp == NW) {
    // ======================= producer warp =======================
    // Walks the part's unit segments.  For each it hands the consumers a
    // segment slot (header + the unit's query rows) and streams
    // the pages into the ring.  Row lengths of the part's first 64 rows and the
    // next segment's first block ids are read ahead, so a unit boundary costs
    // no dependent global read.
    constexpr int kBatch = NS >= 8 ? 4 : (NS >= 2 ? NS / 2 : 1);
    const uint64_t l2_stream = l2_policy_evict_first();
    const int b0 = first_row;
    // row lengths: the prologue's copy for the first rows (or the plan's for
    // rows b0 and b0 + 1), read ahead beyond
    const int lc = scanned ? Q::kLensCache : 0;
    const int rl0 = b0 + lane < p.B && b0 + lane >= lc ? p.seq_lens[b0 + lane] : 0;
    const int rl1 = b0 + 32 + lane < p.B && b0 + 32 + lane >= lc ? p.seq_lens[b0 + 32 + lane] : 0;
    auto row_len = [&](int b) {   // b is warp-uniform
      if (b < lc) return lens_s[b];
      if (use_plan && b == b0) return rec_h.z;
      if (use_plan && b == b0 + 1) return rec_h.w;
      const int r = b - b0;
      if (r < 32) return __shfl_sync(0xffffffffu, rl0, r);
      if (r < 64) return __shfl_sync(0xffffffffu, rl1, r - 32);
      return p.seq_lens[b];
    };
    auto advance = [&](UnitCursor &c) {   // the next unit, with the read-ahead lengths
      c.off += c.n + A;
      if (++c.g < p.Hkv) return;
      c.g = 0;
      bool bad;
      for (++c.b; c.b < p.B; ++c.b) {
        c.n = pages_of_len(row_len(c.b), p.bt_stride, has_bias, p.bias_stride, &bad);
        if (c.n > 0) return;
      }
      c.n = 0;
    };
    UnitCursor u;
    {
      const long long rowoff = use_plan ? rec_h.y : misc[1];
      bool bad;
      u.b = b0;
      u.n = pages_of_len(row_len(b0), p.bt_stride, has_bias, p.bias_stride, &bad);
      u.g = static_cast<int>(div_floor(start - rowoff * p.Hkv, u.n + A));
      u.off = rowoff * p.Hkv + static_cast<long long>(u.g) * (u.n + A);   // first position
    }
    const uint32_t qbytes = static_cast<uint32_t>(p.G * D * sizeof(T));
    // FUSE: the raw query rows of the next segment's unit (16-byte pieces,
    // lane-strided) and its row's position, loaded while the current segment
    // streams and stored into the segment slot when it is handed over
    constexpr int kQV = FUSE ? (8 * D * static_cast<int>(sizeof(T))) / (16 * 32) : 1;
    uint4 qraw[kQV];
    uint32_t qpos = 0;
    auto fetch_q = [&](int b, int g) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          static_cast<const T *>(p.q_new) + (static_cast<size_t>(b) * p.Hq + g * p.G) * D);
      const int nv = static_cast<int>(qbytes / 16);
#pragma unroll
      for (int i = 0; i < kQV; ++i)
        qraw[i] = lane + 32 * i < nv ? src[lane + 32 * i] : make_uint4(0u, 0u, 0u, 0u);
      qpos = static_cast<uint32_t>(p.positions[b]);
    };
    int x = 0, k = 0;
    bool aborted = false, waited = FUSE;
    // pages [j0, j1) of unit u lie in this part's positions [start, end); the
    // unit's pages sit at positions off + A .. off + A + n - 1.  Only a part
    // that lies inside one unit's first A positions has no page at all.
    int j0 = static_cast<int>(max(0ll, start - u.off - A));
    int j1 = static_cast<int>(min(static_cast<long long>(u.n), end - u.off - A));
    bool last = false;
    if (j1 <= j0) {   // no page: tell the consumers and stop
      j0 = j1 = 0;
      last = true;
    }
    // block ids of the first chunk of pages: the plan's first kPlanIds (the
    // table read of the next chunk is then in flight behind them), or the first
    // 32 read from the table (and, when the plan is checked, compared with it)
    int ids, chunk = 32;
    if (PLAN || (use_plan && !p.check_plan)) {
      ids = plan_ids;
      chunk = kPlanIds;
    } else {
      ids = (j0 + lane < j1) ? p.block_tables[static_cast<size_t>(u.b) * p.bt_stride + j0 + lane]
                             : -1;
      if (use_plan && lane < kPlanIds && j0 + lane < j1 && plan_ids != ids)
        set_dev_err(p.err, PKV_DEVERR_BAD_PLAN);
    }
    if constexpr (FUSE) {
#pragma unroll
      for (int i = 0; i < kQV; ++i) qraw[i] = make_uint4(0u, 0u, 0u, 0u);
      if (j1 > j0) fetch_q(u.b, u.g);
    }
    while (!aborted) {
      const int32_t *bt = p.block_tables + static_cast<size_t>(u.b) * p.bt_stride;
      // read ahead: the next unit (if the part reaches its pages) and its
      // first 32 block ids
      const long long noff = u.off + u.n + A;
      const bool more = !last && end > noff + A;
      last = !more;
      UnitCursor nx = u;
      int nj1 = 0, nids = -1;
      if (more) {
        advance(nx);
        nj1 = static_cast<int>(min(static_cast<long long>(nx.n), end - nx.off - A));
        nids = lane < nj1 ? p.block_tables[static_cast<size_t>(nx.b) * p.bt_stride + lane] : -1;
      }
      const int L = row_len(u.b);
      FusedAppend<T, D> app;
      if constexpr (FUSE) {
        if (j1 == u.n) app.fetch(p, u.b, u.g, lane);   // this part owns the last page
      }
      bool sent = false;
      // the segment slot: header, then the query rows (after the first batch
      // of pages, so the first pages are on their way before any wait)
      auto send_segment = [&]() {
        const int slot = k % Q::kSegSlots;
        unsigned char *sp = smem + Q::kOffSeg + slot * Q::kSegBytes;
        bool dead = false;
        if (lane == 0) {
          const uint32_t sph = static_cast<uint32_t>(k / Q::kSegSlots) & 1u;
          dead = misc[2] != 0;
          if (!dead && !mbar_wait_bounded(&segempty[slot], sph ^ 1u, p.wait_limit)) {
            misc[2] = 1;
            dead = true;
            set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
          }
        }
        if constexpr (FUSE) {
          // the raw query rows, by every lane, once lane 0 has seen the slot
          // free (the warp barrier orders its wait before the other lanes'
          // stores)
          __syncwarp();
          if (!__shfl_sync(0xffffffffu, dead, 0)) {
            uint4 *dst = reinterpret_cast<uint4 *>(sp + 64);
            const int nv = static_cast<int>(qbytes / 16);
#pragma unroll
            for (int i = 0; i < kQV; ++i)
              if (lane + 32 * i < nv) dst[lane + 32 * i] = qraw[i];
          }
          __syncwarp();
        }
        if (lane == 0) {
          // once anything has given up, nothing more is handed over (the
          // consumers stop too), so no barrier gets an arrival for a phase the
          // other side never finished
          if (!dead) {
            int *h = reinterpret_cast<int *>(sp);
            h[0] = u.b;
            h[1] = u.g;
            h[2] = u.n;
            h[3] = L;
            h[4] = j0;
            h[5] = j1;
            *reinterpret_cast<long long *>(h + 6) = u.off;
            // parts spanned by the unit's pages (two 64-bit divisions, off the
            // consumers' path), and whether this is the part's last segment
            const int cf = part_of(u.off + A, P, C);
            h[8] = cf;
            h[9] = part_of(u.off + A + u.n - 1, P, C) - cf + 1;
            h[10] = last ? 1 : 0;
            h[11] = static_cast<int>(qpos);
            if (!FUSE) {
              if (!waited) {
                pdl_wait();   // the query rows come from the kernel before this one
                waited = true;
              }
              mbar_arrive_expect_tx(&segfull[slot], qbytes);
              bulk_copy_g2s(smem_u32(sp + 64),
                            static_cast<const T *>(p.q) +
                                (static_cast<size_t>(u.b) * p.Hq + u.g * p.G) * D,
                            qbytes, &segfull[slot]);
            } else {
              mbar_arrive(&segfull[slot]);
            }
            slot_seg[slot] = k;
          }
        }
        __syncwarp();
      };
      for (int jb = j0; jb < j1 && !aborted; jb += chunk, chunk = 32) {
        const int cur_ids = ids;
        ids = (jb + chunk + lane < j1) ? bt[jb + chunk + lane] : -1;
        const int cnt = min(chunk, j1 - jb);
        // pages go out kBatch at a time, lane l < kBatch taking page i + l, so
        // the barrier waits, arrivals and TMA issues of a batch share warp
        // instructions (one page per lane-instruction costs ~600 cycles)
        for (int i = 0; i < cnt; i += kBatch) {
          if constexpr (FUSE) {
            // this part owns the unit's last page: append the step's token
            // before the batch that loads that page
            if (j1 == u.n && jb + i <= u.n - 1 && u.n - 1 < jb + i + kBatch)
              app.put(p, turns_s, u.b, u.g, lane);
          }
          const int blk = __shfl_sync(0xffffffffu, cur_ids, (i + lane) & 31);
          if (lane < kBatch && i + lane < cnt) {
            const int xx = x + (jb - j0) + i + lane;
            const int st = xx % NS;
            const uint32_t ph = static_cast<uint32_t>(xx / NS) & 1u;
            bool dead = misc[2] != 0;
            if (!dead && !mbar_wait_bounded(&empty[st], ph ^ 1u, p.wait_limit)) {
              misc[2] = 1;
              dead = true;
              set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
            }
            const bool ok = !dead && blk >= 0 && blk < p.num_blocks;
            if (!dead) {
              stage_bad[st] = ok ? 0 : 1;
              stage_pg[st] = xx;
            }
            if (ok) {
              // the last page of a unit holds the token appended by the kernel
              // before this one: wait for that grid before reading it
              if (!FUSE && jb + i + lane == u.n - 1) pdl_wait();
              mbar_arrive_expect_tx(&full[st], Q::kStageBytes);
              const uint32_t kdst = smem_u32(smem + st * Q::kStageBytes);
              const uint32_t vdst = kdst + Q::kTileBytes;
              const int y = (blk * p.Hkv + u.g) * kBlockTokens;
#pragma unroll
              for (int sub = 0; sub < Q::kSubs; ++sub) {
                tma_load_2d_hint(kdst + sub * Q::kSubBytes, &tmap_k, sub * Q::kSubCols, y,
                                 &full[st], l2_stream);
                tma_load_2d_hint(vdst + sub * Q::kSubBytes, &tmap_v, sub * Q::kSubCols, y,
                                 &full[st], l2_stream);
              }
            } else if (!dead) {
              set_dev_err(p.err, PKV_DEVERR_BAD_BLOCK);
              mbar_arrive(&full[st]);
            }
          }
          __syncwarp();
          if (!sent) {
            send_segment();
            sent = true;
            if constexpr (FUSE) {
              if (more) fetch_q(nx.b, nx.g);
            }
          }
        }
        aborted = __shfl_sync(0xffffffffu, misc[2], 0) != 0;
      }
      if (!sent) {   // (a part with no page, or aborted before a batch)
        send_segment();
        if constexpr (FUSE) {
          if (more) fetch_q(nx.b, nx.g);
        }
      }
      x += j1 - j0;
      ++k;
      if (!more) break;
      u = nx;
      j0 = 0;
      j1 = nj1;
      ids = nids;
    }
    // Every copy this warp issued must land before the CTA exits.  Normally
    // the consumers wait for all of them anyway; consumers that gave up a
    // wait may not.  The producer marks itself finished, then looks for an
    // abort; a consumer that aborts marks that, then looks for a finished
    // producer (store, sequentially consistent fence, load on both sides): at
    // least one of them sees the other and drains.
    __syncwarp();
    if (lane == 0) {
      fence_sc_cta();   // this warp's stage and slot records before the mark
      misc[3] = 1;
      fence_sc_cta();
    }
    if (__shfl_sync(0xffffffffu, misc[2], 0) != 0)
      drain_copies<NS, Q::kSegSlots>(full, segfull, stage_pg, slot_seg, lane);
    return;
  }

  // ======================= consumer warps =======================
  float *my_acc = red_acc + warp * Q::kHeadsPad * D;
  float *my_m = red_m + warp * Q::kHeadsPad;
  float *my_l = red_l + warp * Q::kHeadsPad;
  float *pbuf = pbuf_all + warp * kBlockTokens * Q::kHeadsPad;
  float *abuf = abuf_all + warp * Q::kHeadsPad;
  constexpr int kConsumers = NW * 32;

  int pend_u[2], pend_c[2], pend_n[2], pend_b[2], pend_g[2];   // at most two (see below)
  int npend = 0;
  int x = 0, k = 0;
  // One consumer thread waits for each segment slot; the others read it after
  // the consumer barrier that ends the previous segment, so every consumer
  // sees the same header and the same stop decision (misc[6]).
  auto wait_segment = [&](int kk) {
    const int slot = kk % Q::kSegSlots;
    const uint32_t sph = static_cast<uint32_t>(kk / Q::kSegSlots) & 1u;
    bool ok = misc[2] == 0;
    if (ok && !mbar_wait_bounded(&segfull[slot], sph, p.wait_limit)) {
      consumer_abort<NS, Q::kSegSlots>(misc, full, segfull, stage_pg, slot_seg);
      set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
      ok = false;
    }
    misc[6] = ok ? 0 : 1;
  };
  if (tid == 0) wait_segment(0);
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
  while (misc[6] == 0) {
    const int slot = k % Q::kSegSlots;
    const unsigned char *sp = smem + Q::kOffSeg + slot * Q::kSegBytes;
    const int *hdr = reinterpret_cast<const int *>(sp);
    UnitCursor u;
    u.b = hdr[0];
    u.g = hdr[1];
    u.n = hdr[2];
    const int L = hdr[3];
    const int j0 = hdr[4], j1 = hdr[5];
    u.off = *reinterpret_cast<const long long *>(hdr + 6);
    const int c_first = hdr[8], nseg = hdr[9];
    const bool seg_last = hdr[10] != 0;
    if (j1 <= j0) break;   // a part without pages (every consumer read the same header)
    const T *qslot = reinterpret_cast<const T *>(sp + 64);
    // ---- this warp's pages of the segment ----
    if constexpr (KIND == 0) {
      MmaState<D> s;
      if constexpr (FUSE) {
        T *qs = reinterpret_cast<T *>(const_cast<unsigned char *>(sp) + 64);
        fused_rotate_q<T, D, kConsumers>(p, turns_s, u.b, u.g, static_cast<uint32_t>(hdr[11]),
                                         j0 == 0, qs, tid);
        mma_begin_smem<D>(s, reinterpret_cast<const __nv_bfloat16 *>(qs), p.G, lane);
      } else {
        mma_begin_smem<D>(s, reinterpret_cast<const __nv_bfloat16 *>(qslot), p.G, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&segempty[slot]);
      int j = j0 + ((warp - x % NW) + NW) % NW;
      for (; j < j1; j += NW) {
        const int xx = x + (j - j0);
        const int st = xx % NS;
        const uint32_t ph = static_cast<uint32_t>(xx / NS) & 1u;
        bool ready = !misc[2];
        if (ready && !mbar_wait_bounded(&full[st], ph, p.wait_limit)) {
          consumer_abort<NS, Q::kSegSlots>(misc, full, segfull, stage_pg, slot_seg);
          set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
          ready = false;
        }
        if (ready && !stage_bad[st]) {
          const uint32_t kt = smem_u32(smem + st * Q::kStageBytes);
          mma_page<D>(s, p, kt, kt + Q::kTileBytes, min(kBlockTokens, L - j * kBlockTokens), u.b,
                      j * kBlockTokens, lane, !PLAN);
        }
        __syncwarp();
        // a stage is handed back only after its page was seen to land
        if (lane == 0 && ready) mbar_arrive(&empty[st]);
      }
      mma_stash<D>(s, my_acc, my_m, my_l, lane);
    } else {
      SimtState<T, D, G> s;
      if constexpr (FUSE) {
        T *qs = reinterpret_cast<T *>(const_cast<unsigned char *>(sp) + 64);
        fused_rotate_q<T, D, kConsumers>(p, turns_s, u.b, u.g, static_cast<uint32_t>(hdr[11]),
                                         j0 == 0, qs, tid);
        simt_begin_smem<T, D, G>(s, qs, p.G, p.scale_log2, lane);
      } else {
        simt_begin_smem<T, D, G>(s, qslot, p.G, p.scale_log2, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&segempty[slot]);
      int j = j0 + ((warp - x % NW) + NW) % NW;
      for (; j < j1; j += NW) {
        const int xx = x + (j - j0);
        const int st = xx % NS;
        const uint32_t ph = static_cast<uint32_t>(xx / NS) & 1u;
        bool ready = !misc[2];
        if (ready && !mbar_wait_bounded(&full[st], ph, p.wait_limit)) {
          consumer_abort<NS, Q::kSegSlots>(misc, full, segfull, stage_pg, slot_seg);
          set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
          ready = false;
        }
        if (ready && !stage_bad[st]) {
          const char *kt = reinterpret_cast<const char *>(smem + st * Q::kStageBytes);
          simt_page<T, D, G>(s, p, kt, kt + Q::kTileBytes, min(kBlockTokens, L - j * kBlockTokens),
                             u.b, j * kBlockTokens, lane, pbuf, abuf, !PLAN);
        }
        __syncwarp();
        if (lane == 0 && ready) mbar_arrive(&empty[st]);
      }
      simt_stash<T, D, G>(s, my_acc, my_m, my_l, lane);
    }
    // ---- combine the consumer warps' states for this segment ----
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
    const int u_idx = u.b * p.Hkv + u.g;
    const int gq = p.G;
    // each output float4 combines the NW warp states of its head; the head's
    // rescale factors are recomputed by every thread that needs them (a few
    // shared loads and NW ex2), which costs less than a separate pass and a
    // barrier
    for (int e4 = tid; e4 < gq * (D / 4); e4 += kConsumers) {
      const int h = e4 / (D / 4), d4 = e4 - h * (D / 4);
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w * Q::kHeadsPad + h]);
      float f[NW];
      float den = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        f[w] = M == -INFINITY ? 0.f : ex2(red_m[w * Q::kHeadsPad + h] - M);
        den += f[w] * red_l[w * Q::kHeadsPad + h];
      }
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float4 a =
            *reinterpret_cast<const float4 *>(red_acc + (w * Q::kHeadsPad + h) * D + 4 * d4);
        o.x = fmaf(f[w], a.x, o.x);
        o.y = fmaf(f[w], a.y, o.y);
        o.z = fmaf(f[w], a.z, o.z);
        o.w = fmaf(f[w], a.w, o.w);
      }
      const float inv = den > 0.f ? __frcp_rn(den) : 0.f;
      o.x *= inv;
      o.y *= inv;
      o.z *= inv;
      o.w *= inv;
      if (nseg == 1) {
        store4<T>(static_cast<T *>(p.out) + (static_cast<size_t>(u.b) * p.Hq + u.g * gq + h) * D +
                      4 * d4,
                  o);
      } else {
        const size_t idx = static_cast<size_t>(u_idx) + blockIdx.x;
        *reinterpret_cast<float4 *>(p.o_part + (idx * gq + h) * D + 4 * d4) = o;
        if (d4 == 0) p.lse_part[idx * gq + h] = den > 0.f ? M + lg2(den) : -INFINITY;
      }
    }
    if (tid == 0 && j0 == 0) {
      p.meta[2 * u_idx] = c_first;
      p.meta[2 * u_idx + 1] = nseg;
    }
    if (nseg > 1 && p.fuse_merge && npend < 2) {
      // only the first and last segment of a part can belong to a unit split
      // across parts: remember it and merge after streaming, so merges never
      // stall the consumer warps while the producer keeps the ring full
      const int q = npend++;   // constant indices keep these in registers
      if (q == 0) {
        pend_u[0] = u_idx;
        pend_c[0] = c_first;
        pend_n[0] = nseg;
        pend_b[0] = u.b;
        pend_g[0] = u.g;
      } else {
        pend_u[1] = u_idx;
        pend_c[1] = c_first;
        pend_n[1] = nseg;
        pend_b[1] = u.b;
        pend_g[1] = u.g;
      }
    }
    x += j1 - j0;
    ++k;
    if (tid == 0) {
      if (!seg_last)
        wait_segment(k);
      else
        misc[6] = 1;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
  }
  if (npend == 0) return;
  // ---- a4 in the epilogue.  Both pending units (a part's first and last
  // segment) report at once: one release fence, both counter increments in
  // flight, one acquire fence.  A part among the last H of a unit to arrive
  // is one of its merge helpers (see merge_slice); helpers that are not the
  // last to arrive wait for the rest.  Then every slice this part merges goes
  // out in one pass. ----
  // (the segment loop ended with a consumer barrier: all partials are written)
  volatile int *roles = misc + 8;   // per pending unit: helper index (-1: none), H
  if (tid == 0) {
    fence_acq_rel_gpu();   // release this part's partials
    int prev[2];
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (q < npend) prev[q] = atom_add_relaxed_gpu(&p.counters[pend_u[q]], 1);
    fence_acq_rel_gpu();   // acquire the partials of the parts that arrived before
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      int r = -1, H = 1;
      if (q < npend) {
        const int n = real_parts(pend_c[q], pend_n[q], P, C);
        H = n < kHelperMinSplit ? 1 : merge_helpers(n, p.G * (D / 4), p.max_helpers);
        r = prev[q] - (n - H);
        if (r >= 0 && r < H - 1 && !wait_count(&p.counters[pend_u[q]], n, p.wait_limit)) {
          set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
          r = -1;   // (the counters stay set: the workspace must be cleared)
        }
      }
      roles[2 * q] = r;
      roles[2 * q + 1] = H;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
  const int ra = roles[0], Ha = roles[1], rb = roles[2], Hb = roles[3];
  if (ra < 0 && rb < 0) return;   // (the same for every consumer thread)
  float *scratch = red_acc;       // free: the segment combines are done
  auto rows_of = [&](int q) {
    return static_cast<T *>(p.out) +
           (static_cast<size_t>(q ? pend_b[1] : pend_b[0]) * p.Hq + (q ? pend_g[1] : pend_g[0]) * p.G) *
               D;
  };
  const int NC = p.G * (D / 4);
  if (Ha == 1 && Hb == 1) {
    // the last part of each unit merges all of it: the columns of both units
    // are spread over the threads in one pass
    const int n0 = ra >= 0 ? NC : 0, n1 = rb >= 0 ? NC : 0;
    for (int item = tid; item < n0 + n1; item += kConsumers) {
      const int q = item >= n0 ? 1 : 0;
      const int col = item - q * n0;
      merge_store<T>(rows_of(q), col, D,
                     merge_partials(p.o_part, p.lse_part, q ? pend_u[1] : pend_u[0],
                                    q ? pend_c[1] : pend_c[0], q ? pend_n[1] : pend_n[0], 0, 1,
                                    col, p.G, D, P, C));
    }
  } else {
    for (int q = 0; q < npend; ++q) {
      const int r = q ? rb : ra, H = q ? Hb : Ha;
      if (r < 0) continue;
      merge_slice<T, kConsumers>(p, q ? pend_u[1] : pend_u[0], q ? pend_c[1] : pend_c[0],
                                 q ? pend_n[1] : pend_n[0], P, C, r, H, D, rows_of(q), scratch,
                                 tid);
      asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");   // scratch reuse
    }
  }
  if (tid == 0) {
    // this part is done with the partials: the last helper of a unit to finish
    // resets its counters for the next call
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int r = q ? rb : ra, H = q ? Hb : Ha;
      if (r < 0) continue;
      const int u_idx = q ? pend_u[1] : pend_u[0];
      if (H == 1 || atom_add_relaxed_gpu(&p.done[u_idx], 1) == H - 1) {
        p.counters[u_idx] = 0;
        if (H > 1) p.done[u_idx] = 0;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// host-side launch table entry for one compiled variant
// ---------------------------------------------------------------------------
struct AttnVariant {
  cudaError_t (*launch)(const CUtensorMap &, const CUtensorMap &, const AttnParams &,
                        cudaStream_t);
  cudaError_t (*launch_step)(const CUtensorMap &, const CUtensorMap &, const AttnParams &,
                             cudaStream_t);
  cudaError_t (*occupancy)(int *blocks_per_sm);
  int smem_bytes;
  int threads;
};

template <typename T, int D, int NW, int NS, int KIND, int G>
struct AttnLauncher {
  using Q = Geo<T, D, NW, NS>;
  template <bool FUSE, bool PLAN>
  static cudaError_t launch_impl(const CUtensorMap &tk, const CUtensorMap &tv,
                                 const AttnParams &p, cudaStream_t s) {
    auto kern = attn_split_kernel<T, D, NW, NS, KIND, G, FUSE, PLAN>;
    static std::atomic<unsigned long long> attrs_set{0};
    cudaError_t e = set_attributes_once(attrs_set, [&] {
      cudaError_t r =
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Q::kSmemBytes);
      if (r != cudaSuccess) return r;
      return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared);
    });
    if (e != cudaSuccess) return e;
    // launched as a programmatic dependent: the prologue (row scan, barrier
    // set-up, block-id prefetch, TMA of pages that do not hold this step's
    // token) overlaps the RoPE/append kernel before it (when there is one)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_parts);
    cfg.blockDim = dim3(Q::kThreads);
    cfg.dynamicSmemBytes = Q::kSmemBytes;
    cfg.stream = s;
    // merge helpers wait for other CTAs of the grid: a cooperative launch
    // guarantees that all of them are resident (the host enables helpers only
    // for grids that fit)
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (p.max_helpers > 1) {
      attr[na].id = cudaLaunchAttributeCooperative;
      attr[na++].val.cooperative = 1;
    }
    if (!FUSE) {
      attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[na++].val.programmaticStreamSerializationAllowed = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  // a launch with an unchecked plan and no bias runs the smaller variant
  static bool lean(const AttnParams &p) { return p.plan && !p.check_plan && !p.bias; }
  static cudaError_t launch(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                            cudaStream_t s) {
    return lean(p) ? launch_impl<false, true>(tk, tv, p, s)
                   : launch_impl<false, false>(tk, tv, p, s);
  }
  static cudaError_t launch_step(const CUtensorMap &tk, const CUtensorMap &tv,
                                 const AttnParams &p, cudaStream_t s) {
    return lean(p) ? launch_impl<true, true>(tk, tv, p, s)
                   : launch_impl<true, false>(tk, tv, p, s);
  }
  static cudaError_t occupancy(int *n) {
    auto kern = attn_split_kernel<T, D, NW, NS, KIND, G, false, false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Q::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kern, Q::kThreads, Q::kSmemBytes);
  }
  static AttnVariant variant() {
    return AttnVariant{&launch, &launch_step, &occupancy, Q::kSmemBytes, Q::kThreads};
  }
};

// Variant lookup, one per translation unit (returns false if not built).
bool attn_variant_mma(int D, AttnVariant *v);
bool attn_variant_simt_bf16(int D, int G, AttnVariant *v);
bool attn_variant_simt_f32(int D, int G, AttnVariant *v);

}  // namespace pkv
