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
//    mix.  A unit split across CTAs leaves one (o, lse) partial per CTA, merged
//    in the epilogue by the last CTA to finish it (or by the LSE merge kernel);
//    a unit inside one CTA is written to the output directly.
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
  int32_t *counters;        // [U + C] finished-part counters per merge group (kept at 0)
  int32_t *unit_counters;   // [U] finished-group counters per unit (kept at 0)
  float *o_group;           // [(U + C), G, D] merged groups of a unit's partials
  float *lse_group;         // [(U + C), G]
  void *out;                // [B, Hq, D]
  int32_t *err;
  int bt_stride, bias_stride;
  int B, Hq, Hkv, G;
  int num_blocks, num_parts;
  int fuse_merge;           // 1: the last part of a unit merges it (a4 in the epilogue)
  int seg_cost;             // pages of work a unit boundary is worth to the partition
  float scale_log2;         // softmax scale * log2(e)
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

// The fused merge combines a unit's partials in groups of kMergeGroup parts
// (the last part of a group to finish merges the group), then the last group
// merger combines the group results: no CTA ever merges more than
// max(kMergeGroup, groups) partials, whatever the split count.
constexpr int kMergeGroup = 16;

// A part owns no page when C > P and its page range is empty.
__device__ __forceinline__ bool part_empty(long long c, long long P, int C) {
  return div_floor(P * c, C) == div_floor(P * (c + 1), C);
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

// Merge groups of a unit spanning parts c0 .. c0+nseg-1 that own a page.
static __device__ __noinline__ int count_real_groups(int c0, int nseg, long long P, int C) {
  const int ng = (nseg + kMergeGroup - 1) / kMergeGroup;
  int r = 0;
  for (int k = 0; k < ng; ++k)
    r += count_real_parts(c0 + k * kMergeGroup, min(kMergeGroup, nseg - k * kMergeGroup), P, C) > 0;
  return r;
}
__device__ __forceinline__ int real_groups(int c0, int nseg, long long P, int C) {
  return C <= P ? (nseg + kMergeGroup - 1) / kMergeGroup : count_real_groups(c0, nseg, P, C);
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

// One merge of the fused a4: the partials i < n stored at slots
// slot0 + i*stride of (o, lse).  Level 1 merges up to kMergeGroup partials of
// consecutive parts c0 + i; level 2 merges the group results of a unit whose
// parts c0 .. c0+nseg-1 formed several groups.  The result goes to the group
// buffers at grp_slot (a level-1 merge of a multi-group unit) or to the unit's
// output rows.
struct MergeJob {
  const float *o, *lse;
  size_t slot0;
  int n, stride;
  int c0, nseg, level;
  float *o_grp, *lse_grp;   // non-null: write the merged group here
  size_t grp_slot;
  void *out;                // else: the unit's [G, D] output rows
};

// Partial i of job J does not exist: its part (level 1), or every part of its
// group (level 2), owns no page (only possible when C > P).
static __device__ __noinline__ bool merge_skip_slow(const MergeJob &J, int i, long long P, int C) {
  if (J.level == 1) return part_empty(J.c0 + i, P, C);
  return count_real_parts(J.c0 + i * kMergeGroup, min(kMergeGroup, J.nseg - i * kMergeGroup), P,
                          C) == 0;
}
__device__ __forceinline__ bool merge_skip(const MergeJob &J, int i, long long P, int C) {
  return C > P && merge_skip_slow(J, i, P, C);
}

// The merge of one float4 column (head h, dims 4*d4 .. 4*d4+3) of job J by one
// thread.  The lse and o loads of K partials are issued together, so a merge of
// n <= K partials costs one L2 round trip; longer ones rescale a running
// maximum chunk by chunk.  Loads bypass L1: other CTAs wrote the partials.
template <typename T, int K>
__device__ __forceinline__ void merge_job_column(const MergeJob J, int G, int D, int h, int d4,
                                                 long long P, int C) {
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < J.n; s0 += K) {
    float l[K];
    float4 v[K];
#pragma unroll
    for (int u = 0; u < K; ++u) {
      const int s = s0 + u;
      const bool on = s < J.n && !merge_skip(J, s, P, C);
      const size_t slot = J.slot0 + static_cast<size_t>(s) * J.stride;
      l[u] = on ? __ldcg(J.lse + slot * G + h) : -INFINITY;
      v[u] = on ? __ldcg(reinterpret_cast<const float4 *>(J.o + (slot * G + h) * D) + d4)
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m = M;
#pragma unroll
    for (int u = 0; u < K; ++u) m = fmaxf(m, l[u]);
    if (m == -INFINITY) continue;
    const float r = ex2(M - m);   // 0 while nothing was accumulated
    den *= r;
    acc.x *= r;
    acc.y *= r;
    acc.z *= r;
    acc.w *= r;
#pragma unroll
    for (int u = 0; u < K; ++u) {
      const float w = ex2(l[u] - m);
      if (w != 0.f) {
        den += w;
        acc.x = fmaf(w, v[u].x, acc.x);
        acc.y = fmaf(w, v[u].y, acc.y);
        acc.z = fmaf(w, v[u].z, acc.z);
        acc.w = fmaf(w, v[u].w, acc.w);
      }
    }
    M = m;
  }
  float lse = -INFINITY;
  if (den > 0.f) {
    const float inv = __frcp_rn(den);
    acc.x *= inv;
    acc.y *= inv;
    acc.z *= inv;
    acc.w *= inv;
    lse = M + lg2(den);
  }
  if (J.o_grp) {
    *(reinterpret_cast<float4 *>(J.o_grp + (J.grp_slot * G + h) * D) + d4) = acc;
    if (d4 == 0) J.lse_grp[J.grp_slot * G + h] = lse;
  } else {
    store4<T>(static_cast<T *>(J.out) + h * D + 4 * d4, acc);
  }
}

// The jobs' columns spread over the nthr consumer threads: with two jobs of a
// small unit every thread has one column, and all loads are in flight at once.
template <typename T>
__device__ __forceinline__ void merge_jobs(const MergeJob J0, const MergeJob J1, int njobs,
                                           int G, int D, long long P, int C, int tid, int nthr) {
  const int cols = G * (D / 4);
  for (int item = tid; item < njobs * cols; item += nthr) {
    const int q = item >= cols ? 1 : 0;
    const int col = item - q * cols;
    const int h = col / (D / 4), d4 = col - h * (D / 4);
    merge_job_column<T, 8>(q ? J1 : J0, G, D, h, d4, P, C);
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
  static constexpr int kOffMisc = kOffScan + (kThreads / 32) * 4;
  // segment slots: the producer hands each unit segment to the consumers as a
  // 64-byte header (row, KV head, pages, length, page range, first page) and
  // the unit's query rows (up to 8 heads), bulk-copied from global memory
  static constexpr int kSegSlots = 4;
  static constexpr int kSegQBytes = 8 * D * kElem;
  static constexpr int kSegBytes = 64 + kSegQBytes;
  static constexpr int kOffSeg = (kOffMisc + 32 + 127) / 128 * 128;
  static constexpr int kOffSegBars = kOffSeg + kSegSlots * kSegBytes;
  // row lengths of the first kLensCache rows, as the prologue read them
  static constexpr int kLensCache = 256;
  static constexpr int kOffLens = kOffSegBars + 2 * kSegSlots * 8;
  static constexpr int kSmemBytes = kOffLens + kLensCache * 4 + 1024;   // + alignment slack
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
                                         uint32_t vtile, int valid, int b, int t0, int lane) {
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
  if (p.bias) {
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
// Rotated queries of unit (b, g) built by the consumer threads into shared
// memory qs [G][D] (storage type T, rounded once as pkv_rope does); the part
// that owns the unit's first page also reports them in q_rot_out.  Every load
// (position, both halves of each pair) is issued before any is used, and each
// thread forms the angles of its own pairs, so this costs one memory round
// trip and one barrier.
template <typename T, int D, int NTHR>
__device__ __forceinline__ void fused_rotate_q(const AttnParams &p, int b, int g, bool report,
                                               T *qs, int tid) {
  constexpr int half = D / 2;
  constexpr int KM = (8 * half + NTHR - 1) / NTHR;   // pairs per thread (G <= 8)
  const int npairs = p.G * half;
  const T *q = static_cast<const T *>(p.q_new) + (static_cast<size_t>(b) * p.Hq + g * p.G) * D;
  const uint32_t pos = static_cast<uint32_t>(p.positions[b]);
  float x1[KM], x2[KM];
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    const int e = tid + k * NTHR;
    const int h = e / half, i = e - h * half;
    x1[k] = e < npairs ? to_f32(q[h * D + i]) : 0.f;
    x2[k] = e < npairs ? to_f32(q[h * D + half + i]) : 0.f;
  }
  T *qo = static_cast<T *>(p.q_rot_out) + (static_cast<size_t>(b) * p.Hq + g * p.G) * D;
#pragma unroll
  for (int k = 0; k < KM; ++k) {
    const int e = tid + k * NTHR;
    if (e < npairs) {
      const int h = e / half, i = e - h * half;
      float c, s, y1, y2;
      rope_cossin(pos, p.turns[i], &c, &s);
      rope_rotate(x1[k], x2[k], c, s, &y1, &y2);
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
  float x1[KP], x2[KP], v[KV];
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
      x1[k] = i < half ? to_f32(kn[i]) : 0.f;
      x2[k] = i < half ? to_f32(kn[half + i]) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < KV; ++k) {
      const int i = lane + 32 * k;
      v[k] = i < D ? to_f32(vn[i]) : 0.f;
    }
  }

  __device__ __forceinline__ void put(const AttnParams &p, int b, int g, int lane) {
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
          rope_cossin(pos, p.turns[i], &c, &s);
          rope_rotate(x1[k], x2[k], c, s, &y1, &y2);
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
        if (i < D) vc[i] = from_f32<T>(v[k]);
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
                                          int t0, int lane, float *pbuf, float *abuf) {
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
  const float *bias = p.bias ? p.bias + static_cast<size_t>(b) * p.bias_stride + t0 : nullptr;
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
template <typename T, int D, int NW, int NS, int KIND, int G, bool FUSE>
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
  volatile int *misc = reinterpret_cast<volatile int *>(smem + Q::kOffMisc);  // b0, rowoff0, abort

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int C = p.num_parts;
  const bool has_bias = p.bias != nullptr;
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
    misc[2] = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == NW && lane == 0) {
    prefetch_tmap(&tmap_k);
    prefetch_tmap(&tmap_v);
  }

  // ---- page counts of all rows: per-thread chunk sums, block-wide scan ----
  const int nthreads = Q::kThreads;
  const int chunk = (p.B + nthreads - 1) / nthreads;
  const int r0 = min(p.B, tid * chunk), r1 = min(p.B, r0 + chunk);
  // The partition balances pages plus seg_cost per unit: a unit of n pages
  // spans n + seg_cost positions, the first seg_cost of them holding no page
  // (a part that starts a unit pays for the boundary with fewer pages).
  const int A = p.seg_cost;
  auto upos = [A](int n) { return n > 0 ? n + A : 0; };
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
  const long long P = static_cast<long long>(total) * p.Hkv;
  const long long start = div_floor(P * blockIdx.x, C);
  const long long end = div_floor(P * (blockIdx.x + 1), C);
  if (start < end && mysum > 0 && start >= excl * p.Hkv && start < (excl + mysum) * p.Hkv) {
    long long acc = excl;
    for (int b = r0; b < r1; ++b) {
      bool bad;
      const int len = b < Q::kLensCache ? lens_s[b] : p.seq_lens[b];   // own rows: written above
      const int n = upos(pages_of_len(len, p.bt_stride, has_bias, p.bias_stride, &bad));
      if (start < (acc + n) * p.Hkv) {
        misc[0] = b;
        misc[1] = static_cast<int>(acc);
        break;
      }
      acc += n;
    }
  }
  // rows with no token (or an invalid length) output zeros; part c clears rows
  // c, c + C, ...
  for (int b = blockIdx.x; b < p.B; b += C) {   // (after the barrier above: lens_s is complete)
    bool bad;
    const int len = b < Q::kLensCache ? lens_s[b] : p.seq_lens[b];
    if (pages_of_len(len, p.bt_stride, has_bias, p.bias_stride, &bad) == 0) {
      T *o = static_cast<T *>(p.out) + static_cast<size_t>(b) * p.Hq * D;
      for (int e = tid; e < p.Hq * D; e += nthreads) o[e] = from_f32<T>(0.f);
    }
  }
  if (blockIdx.x == 0 && tid == 0) {
    // total position count, for the merge to tell empty parts (C > P) from real ones
    p.meta[2 * p.B * p.Hkv] = static_cast<int32_t>(P & 0xffffffffll);
    p.meta[2 * p.B * p.Hkv + 1] = static_cast<int32_t>(P >> 32);
  }
  __syncthreads();
  if (start >= end) return;
  if (misc[0] < 0) {   // the row scan found no owner of `start` (never expected)
    if (tid == 0) set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
    return;
  }

  if (warp == NW) {
    // ======================= producer warp =======================
    // Walks the part's unit segments.  For each it hands the consumers a
    // segment slot (header + the unit's query rows, bulk-copied) and streams
    // the pages into the ring.  Row lengths of the part's first 64 rows and the
    // next segment's first block ids are read ahead, so a unit boundary costs
    // no dependent global read.
    constexpr int kBatch = NS >= 8 ? 4 : (NS >= 2 ? NS / 2 : 1);
    const uint64_t l2_stream = l2_policy_evict_first();
    const int b0 = misc[0];
    // row lengths: the prologue's copy for the first rows, read ahead beyond
    const int rl0 = b0 + lane < p.B && b0 + lane >= Q::kLensCache ? p.seq_lens[b0 + lane] : 0;
    const int rl1 =
        b0 + 32 + lane < p.B && b0 + 32 + lane >= Q::kLensCache ? p.seq_lens[b0 + 32 + lane] : 0;
    auto row_len = [&](int b) {   // b is warp-uniform
      if (b < Q::kLensCache) return lens_s[b];
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
      const long long rowoff = misc[1];
      bool bad;
      u.b = b0;
      u.n = pages_of_len(row_len(b0), p.bt_stride, has_bias, p.bias_stride, &bad);
      u.g = static_cast<int>(div_floor(start - rowoff * p.Hkv, u.n + A));
      u.off = rowoff * p.Hkv + static_cast<long long>(u.g) * (u.n + A);   // first position
    }
    const uint32_t qbytes = static_cast<uint32_t>(p.G * D * sizeof(T));
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
    int ids = (j0 + lane < j1) ? p.block_tables[static_cast<size_t>(u.b) * p.bt_stride + j0 + lane]
                               : -1;
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
        if (lane == 0) {
          const int slot = k % Q::kSegSlots;
          const uint32_t sph = static_cast<uint32_t>(k / Q::kSegSlots) & 1u;
          bool dead = misc[2] != 0;
          if (!dead && !mbar_wait_bounded(&segempty[slot], sph ^ 1u, kWaitLimitCycles)) {
            misc[2] = 1;
            dead = true;
            set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
          }
          unsigned char *sp = smem + Q::kOffSeg + slot * Q::kSegBytes;
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
          if (!FUSE && !dead) {
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
        }
        __syncwarp();
      };
      for (int jb = j0; jb < j1 && !aborted; jb += 32) {
        const int cur_ids = ids;
        ids = (jb + 32 + lane < j1) ? bt[jb + 32 + lane] : -1;
        const int cnt = min(32, j1 - jb);
        // pages go out kBatch at a time, lane l < kBatch taking page i + l, so
        // the barrier waits, arrivals and TMA issues of a batch share warp
        // instructions (one page per lane-instruction costs ~600 cycles)
        for (int i = 0; i < cnt; i += kBatch) {
          if constexpr (FUSE) {
            // this part owns the unit's last page: append the step's token
            // before the batch that loads that page
            if (j1 == u.n && jb + i <= u.n - 1 && u.n - 1 < jb + i + kBatch)
              app.put(p, u.b, u.g, lane);
          }
          const int blk = __shfl_sync(0xffffffffu, cur_ids, (i + lane) & 31);
          if (lane < kBatch && i + lane < cnt) {
            const int xx = x + (jb - j0) + i + lane;
            const int st = xx % NS;
            const uint32_t ph = static_cast<uint32_t>(xx / NS) & 1u;
            bool dead = misc[2] != 0;
            if (!dead && !mbar_wait_bounded(&empty[st], ph ^ 1u, kWaitLimitCycles)) {
              misc[2] = 1;
              dead = true;
              set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
            }
            const bool ok = !dead && blk >= 0 && blk < p.num_blocks;
            stage_bad[st] = ok ? 0 : 1;
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
            } else {
              if (!dead) set_dev_err(p.err, PKV_DEVERR_BAD_BLOCK);
              mbar_arrive(&full[st]);
            }
          }
          __syncwarp();
          if (!sent) {
            send_segment();
            sent = true;
          }
        }
        aborted = __shfl_sync(0xffffffffu, misc[2], 0) != 0;
      }
      if (!sent) send_segment();   // (a part with no page, or aborted before a batch)
      x += j1 - j0;
      ++k;
      if (!more) break;
      u = nx;
      j0 = 0;
      j1 = nj1;
      ids = nids;
    }
    if (aborted && lane == 0) {
      // never expected: let any copy still in flight land before the CTA exits
      for (int xx = max(0, x - NS); xx < x; ++xx)
        mbar_wait_bounded(&full[xx % NS], static_cast<uint32_t>(xx / NS) & 1u, kWaitLimitCycles);
      if (k > 0) {
        const int s = (k - 1) % Q::kSegSlots;
        mbar_wait_bounded(&segfull[s], static_cast<uint32_t>((k - 1) / Q::kSegSlots) & 1u,
                          kWaitLimitCycles);
      }
    }
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
    if (ok && !mbar_wait_bounded(&segfull[slot], sph, kWaitLimitCycles)) {
      misc[2] = 1;
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
        T *qs = reinterpret_cast<T *>(red_acc);
        fused_rotate_q<T, D, kConsumers>(p, u.b, u.g, j0 == 0, qs, tid);
        mma_begin_smem<D>(s, reinterpret_cast<const __nv_bfloat16 *>(qs), p.G, lane);
        // qs sits in the reduction buffer: nobody stashes before all have read
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
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
        if (ready && !mbar_wait_bounded(&full[st], ph, kWaitLimitCycles)) {
          misc[2] = 1;
          set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
          ready = false;
        }
        if (ready && !stage_bad[st]) {
          const uint32_t kt = smem_u32(smem + st * Q::kStageBytes);
          mma_page<D>(s, p, kt, kt + Q::kTileBytes, min(kBlockTokens, L - j * kBlockTokens), u.b,
                      j * kBlockTokens, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      mma_stash<D>(s, my_acc, my_m, my_l, lane);
    } else {
      SimtState<T, D, G> s;
      if constexpr (FUSE) {
        T *qs = reinterpret_cast<T *>(red_acc);
        fused_rotate_q<T, D, kConsumers>(p, u.b, u.g, j0 == 0, qs, tid);
        simt_begin_smem<T, D, G>(s, qs, p.G, p.scale_log2, lane);
        asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
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
        if (ready && !mbar_wait_bounded(&full[st], ph, kWaitLimitCycles)) {
          misc[2] = 1;
          set_dev_err(p.err, PKV_DEVERR_TIMEOUT);
          ready = false;
        }
        if (ready && !stage_bad[st]) {
          const char *kt = reinterpret_cast<const char *>(smem + st * Q::kStageBytes);
          simt_page<T, D, G>(s, p, kt, kt + Q::kTileBytes, min(kBlockTokens, L - j * kBlockTokens),
                             u.b, j * kBlockTokens, lane, pbuf, abuf);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
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
  // ---- a4 in the epilogue: the last part to finish a merge group merges it,
  // the last group merger of a unit merges the groups (threadfence-reduction
  // pattern; every counter is reset by the CTA that consumes it).  Both
  // pending units go through each phase together, so the counters cost one
  // round trip and the merges one or two more. ----
  // (the segment loop ended with a consumer barrier: all partials are written)
  MergeJob job[2];
  int first_g[2], ngroups[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int u_idx = q < npend ? pend_u[q] : pend_u[0];
    const int c_first = q < npend ? pend_c[q] : pend_c[0];
    const int nseg = q < npend ? pend_n[q] : pend_n[0];
    const int grp = (static_cast<int>(blockIdx.x) - c_first) / kMergeGroup;
    first_g[q] = c_first + grp * kMergeGroup;
    ngroups[q] = (nseg + kMergeGroup - 1) / kMergeGroup;
    MergeJob &J = job[q];
    J.o = p.o_part;
    J.lse = p.lse_part;
    J.slot0 = static_cast<size_t>(u_idx) + first_g[q];
    J.n = min(kMergeGroup, nseg - grp * kMergeGroup);
    J.stride = 1;
    J.c0 = first_g[q];
    J.nseg = nseg;
    J.level = 1;
    J.o_grp = ngroups[q] > 1 ? p.o_group : nullptr;
    J.lse_grp = p.lse_group;
    J.grp_slot = J.slot0;
    const int bq = q < npend ? pend_b[q] : pend_b[0], gq2 = q < npend ? pend_g[q] : pend_g[0];
    J.out = static_cast<T *>(p.out) + (static_cast<size_t>(bq) * p.Hq + gq2 * p.G) * D;
  }
  if (tid == 0) {
    fence_acq_rel_gpu();   // release this part's partials
    int prev[2];
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (q < npend) prev[q] = atom_add_relaxed_gpu(&p.counters[pend_u[q] + first_g[q]], 1);
    fence_acq_rel_gpu();   // acquire the other parts' partials
    int last = 0;
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (q < npend && prev[q] == real_parts(first_g[q], job[q].n, P, C) - 1) {
        last |= 1 << q;
        p.counters[pend_u[q] + first_g[q]] = 0;
      }
    misc[4] = last;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
  const int last1 = misc[4];
  if (last1 == 0) return;
  merge_jobs<T>((last1 & 1) ? job[0] : job[1], job[1], last1 == 3 ? 2 : 1, p.G, D, P, C, tid, kConsumers);
  // level 2 for the units that have several groups
  int multi = 0;
#pragma unroll
  for (int q = 0; q < 2; ++q)
    if ((last1 >> q & 1) && ngroups[q] > 1) multi |= 1 << q;
  if (multi == 0) return;
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");   // group results written
  if (tid == 0) {
    fence_acq_rel_gpu();
    int prev[2];
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (multi >> q & 1) prev[q] = atom_add_relaxed_gpu(&p.unit_counters[pend_u[q]], 1);
    fence_acq_rel_gpu();
    int last = 0;
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if ((multi >> q & 1) && prev[q] == real_groups(pend_c[q], pend_n[q], P, C) - 1) {
        last |= 1 << q;
        p.unit_counters[pend_u[q]] = 0;
      }
    misc[5] = last;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory");
  const int last2 = misc[5];
  if (last2 == 0) return;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    MergeJob &J = job[q];
    J.o = p.o_group;
    J.lse = p.lse_group;
    J.slot0 = static_cast<size_t>(q < npend ? pend_u[q] : pend_u[0]) +
              (q < npend ? pend_c[q] : pend_c[0]);
    J.n = ngroups[q];
    J.stride = kMergeGroup;
    J.c0 = q < npend ? pend_c[q] : pend_c[0];
    J.level = 2;
    J.o_grp = nullptr;
  }
  merge_jobs<T>((last2 & 1) ? job[0] : job[1], job[1], last2 == 3 ? 2 : 1, p.G, D, P, C, tid,
                kConsumers);
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
  template <bool FUSE>
  static cudaError_t launch_impl(const CUtensorMap &tk, const CUtensorMap &tv,
                                 const AttnParams &p, cudaStream_t s) {
    auto kern = attn_split_kernel<T, D, NW, NS, KIND, G, FUSE>;
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = FUSE ? 0 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  static cudaError_t launch(const CUtensorMap &tk, const CUtensorMap &tv, const AttnParams &p,
                            cudaStream_t s) {
    return launch_impl<false>(tk, tv, p, s);
  }
  static cudaError_t launch_step(const CUtensorMap &tk, const CUtensorMap &tv,
                                 const AttnParams &p, cudaStream_t s) {
    return launch_impl<true>(tk, tv, p, s);
  }
  static cudaError_t occupancy(int *n) {
    auto kern = attn_split_kernel<T, D, NW, NS, KIND, G, false>;
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
