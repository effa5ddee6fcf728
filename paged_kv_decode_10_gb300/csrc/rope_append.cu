// a1 RoPE and a2 append of the decode step (separately and fused).
//
// RoPE: helexa issue 121, slice 1 -- cos/sin gathered at arbitrary per-row
// positions ((B,1,half)) and applied with the rotate-half convention; keys are
// stored post-RoPE.  Append: "neurogrid releases" v0.7.0 -- the KV cache is a
// pool of fixed 16-token blocks; the new token's K/V go to slot_mapping[b].
//
// Angles.  theta_i = p * base^(-2i/d) can reach 1.3e5 rad at p = 131072, where
// a float32 product would be off by ~0.008 rad; the angle is formed in 64-bit
// fixed-point turns instead (rope_cossin in common.cuh), exact to float32
// rounding, and sincosf then only sees reduced arguments.
#include <cmath>
#include <cstdint>

#include "common.cuh"

namespace pkv {
namespace {

constexpr int kMaxHalf = 128;

struct RopeTurns {
  unsigned long long f[kMaxHalf];   // 2^64 * base^(-2i/d) / (2 pi)
};

template <typename T, int VEC>
struct Vec;
template <> struct Vec<float, 4> { using type = float4; };
template <> struct Vec<__nv_bfloat16, 4> { using type = uint2; };
template <> struct Vec<float, 1> { using type = float; };
template <> struct Vec<__nv_bfloat16, 1> { using type = __nv_bfloat16; };

template <typename T, int VEC>
__device__ __forceinline__ void unpack(const typename Vec<T, VEC>::type &w, float (&x)[VEC]) {
  if constexpr (VEC == 1) {
    x[0] = to_f32(w);
  } else if constexpr (sizeof(T) == 4) {
    x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
  } else {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
  }
}

template <typename T, int VEC>
__device__ __forceinline__ typename Vec<T, VEC>::type pack(const float (&x)[VEC]) {
  typename Vec<T, VEC>::type w;
  if constexpr (VEC == 1) {
    w = from_f32<T>(x[0]);
  } else if constexpr (sizeof(T) == 4) {
    w = make_float4(x[0], x[1], x[2], x[3]);
  } else {
    w.x = pack_bf16(x[0], x[1]);
    w.y = pack_bf16(x[2], x[3]);
  }
  return w;
}

// One CTA per batch row, one work item per thread so every load of the row is
// issued in one round.  Items: VEC consecutive rotation pairs of one head of q
// or k ((Hq + Hkv) * half / VEC of them) and, with APPEND, 16-byte chunks of
// the row's values (copied into the cache slot).  cos/sin of the row's
// position are built first in shared memory.  DEP: launched as a programmatic
// dependent of the previous layer's attention kernel; the new q/k/v are that
// layer's product, so they are read only after griddepcontrol.wait (the
// angles are formed before it).
template <typename T, int VEC, bool APPEND, bool DEP>
__global__ void rope_kernel(const T *__restrict__ q, const T *__restrict__ k,
                            const T *__restrict__ v, T *__restrict__ q_out,
                            T *__restrict__ k_out, const int32_t *__restrict__ positions,
                            const int64_t *__restrict__ slots, T *__restrict__ k_cache,
                            T *__restrict__ v_cache, int Hq, int Hkv, int d, int64_t num_slots,
                            int32_t *err, const RopeTurns turns) {
  using W = typename Vec<T, VEC>::type;
  extern __shared__ float cs[];  // cos[half], sin[half]
  // the attention kernel that follows may start its own prologue now; it waits
  // for this grid before reading q_rot or the appended slot
  pdl_launch_dependents();
  const int b = blockIdx.x;
  const int half = d >> 1;
  const int tid = threadIdx.x;
  const int rot_items = (Hq + Hkv) * (half / VEC);
  const int v_chunks = APPEND ? Hkv * d * static_cast<int>(sizeof(T)) / 16 : 0;

  // issue this thread's loads before anything waits
  const uint32_t pos = static_cast<uint32_t>(positions[b]);
  int64_t slot = -1;
  if (APPEND) slot = slots[b];
  W x1w{}, x2w{};
  int h = 0, c = 0;
  const bool rot = tid < rot_items;
  if (rot) {
    h = tid / (half / VEC);
    c = (tid - h * (half / VEC)) * VEC;
  }
  uint4 vw{};
  const bool vcopy = APPEND && tid < v_chunks;
  auto load_inputs = [&]() {
    if (rot) {
      const T *src = h < Hq ? q + (static_cast<size_t>(b) * Hq + h) * d
                            : k + (static_cast<size_t>(b) * Hkv + (h - Hq)) * d;
      x1w = *reinterpret_cast<const W *>(src + c);
      x2w = *reinterpret_cast<const W *>(src + half + c);
    }
    if (vcopy) vw = reinterpret_cast<const uint4 *>(v + static_cast<size_t>(b) * Hkv * d)[tid];
  };
  if constexpr (!DEP) load_inputs();

  for (int i = tid; i < half; i += blockDim.x) {
    float s, co;
    rope_cossin(pos, turns.f[i], &co, &s);
    cs[i] = co;
    cs[half + i] = s;
  }
  if constexpr (DEP) {
    pdl_wait();
    load_inputs();
  }
  if (APPEND && slot >= num_slots) {
    if (tid == 0) set_dev_err(err, PKV_DEVERR_BAD_SLOT);
    slot = -1;
  }
  __syncthreads();

  const int64_t blk = slot / kBlockTokens;
  const size_t row0 =
      APPEND && slot >= 0
          ? static_cast<size_t>((blk * Hkv) * kBlockTokens + (slot - blk * kBlockTokens)) * d
          : 0;
  if (rot) {
    float x1[VEC], x2[VEC], y1[VEC], y2[VEC];
    unpack<T, VEC>(x1w, x1);
    unpack<T, VEC>(x2w, x2);
#pragma unroll
    for (int e = 0; e < VEC; ++e) rope_rotate(x1[e], x2[e], cs[c + e], cs[half + c + e], &y1[e], &y2[e]);
    const W o1 = pack<T, VEC>(y1), o2 = pack<T, VEC>(y2);
    T *dst = h < Hq ? q_out + (static_cast<size_t>(b) * Hq + h) * d
                    : (k_out ? k_out + (static_cast<size_t>(b) * Hkv + (h - Hq)) * d : nullptr);
    if (dst) {   // a prefill does not report the rotated keys
      *reinterpret_cast<W *>(dst + c) = o1;
      *reinterpret_cast<W *>(dst + half + c) = o2;
    }
    if (APPEND && slot >= 0 && h >= Hq) {
      T *cdst = k_cache + row0 + static_cast<size_t>(h - Hq) * kBlockTokens * d;
      *reinterpret_cast<W *>(cdst + c) = o1;
      *reinterpret_cast<W *>(cdst + half + c) = o2;
    }
  }
  if (vcopy && slot >= 0) {
    const int per_head = d * static_cast<int>(sizeof(T)) / 16;
    const int hk = tid / per_head, ch = tid - hk * per_head;
    reinterpret_cast<uint4 *>(v_cache + row0 + static_cast<size_t>(hk) * kBlockTokens * d)[ch] = vw;
  }
}

// Grid-stride copy of 16-byte chunks: for each (row, KV head, chunk) move the
// rotated key and the value into the cache slot of the row.
__global__ void append_kernel(const uint4 *__restrict__ k_rot, const uint4 *__restrict__ v,
                              const int64_t *__restrict__ slots, uint4 *__restrict__ k_cache,
                              uint4 *__restrict__ v_cache, int B, int Hkv, int chunks_per_row,
                              int64_t num_slots, int32_t *err) {
  const int64_t total = static_cast<int64_t>(B) * Hkv * chunks_per_row;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(e % chunks_per_row);
    const int64_t bh = e / chunks_per_row;
    const int h = static_cast<int>(bh % Hkv);
    const int b = static_cast<int>(bh / Hkv);
    const int64_t slot = slots[b];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (c == 0 && h == 0) set_dev_err(err, PKV_DEVERR_BAD_SLOT);
      continue;
    }
    const int64_t blk = slot / kBlockTokens;
    const int64_t off = slot - blk * kBlockTokens;
    const size_t dst =
        ((static_cast<size_t>(blk) * Hkv + h) * kBlockTokens + off) * chunks_per_row + c;
    const size_t src = (static_cast<size_t>(b) * Hkv + h) * chunks_per_row + c;
    k_cache[dst] = k_rot[src];
    v_cache[dst] = v[src];
  }
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// pkv_prefill_kv: the prefix keys and values of joining sequences, many tokens
// per CTA.  A token is served by TPT = (D/2) / E threads (E = elements per
// 16-byte vector): thread l owns rotation pairs [l*E, l*E+E) of every KV head,
// forms their E angles once (rope_cossin of the token's position, the same
// table and arithmetic as the decode append, so a prefix key is bit-identical
// to the key a decode step stores for it) and moves 16-byte vectors; it also
// copies every TPT-th 16-byte chunk of the token's values.  Loads of four heads
// (or eight value chunks) are issued together.
template <typename T, int D>
__global__ void __launch_bounds__(256) prefill_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const int32_t *__restrict__ positions,
    const int64_t *__restrict__ slots, uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
    int n_tokens, int Hkv, int64_t num_slots, int32_t *err, const RopeTurns turns) {
  constexpr int E = 16 / static_cast<int>(sizeof(T));
  constexpr int HALF = D / 2;
  constexpr int TPT = HALF / E;        // threads per token
  constexpr int VPR = D / E;           // 16-byte vectors per head row
  constexpr int TOK = 256 / TPT;       // tokens per CTA
  const int l = threadIdx.x % TPT;
  const int t = blockIdx.x * TOK + threadIdx.x / TPT;
  if (t >= n_tokens) return;
  const int64_t slot = slots[t];
  const uint32_t pos = static_cast<uint32_t>(positions[t]);
  const uint4 *kt = k + static_cast<size_t>(t) * Hkv * VPR;
  const uint4 *vt = v + static_cast<size_t>(t) * Hkv * VPR;
  // the first heads' keys are in flight while the angles are formed
  uint4 x[8];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < Hkv) {
      x[2 * j] = kt[j * VPR + l];
      x[2 * j + 1] = kt[j * VPR + TPT + l];
    }
  float co[E], sn[E];
#pragma unroll
  for (int e = 0; e < E; ++e) rope_cossin(pos, turns.f[l * E + e], &co[e], &sn[e]);
  bool write = slot >= 0;
  if (slot >= num_slots) {
    if (l == 0) set_dev_err(err, PKV_DEVERR_BAD_SLOT);
    write = false;
  }
  const int64_t blk = slot / kBlockTokens;
  // vector index of (block, head 0, row) in the cache viewed as 16-byte vectors
  const size_t row0 = write ? static_cast<size_t>((blk * Hkv) * kBlockTokens +
                                                  (slot - blk * kBlockTokens)) * VPR
                            : 0;
  for (int h0 = 0; h0 < Hkv; h0 += 4) {
    if (h0 > 0) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (h0 + j < Hkv) {
          x[2 * j] = kt[(h0 + j) * VPR + l];
          x[2 * j + 1] = kt[(h0 + j) * VPR + TPT + l];
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (h0 + j >= Hkv) break;
      const T *a = reinterpret_cast<const T *>(&x[2 * j]);
      const T *b = reinterpret_cast<const T *>(&x[2 * j + 1]);
      uint4 ya, yb;
      T *pa = reinterpret_cast<T *>(&ya);
      T *pb = reinterpret_cast<T *>(&yb);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        float y1, y2;
        rope_rotate(to_f32(a[e]), to_f32(b[e]), co[e], sn[e], &y1, &y2);
        pa[e] = from_f32<T>(y1);
        pb[e] = from_f32<T>(y2);
      }
      if (write) {
        uint4 *dst = k_cache + row0 + static_cast<size_t>(h0 + j) * kBlockTokens * VPR;
        dst[l] = ya;
        dst[TPT + l] = yb;
      }
    }
  }
  // values: vector c of the token's [Hkv, D] row for c = l, l + TPT, ...
  const int nv = Hkv * VPR;
  for (int c0 = l; c0 < nv; c0 += 8 * TPT) {
    uint4 w[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (c0 + j * TPT < nv) w[j] = vt[c0 + j * TPT];
    if (write) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = c0 + j * TPT;
        if (c < nv) {
          const int h = c / VPR, r = c - h * VPR;
          v_cache[row0 + static_cast<size_t>(h) * kBlockTokens * VPR + r] = w[j];
        }
      }
    }
  }
}

template <typename T, int D>
int launch_prefill(const void *k, const void *v, const int32_t *positions, const int64_t *slots,
                   void *k_cache, void *v_cache, int n_tokens, int Hkv, int64_t num_slots,
                   int32_t *err, const RopeTurns &turns, cudaStream_t s) {
  constexpr int TPT = (D / 2) / (16 / static_cast<int>(sizeof(T)));
  constexpr int TOK = 256 / TPT;
  const int grid = (n_tokens + TOK - 1) / TOK;
  prefill_kernel<T, D><<<grid, 256, 0, s>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), positions, slots,
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), n_tokens, Hkv, num_slots,
      err, turns);
  PKV_LAUNCH_CHECK("prefill_kernel");
  return PKV_OK;
}

template <typename T, int VEC, bool APPEND>
void launch_rope(int B, int threads, size_t smem, cudaStream_t s, const void *q, const void *k,
                 const void *v, void *q_out, void *k_out, const int32_t *positions,
                 const int64_t *slots, void *k_cache, void *v_cache, int Hq, int Hkv, int d,
                 int64_t num_slots, int32_t *err, const RopeTurns &turns, bool dependent) {
  if (!dependent) {
    // same L1/shared split as the attention kernel that follows, so the SMs
    // need no reconfiguration between the two launches of a step
    static std::atomic<unsigned long long> attrs_set{0};
    set_attributes_once(attrs_set, [] {
      return cudaFuncSetAttribute(rope_kernel<T, VEC, APPEND, false>,
                                  cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared);
    });
    rope_kernel<T, VEC, APPEND, false><<<B, threads, smem, s>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v),
        static_cast<T *>(q_out), static_cast<T *>(k_out), positions, slots,
        static_cast<T *>(k_cache), static_cast<T *>(v_cache), Hq, Hkv, d, num_slots, err, turns);
    return;
  }
  auto kern = rope_kernel<T, VEC, APPEND, true>;
  static std::atomic<unsigned long long> attrs_set{0};
  set_attributes_once(attrs_set, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
  });
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kern, static_cast<const T *>(q), static_cast<const T *>(k),
                     static_cast<const T *>(v), static_cast<T *>(q_out), static_cast<T *>(k_out),
                     positions, slots, static_cast<T *>(k_cache), static_cast<T *>(v_cache), Hq,
                     Hkv, d, num_slots, err, turns);
}

int rope_launch(const void *q, const void *k, const void *v, void *q_out, void *k_out,
                const int32_t *positions, const int64_t *slots, void *k_cache, void *v_cache,
                int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_blocks, float base,
                int32_t dtype, int32_t *err, void *stream, bool append, bool k_out_optional = false,
                bool dependent = false) {
  PKV_REQUIRE(B >= 0 && Hq >= 0 && Hkv >= 0, PKV_ERR_INVALID_ARG, "negative size");
  PKV_REQUIRE(d >= 2 && d <= 2 * kMaxHalf && d % 2 == 0, PKV_ERR_UNSUPPORTED, "head_dim %d", d);
  PKV_REQUIRE(dtype_ok(dtype), PKV_ERR_UNSUPPORTED, "dtype %d", dtype);
  PKV_REQUIRE(base > 0.0f, PKV_ERR_INVALID_ARG, "rope base must be positive");
  if (B == 0 || Hq + Hkv == 0) return PKV_OK;
  PKV_REQUIRE(positions, PKV_ERR_INVALID_ARG, "positions is NULL");
  PKV_REQUIRE((Hq == 0 || (q && q_out)) && (Hkv == 0 || (k && (k_out || k_out_optional))),
              PKV_ERR_INVALID_ARG, "NULL tensor");
  const int elem = static_cast<int>(dtype_size(dtype));
  const int vec = (d % 8 == 0) ? 4 : 1;
  if (vec == 4)
    PKV_REQUIRE((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                 reinterpret_cast<uintptr_t>(q_out) | reinterpret_cast<uintptr_t>(k_out)) %
                        (4 * elem) == 0,
                PKV_ERR_INVALID_ARG, "q/k tensors must be aligned to 4 elements");
  if (append) {
    PKV_REQUIRE(v && slots && k_cache && v_cache && num_blocks >= 0, PKV_ERR_INVALID_ARG,
                "NULL append argument");
    PKV_REQUIRE(d * elem % 16 == 0 && aligned16(v) && aligned16(k_cache) && aligned16(v_cache),
                PKV_ERR_INVALID_ARG, "append needs 16-byte rows and 16-byte aligned tensors");
  }
  RopeTurns t;
  fill_rope_turns(base, d, t.f);
  const int rot_items = (Hq + Hkv) * (d / 2 / vec);
  const int v_chunks = append ? Hkv * d * elem / 16 : 0;
  int items = rot_items > v_chunks ? rot_items : v_chunks;
  if (items < d / 2) items = d / 2;
  PKV_REQUIRE(items <= 1024, PKV_ERR_UNSUPPORTED, "too many heads for one CTA per row (%d items)",
              items);
  const int threads = (items + 31) / 32 * 32;
  const size_t smem = sizeof(float) * d;
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * kBlockTokens;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
#define PKV_ROPE_ARGS                                                                     \
  B, threads, smem, s, q, k, v, q_out, k_out, positions, slots, k_cache, v_cache, Hq, Hkv, d, \
      num_slots, err, t, dependent
  if (dtype == PKV_BF16) {
    using T = __nv_bfloat16;
    if (vec == 4)
      append ? launch_rope<T, 4, true>(PKV_ROPE_ARGS) : launch_rope<T, 4, false>(PKV_ROPE_ARGS);
    else
      append ? launch_rope<T, 1, true>(PKV_ROPE_ARGS) : launch_rope<T, 1, false>(PKV_ROPE_ARGS);
  } else {
    using T = float;
    if (vec == 4)
      append ? launch_rope<T, 4, true>(PKV_ROPE_ARGS) : launch_rope<T, 4, false>(PKV_ROPE_ARGS);
    else
      append ? launch_rope<T, 1, true>(PKV_ROPE_ARGS) : launch_rope<T, 1, false>(PKV_ROPE_ARGS);
  }
#undef PKV_ROPE_ARGS
  PKV_LAUNCH_CHECK("rope_kernel");
  return PKV_OK;
}

}  // namespace

int rope_append_dependent(const void *q, const void *k, const void *v, void *q_out, void *k_out,
                          const int32_t *positions, const int64_t *slot_mapping, void *k_cache,
                          void *v_cache, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                          int32_t num_blocks, float base, int32_t dtype, int32_t *dev_err_flag,
                          void *stream) {
  return rope_launch(q, k, v, q_out, k_out, positions, slot_mapping, k_cache, v_cache, B, Hq, Hkv,
                     d, num_blocks, base, dtype, dev_err_flag, stream, true, false, true);
}

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_rope(const void *q, const void *k, void *q_out, void *k_out,
                        const int32_t *positions, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                        float base, int32_t dtype, void *stream) {
  clear_error();
  return rope_launch(q, k, nullptr, q_out, k_out, positions, nullptr, nullptr, nullptr, B, Hq,
                     Hkv, d, 0, base, dtype, nullptr, stream, false);
}

extern "C" int pkv_rope_append(const void *q, const void *k, const void *v, void *q_out,
                               void *k_out, const int32_t *positions,
                               const int64_t *slot_mapping, void *k_cache, void *v_cache,
                               int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_blocks,
                               float base, int32_t dtype, int32_t *dev_err_flag, void *stream) {
  clear_error();
  return rope_launch(q, k, v, q_out, k_out, positions, slot_mapping, k_cache, v_cache, B, Hq, Hkv,
                     d, num_blocks, base, dtype, dev_err_flag, stream, true);
}

extern "C" int pkv_prefill_kv(const void *k, const void *v, const int32_t *positions,
                              const int64_t *slot_mapping, void *k_cache, void *v_cache, int32_t T,
                              int32_t Hkv, int32_t d, int32_t num_blocks, float base,
                              int32_t dtype, int32_t *dev_err_flag, void *stream) {
  clear_error();
  // head sizes of the attention kernels, 16-byte aligned tensors: the prefill
  // kernel; otherwise the decode-step kernel with no query heads and no
  // rotated-key report.  Either way a token's key is rotated and stored exactly
  // as a decode append would store it.
  const bool fast = (d == 64 || d == 128) && dtype_ok(dtype) && T > 0 && Hkv > 0 && k && v &&
                    positions && slot_mapping && k_cache && v_cache && aligned16(k) &&
                    aligned16(v) && aligned16(k_cache) && aligned16(v_cache) && num_blocks >= 0 &&
                    base > 0.0f;
  if (!fast)
    return rope_launch(nullptr, k, v, nullptr, nullptr, positions, slot_mapping, k_cache, v_cache,
                       T, 0, Hkv, d, num_blocks, base, dtype, dev_err_flag, stream, true, true);
  RopeTurns turns;
  fill_rope_turns(base, d, turns.f);
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * kBlockTokens;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == PKV_BF16)
    return d == 64 ? launch_prefill<__nv_bfloat16, 64>(k, v, positions, slot_mapping, k_cache,
                                                        v_cache, T, Hkv, num_slots, dev_err_flag,
                                                        turns, s)
                   : launch_prefill<__nv_bfloat16, 128>(k, v, positions, slot_mapping, k_cache,
                                                         v_cache, T, Hkv, num_slots, dev_err_flag,
                                                         turns, s);
  return d == 64 ? launch_prefill<float, 64>(k, v, positions, slot_mapping, k_cache, v_cache, T,
                                             Hkv, num_slots, dev_err_flag, turns, s)
                 : launch_prefill<float, 128>(k, v, positions, slot_mapping, k_cache, v_cache, T,
                                              Hkv, num_slots, dev_err_flag, turns, s);
}

extern "C" int pkv_append(const void *k_rot, const void *v, const int64_t *slot_mapping,
                          void *k_cache, void *v_cache, int32_t B, int32_t Hkv, int32_t d,
                          int32_t num_blocks, int32_t dtype, int32_t *dev_err_flag,
                          void *stream) {
  clear_error();
  PKV_REQUIRE(B >= 0 && Hkv >= 0 && num_blocks >= 0, PKV_ERR_INVALID_ARG, "negative size");
  PKV_REQUIRE(dtype_ok(dtype), PKV_ERR_UNSUPPORTED, "dtype %d", dtype);
  const size_t row_bytes = static_cast<size_t>(d) * dtype_size(dtype);
  PKV_REQUIRE(d > 0 && row_bytes % 16 == 0, PKV_ERR_UNSUPPORTED,
              "head_dim * sizeof(dtype) must be a multiple of 16 (d=%d)", d);
  if (B == 0 || Hkv == 0) return PKV_OK;
  PKV_REQUIRE(k_rot && v && slot_mapping && k_cache && v_cache, PKV_ERR_INVALID_ARG,
              "NULL pointer");
  PKV_REQUIRE(aligned16(k_rot) && aligned16(v) && aligned16(k_cache) && aligned16(v_cache),
              PKV_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  const int chunks = static_cast<int>(row_bytes / 16);
  const int64_t total = static_cast<int64_t>(B) * Hkv * chunks;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 65535) blocks = 65535;
  append_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(k_rot), static_cast<const uint4 *>(v), slot_mapping,
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), B, Hkv, chunks,
      static_cast<int64_t>(num_blocks) * kBlockTokens, dev_err_flag);
  PKV_LAUNCH_CHECK("append_kernel");
  return PKV_OK;
}
