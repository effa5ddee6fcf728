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
  // the decode-step kernel with no query heads and no rotated-key report: every
  // token's key is rotated and stored exactly as a decode append would store it
  return rope_launch(nullptr, k, v, nullptr, nullptr, positions, slot_mapping, k_cache, v_cache, T,
                     0, Hkv, d, num_blocks, base, dtype, dev_err_flag, stream, true, true);
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
