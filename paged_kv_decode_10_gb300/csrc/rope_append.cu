// a1 RoPE and a2 append of the decode step.
//
// RoPE: helexa issue 121, slice 1 -- cos/sin gathered at arbitrary per-row
// positions ((B,1,half)) and applied with the rotate-half convention; keys are
// stored post-RoPE.  Append: "neurogrid releases" v0.7.0 -- the KV cache is a
// pool of fixed 16-token blocks; the new token's K/V go to slot_mapping[b].
#include <cmath>
#include <cstdint>

#include "common.cuh"

namespace pkv {
namespace {

constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr int kMaxHalf = 128;

// base^(-2i/d) for i < d/2, computed on the host in double precision.
struct RopeFreqs {
  double inv[kMaxHalf];
};

// One CTA per batch row.  Threads first build cos/sin of every pair at the
// row's position (angle p * inv_freq formed and reduced modulo 2*pi in double
// precision, so positions of 10^5 keep float32-accurate angles), then rotate
// every head of q and k.  With APPEND the rotated key and the raw value are
// also written into the row's cache slot (a1 and a2 fused).
template <typename T, bool APPEND>
__global__ void rope_kernel(const T *__restrict__ q, const T *__restrict__ k,
                            const T *__restrict__ v, T *__restrict__ q_out,
                            T *__restrict__ k_out, const int32_t *__restrict__ positions,
                            const int64_t *__restrict__ slots, T *__restrict__ k_cache,
                            T *__restrict__ v_cache, int Hq, int Hkv, int d, int64_t num_slots,
                            int32_t *err, const RopeFreqs freqs) {
  extern __shared__ float cs[];  // cos[half], sin[half]
  const int b = blockIdx.x;
  const int half = d >> 1;
  const double p = static_cast<double>(positions[b]);
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double theta = p * freqs.inv[i];
    const double turns = rint(theta * (1.0 / kTwoPi));
    const double r = fma(-turns, kTwoPi, theta);
    float s, c;
    sincosf(static_cast<float>(r), &s, &c);
    cs[i] = c;
    cs[half + i] = s;
  }
  int64_t slot = -1;
  if (APPEND) {
    slot = slots[b];
    if (slot >= num_slots) {
      if (threadIdx.x == 0) set_dev_err(err, PKV_DEVERR_BAD_SLOT);
      slot = -1;
    }
  }
  // cache row of the slot for KV head 0; head h adds h * 16 * d
  const int64_t blk = slot / kBlockTokens;
  T *kdst0 = APPEND && slot >= 0
                 ? k_cache + ((blk * Hkv) * kBlockTokens + (slot - blk * kBlockTokens)) * d
                 : nullptr;
  T *vdst0 = APPEND && slot >= 0
                 ? v_cache + ((blk * Hkv) * kBlockTokens + (slot - blk * kBlockTokens)) * d
                 : nullptr;
  __syncthreads();
  const int heads = Hq + Hkv;
  for (int e = threadIdx.x; e < heads * half; e += blockDim.x) {
    const int h = e / half;
    const int i = e - h * half;
    const T *src;
    T *dst;
    T *cdst = nullptr;
    if (h < Hq) {
      src = q + (static_cast<size_t>(b) * Hq + h) * d;
      dst = q_out + (static_cast<size_t>(b) * Hq + h) * d;
    } else {
      const int hk = h - Hq;
      src = k + (static_cast<size_t>(b) * Hkv + hk) * d;
      dst = k_out + (static_cast<size_t>(b) * Hkv + hk) * d;
      if (kdst0) cdst = kdst0 + static_cast<size_t>(hk) * kBlockTokens * d;
    }
    const float x1 = to_f32(src[i]);
    const float x2 = to_f32(src[i + half]);
    const float c = cs[i], s = cs[half + i];
    const T y1 = from_f32<T>(x1 * c - x2 * s);
    const T y2 = from_f32<T>(x2 * c + x1 * s);
    dst[i] = y1;
    dst[i + half] = y2;
    if (cdst) {
      cdst[i] = y1;
      cdst[i + half] = y2;
    }
  }
  if (vdst0) {
    for (int e = threadIdx.x; e < Hkv * d; e += blockDim.x) {
      const int hk = e / d, i = e - hk * d;
      vdst0[static_cast<size_t>(hk) * kBlockTokens * d + i] =
          v[(static_cast<size_t>(b) * Hkv + hk) * d + i];
    }
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
    const size_t dst = ((static_cast<size_t>(blk) * Hkv + h) * kBlockTokens + off) * chunks_per_row + c;
    const size_t src = (static_cast<size_t>(b) * Hkv + h) * chunks_per_row + c;
    k_cache[dst] = k_rot[src];
    v_cache[dst] = v[src];
  }
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pkv

using namespace pkv;

namespace {
int rope_launch(const void *q, const void *k, const void *v, void *q_out, void *k_out,
                const int32_t *positions, const int64_t *slots, void *k_cache, void *v_cache,
                int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_blocks, float base,
                int32_t dtype, int32_t *err, void *stream, bool append) {
  PKV_REQUIRE(B >= 0 && Hq >= 0 && Hkv >= 0, PKV_ERR_INVALID_ARG, "negative size");
  PKV_REQUIRE(d >= 2 && d <= 2 * kMaxHalf && d % 2 == 0, PKV_ERR_UNSUPPORTED, "head_dim %d", d);
  PKV_REQUIRE(dtype_ok(dtype), PKV_ERR_UNSUPPORTED, "dtype %d", dtype);
  PKV_REQUIRE(base > 0.0f, PKV_ERR_INVALID_ARG, "rope base must be positive");
  if (B == 0 || Hq + Hkv == 0) return PKV_OK;
  PKV_REQUIRE(positions, PKV_ERR_INVALID_ARG, "positions is NULL");
  PKV_REQUIRE((Hq == 0 || (q && q_out)) && (Hkv == 0 || (k && k_out)), PKV_ERR_INVALID_ARG,
              "NULL tensor");
  if (append)
    PKV_REQUIRE(v && slots && k_cache && v_cache && num_blocks >= 0, PKV_ERR_INVALID_ARG,
                "NULL append argument");
  RopeFreqs f;
  for (int i = 0; i < d / 2; ++i)
    f.inv[i] = std::pow(static_cast<double>(base), -2.0 * i / static_cast<double>(d));
  const size_t smem = sizeof(float) * d;
  const int64_t num_slots = static_cast<int64_t>(num_blocks) * kBlockTokens;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == PKV_BF16) {
    using T = __nv_bfloat16;
    auto kern = append ? rope_kernel<T, true> : rope_kernel<T, false>;
    kern<<<B, 128, smem, s>>>(static_cast<const T *>(q), static_cast<const T *>(k),
                              static_cast<const T *>(v), static_cast<T *>(q_out),
                              static_cast<T *>(k_out), positions, slots, static_cast<T *>(k_cache),
                              static_cast<T *>(v_cache), Hq, Hkv, d, num_slots, err, f);
  } else {
    using T = float;
    auto kern = append ? rope_kernel<T, true> : rope_kernel<T, false>;
    kern<<<B, 128, smem, s>>>(static_cast<const T *>(q), static_cast<const T *>(k),
                              static_cast<const T *>(v), static_cast<T *>(q_out),
                              static_cast<T *>(k_out), positions, slots, static_cast<T *>(k_cache),
                              static_cast<T *>(v_cache), Hq, Hkv, d, num_slots, err, f);
  }
  PKV_LAUNCH_CHECK("rope_kernel");
  return PKV_OK;
}
}  // namespace

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
