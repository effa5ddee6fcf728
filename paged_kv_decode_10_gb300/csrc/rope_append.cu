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

// One CTA per batch row.  Threads first build cos/sin of every pair at the
// row's position (angle formed and reduced modulo 2*pi in double precision so
// that positions of 10^5 keep float32-level angles), then rotate every head of
// q and k.
template <typename T>
__global__ void rope_kernel(const T *__restrict__ q, const T *__restrict__ k,
                            T *__restrict__ q_out, T *__restrict__ k_out,
                            const int32_t *__restrict__ positions, int Hq, int Hkv, int d,
                            double log2_base) {
  extern __shared__ float cs[];  // cos[half], sin[half]
  const int b = blockIdx.x;
  const int half = d >> 1;
  const double p = static_cast<double>(positions[b]);
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const double inv_freq = exp2(-(2.0 * i / d) * log2_base);
    const double theta = p * inv_freq;
    const double turns = rint(theta * (1.0 / kTwoPi));
    const double r = fma(-turns, kTwoPi, theta);
    float s, c;
    sincosf(static_cast<float>(r), &s, &c);
    cs[i] = c;
    cs[half + i] = s;
  }
  __syncthreads();
  const int heads = Hq + Hkv;
  for (int e = threadIdx.x; e < heads * half; e += blockDim.x) {
    const int h = e / half;
    const int i = e - h * half;
    const T *src;
    T *dst;
    if (h < Hq) {
      src = q + (static_cast<size_t>(b) * Hq + h) * d;
      dst = q_out + (static_cast<size_t>(b) * Hq + h) * d;
    } else {
      src = k + (static_cast<size_t>(b) * Hkv + (h - Hq)) * d;
      dst = k_out + (static_cast<size_t>(b) * Hkv + (h - Hq)) * d;
    }
    const float x1 = to_f32(src[i]);
    const float x2 = to_f32(src[i + half]);
    const float c = cs[i], s = cs[half + i];
    dst[i] = from_f32<T>(x1 * c - x2 * s);
    dst[i + half] = from_f32<T>(x2 * c + x1 * s);
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

extern "C" int pkv_rope(const void *q, const void *k, void *q_out, void *k_out,
                        const int32_t *positions, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                        float base, int32_t dtype, void *stream) {
  clear_error();
  PKV_REQUIRE(B >= 0 && Hq >= 0 && Hkv >= 0, PKV_ERR_INVALID_ARG, "negative size");
  PKV_REQUIRE(d >= 2 && d <= 256 && d % 2 == 0, PKV_ERR_UNSUPPORTED, "head_dim %d", d);
  PKV_REQUIRE(dtype_ok(dtype), PKV_ERR_UNSUPPORTED, "dtype %d", dtype);
  PKV_REQUIRE(base > 0.0f, PKV_ERR_INVALID_ARG, "rope base must be positive");
  if (B == 0 || Hq + Hkv == 0) return PKV_OK;
  PKV_REQUIRE(positions, PKV_ERR_INVALID_ARG, "positions is NULL");
  PKV_REQUIRE((Hq == 0 || (q && q_out)) && (Hkv == 0 || (k && k_out)), PKV_ERR_INVALID_ARG,
              "NULL tensor");
  const double log2_base = std::log2(static_cast<double>(base));
  const size_t smem = sizeof(float) * d;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == PKV_BF16) {
    rope_kernel<__nv_bfloat16><<<B, 128, smem, s>>>(
        static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
        static_cast<__nv_bfloat16 *>(q_out), static_cast<__nv_bfloat16 *>(k_out), positions, Hq,
        Hkv, d, log2_base);
  } else {
    rope_kernel<float><<<B, 128, smem, s>>>(static_cast<const float *>(q),
                                            static_cast<const float *>(k),
                                            static_cast<float *>(q_out),
                                            static_cast<float *>(k_out), positions, Hq, Hkv, d,
                                            log2_base);
  }
  PKV_LAUNCH_CHECK("rope_kernel");
  return PKV_OK;
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
