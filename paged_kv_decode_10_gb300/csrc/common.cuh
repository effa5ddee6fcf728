// Device helpers shared by the decode-step kernels: dtype traits, inline PTX
// for mbarriers, TMA tensor loads, ldmatrix, mma.sync, movmatrix and ex2.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>

#include "pkv.h"
#include "status.h"

#define PKV_CUDA_CHECK(expr)                                                   \
  do {                                                                         \
    cudaError_t _e = (expr);                                                   \
    if (_e != cudaSuccess)                                                     \
      return ::pkv::fail(PKV_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(_e)); \
  } while (0)

#define PKV_LAUNCH_CHECK(what)                                                 \
  do {                                                                         \
    cudaError_t _e = cudaGetLastError();                                       \
    if (_e != cudaSuccess)                                                     \
      return ::pkv::fail(PKV_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(_e)); \
  } while (0)

namespace pkv {

constexpr int kBlockTokens = PKV_BLOCK_SIZE;

inline size_t dtype_size(int dtype) { return dtype == PKV_BF16 ? 2 : 4; }
inline bool dtype_ok(int dtype) { return dtype == PKV_BF16 || dtype == PKV_F32; }

// Runs `set` (a kernel's cudaFuncSetAttribute calls) once per device: the
// attributes persist for the process, and a launch then costs no extra driver
// calls.  `done` is one flag word per kernel (bit = device ordinal).
template <typename F>
inline cudaError_t set_attributes_once(std::atomic<unsigned long long> &done, F &&set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = set();
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// ---- conversions ----------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// bf16 pair packed in a 32-bit word: low half = first element.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// ---- fast base-2 exponential (PTX ex2.approx; ex2(-inf) = +0) -------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fast base-2 logarithm (PTX lg2.approx; relative error ~2^-22)
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity; gives up after ~`limit_cycles`
// SM clocks and returns false (the caller then records PKV_DEVERR_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long limit_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit_cycles) return false;
  }
  return true;
}

// ---- TMA: 2-D tiled tensor load into shared memory ------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const void *tmap, int32_t x,
                                            int32_t y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// The same load with an L2 cache policy (createpolicy): pages streamed once
// per step go in as evict-first, so they do not push the kernel's code, the
// step metadata and the merge partials out of L2.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t smem_dst, const void *tmap, int32_t x,
                                                 int32_t y, uint64_t *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// 1-D bulk copy global -> shared completing on an mbarrier (both addresses
// 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_copy_g2s(uint32_t smem_dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---- warp-level tensor core path (bf16 in, f32 accumulate) ----------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a0, uint32_t &a1,
                                        uint32_t &a2, uint32_t &a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &a0, uint32_t &a1,
                                              uint32_t &a2, uint32_t &a3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// ---- rotate-half RoPE arithmetic, shared by every kernel that rotates ------
// Angle of pair i at position p in 64-bit fixed-point turns: `turn` is
// round(2^64 * base^(-2i/d) / (2 pi)) and p * turn mod 2^64 (an exact wrapping
// product) is the fractional turn of theta_i = p * base^(-2i/d).  Read as a
// signed value and scaled by 2 pi / 2^64 it is theta_i reduced to [-pi, pi).
__device__ __forceinline__ void rope_cossin(uint32_t pos, unsigned long long turn, float *c,
                                            float *s) {
  const unsigned long long ph = static_cast<unsigned long long>(pos) * turn;
  const float ang = static_cast<float>(static_cast<long long>(ph)) * 3.4061215800865545e-19f;
  sincosf(ang, s, c);
}
// (x1, x2) -> (x1 c - x2 s, x2 c + x1 s) with a fixed operation order, so every
// kernel produces bit-identical rotated values.
__device__ __forceinline__ void rope_rotate(float x1, float x2, float c, float s, float *y1,
                                            float *y2) {
  *y1 = fmaf(x1, c, -__fmul_rn(x2, s));
  *y2 = fmaf(x2, c, __fmul_rn(x1, s));
}

// Host: the fixed-point turn table of pairs i < d/2.
inline void fill_rope_turns(float base, int d, unsigned long long *turns) {
  for (int i = 0; i < d / 2; ++i) {
    const double f = std::pow(static_cast<double>(base), -2.0 * i / static_cast<double>(d)) /
                     (2.0 * 3.141592653589793238462643383279502884);
    turns[i] = static_cast<unsigned long long>(std::ldexp(f, 64));
  }
}

// ---- programmatic dependent launch (sm_90+) --------------------------------
// The dependent kernel may start before this grid ends; it must call
// pdl_wait() before touching anything this grid writes.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until every prerequisite grid has finished and its writes are visible
// (returns at once when the kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void set_dev_err(int32_t *flag, int bits) {
  if (flag) atomicOr(flag, bits);
}

// pkv_rope_append launched as a programmatic dependent of the kernel before it
// on the stream (a previous layer's attention): its q/k/v reads and cache
// writes wait for that kernel (rope_append.cu).
int rope_append_dependent(const void *q, const void *k, const void *v, void *q_out, void *k_out,
                          const int32_t *positions, const int64_t *slot_mapping, void *k_cache,
                          void *v_cache, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                          int32_t num_blocks, float base, int32_t dtype, int32_t *dev_err_flag,
                          void *stream);

}  // namespace pkv
