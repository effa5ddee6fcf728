// Host side of a3 (split-KV paged attention) and a4 (LSE merge), the merge
// kernel, and the composed decode step.
//
// LSE merge: the split partials of a unit are (o_s, lse_s) with o_s already
// normalised; out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M), M = max_s lse_s
// (base-2 log-sum-exp, which is how the split kernel stores it).  A unit whose
// partials all carry lse = -inf (nothing unmasked) outputs zeros, the
// zero-denominator guard of the "cortex-engine writeup" block-sparse kernel.
#include <cuda.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "attention_host.h"
#include "attention_kernel.cuh"

namespace pkv {
namespace {

constexpr int kMaxB = 65536;
constexpr int kMaxParts = 4096;
// PKV_ATTN_SHORT_WAITS: every wait gives up after this many SM clocks
constexpr long long kShortWaitCycles = 64;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Workspace {
  int32_t *counters;       // [U] partials written, per unit
  int32_t *done;           // [U] merge helpers finished, per unit
  int32_t *meta;           // [U x 2 + 2]
  float *lse, *o;          // [(U + C) x G], [(U + C) x G x D]
  size_t bytes;
  size_t counter_bytes;    // the leading counters and done regions
};

// [counters][done][meta][lse][o], each region 256-byte aligned.  Unit u's
// partial from part c sits at slot u + c (slots of different units never
// coincide: a later unit's parts start no earlier than the previous unit's
// last part).
Workspace workspace_layout(void *base, int B, int Hq, int Hkv, int D, int C) {
  const size_t U = static_cast<size_t>(B) * Hkv;
  const size_t G = static_cast<size_t>(Hq / Hkv);
  const size_t S = U + static_cast<size_t>(C);
  const size_t sizes[5] = {align256(U * sizeof(int32_t)), align256(U * sizeof(int32_t)),
                           align256((U * 2 + 2) * sizeof(int32_t)),
                           align256(S * G * sizeof(float)),
                           align256(S * G * static_cast<size_t>(D) * sizeof(float))};
  char *p = static_cast<char *>(base);
  char *r[5];
  size_t off = 0;
  for (int i = 0; i < 5; ++i) {
    r[i] = p + off;
    off += sizes[i];
  }
  return Workspace{reinterpret_cast<int32_t *>(r[0]), reinterpret_cast<int32_t *>(r[1]),
                   reinterpret_cast<int32_t *>(r[2]), reinterpret_cast<float *>(r[3]),
                   reinterpret_cast<float *>(r[4]), off, sizes[0] + sizes[1]};
}

// ---- cuTensorMapEncodeTiled through the runtime's driver entry point ------
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeFn>(nullptr);
    return reinterpret_cast<EncodeFn>(ptr);
  }();
  return fn;
}

// The cache viewed as a 2-D tensor [num_blocks*Hkv*16 rows, D elements]; the
// box is one 128-byte column slab of one 16-token page, swizzled 128B.
struct TmapKey {
  const void *base;
  long long rows;
  int D, dtype;
};

struct TmapCache {
  static constexpr int kN = 128;   // a K and a V map per layer of a deep model
  std::mutex mu;
  TmapKey key[kN];
  CUtensorMap map[kN];
  int used = 0, next = 0;
};

int get_tmap(const void *base, long long rows, int D, int dtype, CUtensorMap *out) {
  static TmapCache cache;
  std::lock_guard<std::mutex> lock(cache.mu);
  for (int i = 0; i < cache.used; ++i) {
    const TmapKey &k = cache.key[i];
    if (k.base == base && k.rows == rows && k.D == D && k.dtype == dtype) {
      *out = cache.map[i];
      return PKV_OK;
    }
  }
  EncodeFn enc = encode_fn();
  PKV_REQUIRE(enc, PKV_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  const int elem = static_cast<int>(dtype_size(dtype));
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * elem};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem),
                             static_cast<cuuint32_t>(kBlockTokens)};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  std::memset(&m, 0, sizeof(m));
  const CUresult r = enc(&m,
                         dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                         2, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  PKV_REQUIRE(r == CUDA_SUCCESS, PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)",
              static_cast<int>(r));
  const int slot = cache.used < TmapCache::kN ? cache.used++ : (cache.next++ % TmapCache::kN);
  cache.key[slot] = TmapKey{base, rows, D, dtype};
  cache.map[slot] = m;
  *out = m;
  return PKV_OK;
}

bool pick_variant(int dtype, int D, int G, int flags, AttnVariant *v) {
  if (dtype == PKV_BF16 && !(flags & PKV_ATTN_SIMT)) return attn_variant_mma(D, v);
  if (dtype == PKV_BF16) return attn_variant_simt_bf16(D, G, v);
  return attn_variant_simt_f32(D, G, v);
}

// CTAs of a variant that are resident at once on the current device (SMs x
// blocks per SM), remembered per (device, variant).
int resident_ctas(const AttnVariant &v, int *ctas) {
  struct Entry {
    int device;
    cudaError_t (*occupancy)(int *);
    int ctas;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int used = 0;
  int dev = 0;
  PKV_CUDA_CHECK(cudaGetDevice(&dev));
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].device == dev && cache[i].occupancy == v.occupancy) {
        *ctas = cache[i].ctas;
        return PKV_OK;
      }
  }
  int sms = 0, occ = 0;
  PKV_CUDA_CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  PKV_CUDA_CHECK(v.occupancy(&occ));
  PKV_REQUIRE(occ > 0, PKV_ERR_CUDA, "attention kernel cannot be resident (smem %d)",
              v.smem_bytes);
  std::lock_guard<std::mutex> lock(mu);
  if (used < 64) cache[used++] = Entry{dev, v.occupancy, sms * occ};
  *ctas = sms * occ;
  return PKV_OK;
}

}  // namespace

int check_shapes(int B, int Hq, int Hkv, int D, int dtype) {
  PKV_REQUIRE(dtype_ok(dtype), PKV_ERR_UNSUPPORTED, "dtype %d", dtype);
  PKV_REQUIRE(D == 64 || D == 128, PKV_ERR_UNSUPPORTED, "head_dim %d (built: 64, 128)", D);
  PKV_REQUIRE(B >= 0 && B <= kMaxB, PKV_ERR_UNSUPPORTED, "B = %d (max %d)", B, kMaxB);
  PKV_REQUIRE(Hkv > 0 && Hq > 0 && Hq % Hkv == 0, PKV_ERR_INVALID_ARG,
              "Hq (%d) must be a positive multiple of Hkv (%d)", Hq, Hkv);
  const int G = Hq / Hkv;
  PKV_REQUIRE(G == 1 || G == 2 || G == 4 || G == 8, PKV_ERR_UNSUPPORTED,
              "group size %d (built: 1, 2, 4, 8)", G);
  return PKV_OK;
}

int default_parts(int D, int dtype, int flags, int G, int *parts) {
  AttnVariant v;
  PKV_REQUIRE(pick_variant(dtype, D, G, flags, &v), PKV_ERR_UNSUPPORTED, "no kernel variant");
  return resident_ctas(v, parts);
}

size_t workspace_counter_bytes(int B, int Hq, int Hkv, int D, int C) {
  return workspace_layout(nullptr, B, Hq, Hkv, D, C).counter_bytes;
}

namespace {

// ---- a4: LSE merge ----------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) lse_merge_kernel(const float *__restrict__ o_part,
                                                        const float *__restrict__ lse_part,
                                                        const int32_t *__restrict__ meta,
                                                        const int32_t *__restrict__ seq_lens,
                                                        int bt_stride, int bias_stride, int Hq,
                                                        int Hkv, int D, int num_parts,
                                                        T *__restrict__ out) {
  const int u = blockIdx.x;
  const int b = u / Hkv, g = u - b * Hkv;
  const int G = Hq / Hkv;
  bool bad;
  const int n = row_pages(seq_lens, b, bt_stride, bias_stride > 0, bias_stride, &bad);
  T *o = out + (static_cast<size_t>(b) * Hq + g * G) * D;
  if (n == 0) {
    for (int e = threadIdx.x; e < G * D; e += blockDim.x) o[e] = from_f32<T>(0.f);
    return;
  }
  const int c0 = meta[2 * u], nseg = meta[2 * u + 1];
  if (nseg == 1) return;   // written by the split kernel
  if (c0 < 0 || nseg < 1 || c0 + nseg > num_parts) {
    // meta not written by a matching split call: never read outside the workspace
    for (int e = threadIdx.x; e < G * D; e += blockDim.x) o[e] = from_f32<T>(NAN);
    return;
  }
  const int Uall = gridDim.x;
  const long long P = static_cast<long long>(static_cast<uint32_t>(meta[2 * Uall])) |
                      (static_cast<long long>(meta[2 * Uall + 1]) << 32);
  const size_t first = static_cast<size_t>(u) + c0;
  auto skip = [&](int i) { return num_parts > P && part_empty(c0 + i, P, num_parts); };
  for (int col = threadIdx.x; col < G * D / 4; col += blockDim.x) {
    const int h = col / (D / 4), d4 = col - h * (D / 4);
    float l;
    store4<T>(o + h * D + 4 * d4,
              merge_column(o_part, lse_part, first, nseg, 1, G, D, h, d4, skip, &l));
  }
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_attn_default_parts(int32_t d, int32_t Hq, int32_t Hkv, int32_t dtype,
                                      int32_t flags, int32_t *num_parts) {
  clear_error();
  PKV_REQUIRE(num_parts, PKV_ERR_INVALID_ARG, "num_parts is NULL");
  int rc = check_shapes(1, Hq, Hkv, d, dtype);
  if (rc != PKV_OK) return rc;
  int parts = 0;
  rc = default_parts(d, dtype, flags, Hq / Hkv, &parts);
  if (rc != PKV_OK) return rc;
  *num_parts = parts;
  return PKV_OK;
}

extern "C" int pkv_attn_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                                        int32_t num_parts, size_t *bytes) {
  clear_error();
  PKV_REQUIRE(bytes, PKV_ERR_INVALID_ARG, "bytes is NULL");
  PKV_REQUIRE(num_parts > 0 && num_parts <= kMaxParts, PKV_ERR_INVALID_ARG,
              "num_parts must be in [1, %d]", kMaxParts);
  const int rc = check_shapes(B, Hq, Hkv, d, PKV_F32);
  if (rc != PKV_OK) return rc;
  *bytes = workspace_layout(nullptr, B, Hq, Hkv, d, num_parts).bytes;
  return PKV_OK;
}

namespace {

// a3 (+ a4 fused) launch; with `step` the whole-step kernel that also does a1
// + a2 from step->q/k/v, positions and slot_mapping (q_rot then only receives
// the rotated queries).
int attn_launch(const void *q_rot, const void *k_cache, const void *v_cache, int32_t num_blocks,
                const int32_t *block_tables, int32_t bt_stride, const int32_t *seq_lens,
                const float *attn_bias, int32_t bias_stride, int32_t B, int32_t Hq, int32_t Hkv,
                int32_t d, float scale, int32_t num_parts, void *workspace,
                size_t workspace_bytes, void *out, int32_t dtype, int32_t flags,
                int32_t *dev_err_flag, void *stream, const pkv_step_args *step,
                const int32_t *plan, bool allow_helpers = true) {
  int rc = check_shapes(B, Hq, Hkv, d, dtype);
  if (rc != PKV_OK) return rc;
  if (B == 0) return PKV_OK;
  PKV_REQUIRE(q_rot && k_cache && v_cache && block_tables && seq_lens && out && workspace,
              PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(num_blocks > 0, PKV_ERR_INVALID_ARG, "num_blocks must be positive");
  PKV_REQUIRE(static_cast<long long>(num_blocks) * Hkv * kBlockTokens < (1ll << 31),
              PKV_ERR_UNSUPPORTED, "pool too large for 32-bit TMA row coordinates");
  PKV_REQUIRE(bt_stride > 0 && bt_stride < (1 << 26), PKV_ERR_INVALID_ARG, "bt_stride %d",
              bt_stride);
  PKV_REQUIRE(!attn_bias || bias_stride > 0, PKV_ERR_INVALID_ARG,
              "bias_stride must be positive when attn_bias is given");
  PKV_REQUIRE((reinterpret_cast<uintptr_t>(k_cache) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(v_cache) & 15) == 0,
              PKV_ERR_INVALID_ARG, "caches must be 16-byte aligned");
  // q_rot rows are bulk-copied into shared memory: 16-byte alignment
  PKV_REQUIRE((reinterpret_cast<uintptr_t>(q_rot) & 15) == 0 &&
                  (reinterpret_cast<uintptr_t>(workspace) & 255) == 0,
              PKV_ERR_INVALID_ARG, "q_rot must be 16-byte and workspace 256-byte aligned");
  // output rows are written with vector stores
  PKV_REQUIRE((reinterpret_cast<uintptr_t>(out) & 15) == 0, PKV_ERR_INVALID_ARG,
              "out must be 16-byte aligned");
  const int G = Hq / Hkv;
  PKV_REQUIRE(!plan || num_parts > 0, PKV_ERR_INVALID_ARG,
              "a plan is made for a given num_parts: pass it");
  PKV_REQUIRE(!plan || (reinterpret_cast<uintptr_t>(plan) & 15) == 0, PKV_ERR_INVALID_ARG,
              "plan must be 16-byte aligned");
  if (num_parts <= 0) {
    rc = default_parts(d, dtype, flags, G, &num_parts);
    if (rc != PKV_OK) return rc;
  }
  PKV_REQUIRE(num_parts <= kMaxParts, PKV_ERR_INVALID_ARG, "num_parts must be <= %d",
              kMaxParts);
  const Workspace ws = workspace_layout(workspace, B, Hq, Hkv, d, num_parts);
  PKV_REQUIRE(workspace_bytes >= ws.bytes, PKV_ERR_INVALID_ARG,
              "workspace of %zu bytes < %zu needed", workspace_bytes, ws.bytes);
  AttnVariant v;
  PKV_REQUIRE(pick_variant(dtype, d, G, flags, &v), PKV_ERR_UNSUPPORTED, "no kernel variant");
  const long long rows = static_cast<long long>(num_blocks) * Hkv * kBlockTokens;
  CUtensorMap tk, tv;
  rc = get_tmap(k_cache, rows, d, dtype, &tk);
  if (rc != PKV_OK) return rc;
  rc = get_tmap(v_cache, rows, d, dtype, &tv);
  if (rc != PKV_OK) return rc;
  AttnParams p;
  p.q = q_rot;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.bias = attn_bias;
  p.o_part = ws.o;
  p.lse_part = ws.lse;
  p.meta = ws.meta;
  p.counters = ws.counters;
  p.done = ws.done;
  p.fuse_merge = (flags & PKV_ATTN_SEPARATE_MERGE) ? 0 : 1;
  // A grid that fits on the GPU at once is launched cooperatively, which
  // guarantees that every CTA is resident; only then may the merge of a unit
  // be shared by several parts that wait for each other.  (A chain of layers
  // does without: a cooperative grid starts only once all of its CTAs fit, so
  // the next layer could no longer start on the SMs the previous one frees.)
  int resident = 0;
  rc = resident_ctas(v, &resident);
  if (rc != PKV_OK) return rc;
  p.max_helpers = (allow_helpers && num_parts <= resident) ? kMaxHelpers : 1;
  p.wait_limit = (flags & PKV_ATTN_SHORT_WAITS) ? kShortWaitCycles : kWaitLimitCycles;
  p.seg_cost = seg_cost(d);
  p.out = out;
  p.plan = plan;
  p.check_plan = (flags & PKV_ATTN_CHECK_PLAN) ? 1 : 0;
  p.err = dev_err_flag;
  p.bt_stride = bt_stride;
  p.bias_stride = attn_bias ? bias_stride : 0;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.num_blocks = num_blocks;
  p.num_parts = num_parts;
  p.scale_log2 = scale * kLog2e;
  cudaError_t e;
  if (step) {
    PKV_REQUIRE(step->q && step->k && step->v && step->k_rot && step->positions &&
                    step->slot_mapping,
                PKV_ERR_INVALID_ARG, "NULL step argument");
    PKV_REQUIRE(step->rope_base > 0.0f, PKV_ERR_INVALID_ARG, "rope base must be positive");
    PKV_REQUIRE((reinterpret_cast<uintptr_t>(step->q) & 15) == 0, PKV_ERR_INVALID_ARG,
                "the whole-step kernel reads q in 16-byte pieces: q must be 16-byte aligned");
    p.q_new = step->q;
    p.k_new = step->k;
    p.v_new = step->v;
    p.positions = step->positions;
    p.slots = step->slot_mapping;
    p.k_cache_w = const_cast<void *>(k_cache);
    p.v_cache_w = const_cast<void *>(v_cache);
    p.q_rot_out = const_cast<void *>(q_rot);
    p.k_rot_out = step->k_rot;
    p.num_slots = static_cast<long long>(num_blocks) * kBlockTokens;
    fill_rope_turns(step->rope_base, d, p.turns);
    e = v.launch_step(tk, tv, p, static_cast<cudaStream_t>(stream));
  } else {
    e = v.launch(tk, tv, p, static_cast<cudaStream_t>(stream));
  }
  PKV_REQUIRE(e == cudaSuccess, PKV_ERR_CUDA, "attn_split_kernel launch: %s",
              cudaGetErrorString(e));
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_decode_attn_split(const void *q_rot, const void *k_cache, const void *v_cache,
                                     int32_t num_blocks, const int32_t *block_tables,
                                     int32_t bt_stride, const int32_t *seq_lens,
                                     const float *attn_bias, int32_t bias_stride, int32_t B,
                                     int32_t Hq, int32_t Hkv, int32_t d, float scale,
                                     int32_t num_parts, void *workspace, size_t workspace_bytes,
                                     void *out, int32_t dtype, int32_t flags,
                                     int32_t *dev_err_flag, void *stream) {
  clear_error();
  return attn_launch(q_rot, k_cache, v_cache, num_blocks, block_tables, bt_stride, seq_lens,
                     attn_bias, bias_stride, B, Hq, Hkv, d, scale, num_parts, workspace,
                     workspace_bytes, out, dtype, flags, dev_err_flag, stream, nullptr, nullptr);
}

extern "C" int pkv_decode_attn_planned(const void *q_rot, const void *k_cache,
                                       const void *v_cache, int32_t num_blocks,
                                       const int32_t *block_tables, int32_t bt_stride,
                                       const int32_t *seq_lens, const float *attn_bias,
                                       int32_t bias_stride, int32_t B, int32_t Hq, int32_t Hkv,
                                       int32_t d, float scale, int32_t num_parts,
                                       const int32_t *plan, void *workspace,
                                       size_t workspace_bytes, void *out, int32_t dtype,
                                       int32_t flags, int32_t *dev_err_flag, void *stream) {
  clear_error();
  PKV_REQUIRE(plan, PKV_ERR_INVALID_ARG, "plan is NULL");
  return attn_launch(q_rot, k_cache, v_cache, num_blocks, block_tables, bt_stride, seq_lens,
                     attn_bias, bias_stride, B, Hq, Hkv, d, scale, num_parts, workspace,
                     workspace_bytes, out, dtype, flags, dev_err_flag, stream, nullptr, plan);
}

extern "C" int pkv_lse_merge(const void *workspace, size_t workspace_bytes,
                             const int32_t *seq_lens, int32_t bt_stride, int32_t bias_stride,
                             int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_parts,
                             void *out, int32_t dtype, void *stream) {
  clear_error();
  int rc = check_shapes(B, Hq, Hkv, d, dtype);
  if (rc != PKV_OK) return rc;
  if (B == 0) return PKV_OK;
  PKV_REQUIRE(workspace && seq_lens && out, PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_REQUIRE(bt_stride > 0 && bt_stride < (1 << 26), PKV_ERR_INVALID_ARG, "bt_stride %d",
              bt_stride);
  PKV_REQUIRE(bias_stride >= 0, PKV_ERR_INVALID_ARG, "bias_stride < 0");
  if (num_parts <= 0) {
    rc = default_parts(d, dtype, 0, Hq / Hkv, &num_parts);
    if (rc != PKV_OK) return rc;
  }
  const Workspace ws = workspace_layout(const_cast<void *>(workspace), B, Hq, Hkv, d, num_parts);
  PKV_REQUIRE(workspace_bytes >= ws.bytes, PKV_ERR_INVALID_ARG,
              "workspace of %zu bytes < %zu needed", workspace_bytes, ws.bytes);
  const int U = B * Hkv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == PKV_BF16)
    lse_merge_kernel<__nv_bfloat16><<<U, 256, 0, s>>>(ws.o, ws.lse, ws.meta, seq_lens, bt_stride,
                                                      bias_stride, Hq, Hkv, d, num_parts,
                                                      static_cast<__nv_bfloat16 *>(out));
  else
    lse_merge_kernel<float><<<U, 256, 0, s>>>(ws.o, ws.lse, ws.meta, seq_lens, bt_stride,
                                              bias_stride, Hq, Hkv, d, num_parts, static_cast<float *>(out));
  PKV_LAUNCH_CHECK("lse_merge_kernel");
  return PKV_OK;
}

extern "C" int pkv_decode_step(const pkv_step_args *a, void *stream) {
  clear_error();
  PKV_REQUIRE(a, PKV_ERR_INVALID_ARG, "args is NULL");
  PKV_REQUIRE(!a->plan || a->num_parts > 0, PKV_ERR_INVALID_ARG,
              "a plan is made for a given num_parts: set args->num_parts");
  int num_parts = a->num_parts;
  if (num_parts <= 0 && a->B > 0) {
    int rc = check_shapes(a->B, a->Hq, a->Hkv, a->d, a->dtype);
    if (rc != PKV_OK) return rc;
    rc = default_parts(a->d, a->dtype, a->flags, a->Hq / a->Hkv, &num_parts);
    if (rc != PKV_OK) return rc;
  }
  int rc;
  if (!(a->flags & PKV_STEP_FUSED)) {
    rc = pkv_rope_append(a->q, a->k, a->v, a->q_rot, a->k_rot, a->positions, a->slot_mapping,
                         a->k_cache, a->v_cache, a->B, a->Hq, a->Hkv, a->d, a->num_blocks,
                         a->rope_base, a->dtype, a->dev_err_flag, stream);
    if (rc != PKV_OK) return rc;
    clear_error();
    rc = attn_launch(a->q_rot, a->k_cache, a->v_cache, a->num_blocks, a->block_tables,
                     a->bt_stride, a->seq_lens, a->attn_bias, a->bias_stride, a->B, a->Hq, a->Hkv,
                     a->d, a->scale, num_parts, a->workspace, a->workspace_bytes, a->out,
                     a->dtype, a->flags, a->dev_err_flag, stream, nullptr, a->plan);
  } else {
    // PKV_STEP_FUSED: the whole step in one launch
    rc = attn_launch(a->q_rot, a->k_cache, a->v_cache, a->num_blocks, a->block_tables,
                     a->bt_stride, a->seq_lens, a->attn_bias, a->bias_stride, a->B, a->Hq, a->Hkv,
                     a->d, a->scale, num_parts, a->workspace, a->workspace_bytes, a->out,
                     a->dtype, a->flags, a->dev_err_flag, stream, a, a->plan);
  }
  if (rc != PKV_OK) return rc;
  if (!(a->flags & PKV_ATTN_SEPARATE_MERGE)) return PKV_OK;
  return pkv_lse_merge(a->workspace, a->workspace_bytes, a->seq_lens, a->bt_stride,
                       a->attn_bias ? a->bias_stride : 0, a->B, a->Hq, a->Hkv, a->d, num_parts,
                       a->out, a->dtype, stream);
}

extern "C" int pkv_decode_step_layers(const pkv_step_args *layers, int32_t n_layers,
                                      void *stream) {
  clear_error();
  PKV_REQUIRE(n_layers >= 0 && (layers || n_layers == 0), PKV_ERR_INVALID_ARG,
              "bad layer list");
  for (int32_t l = 0; l < n_layers; ++l) {   // checked before anything is launched
    PKV_REQUIRE(!(layers[l].flags & PKV_STEP_FUSED), PKV_ERR_UNSUPPORTED,
                "PKV_STEP_FUSED is a single-layer form");
    PKV_REQUIRE(!layers[l].plan || layers[l].num_parts > 0, PKV_ERR_INVALID_ARG,
                "a plan is made for a given num_parts: set num_parts");
    if (l > 0)
      PKV_REQUIRE(layers[l].workspace != layers[l - 1].workspace, PKV_ERR_INVALID_ARG,
                  "layers %d and %d share a workspace", l - 1, l);
  }
  for (int32_t l = 0; l < n_layers; ++l) {
    const pkv_step_args *a = &layers[l];
    int num_parts = a->num_parts;
    int rc;
    if (num_parts <= 0 && a->B > 0) {
      rc = check_shapes(a->B, a->Hq, a->Hkv, a->d, a->dtype);
      if (rc != PKV_OK) return rc;
      rc = default_parts(a->d, a->dtype, a->flags, a->Hq / a->Hkv, &num_parts);
      if (rc != PKV_OK) return rc;
    }
    if (l == 0) {
      rc = pkv_rope_append(a->q, a->k, a->v, a->q_rot, a->k_rot, a->positions, a->slot_mapping,
                           a->k_cache, a->v_cache, a->B, a->Hq, a->Hkv, a->d, a->num_blocks,
                           a->rope_base, a->dtype, a->dev_err_flag, stream);
    } else {
      clear_error();
      rc = rope_append_dependent(a->q, a->k, a->v, a->q_rot, a->k_rot, a->positions,
                                 a->slot_mapping, a->k_cache, a->v_cache, a->B, a->Hq, a->Hkv,
                                 a->d, a->num_blocks, a->rope_base, a->dtype, a->dev_err_flag,
                                 stream);
    }
    if (rc != PKV_OK) return rc;
    clear_error();
    rc = attn_launch(a->q_rot, a->k_cache, a->v_cache, a->num_blocks, a->block_tables,
                     a->bt_stride, a->seq_lens, a->attn_bias, a->bias_stride, a->B, a->Hq, a->Hkv,
                     a->d, a->scale, num_parts, a->workspace, a->workspace_bytes, a->out,
                     a->dtype, a->flags, a->dev_err_flag, stream, nullptr, a->plan,
                     /*allow_helpers=*/(a->flags & PKV_LAYERS_MERGE_HELPERS) != 0);
    if (rc != PKV_OK) return rc;
    if (a->flags & PKV_ATTN_SEPARATE_MERGE) {
      rc = pkv_lse_merge(a->workspace, a->workspace_bytes, a->seq_lens, a->bt_stride,
                         a->attn_bias ? a->bias_stride : 0, a->B, a->Hq, a->Hkv, a->d, num_parts,
                         a->out, a->dtype, stream);
      if (rc != PKV_OK) return rc;
    }
  }
  return PKV_OK;
}

extern "C" int pkv_mapped_pointer(const void *host_ptr, void **device_ptr) {
  clear_error();
  PKV_REQUIRE(host_ptr && device_ptr, PKV_ERR_INVALID_ARG, "NULL pointer");
  PKV_CUDA_CHECK(cudaHostGetDevicePointer(device_ptr, const_cast<void *>(host_ptr), 0));
  return PKV_OK;
}
