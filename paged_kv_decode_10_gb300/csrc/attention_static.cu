// Split-KV paged attention for callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace: code that runs
// inside another runtime's memory manager with no access to cudaMalloc (or
// where an allocation would have to go through a host round trip the caller
// cannot afford), plugins handed only the tensors they read and write, or
// stream-ordered code paths that must never trigger an allocator.  For them
// pkv_decode_attn_static runs the same attention kernel as
// pkv_decode_attn_split, with its scratch (merge counters, split partials)
// taken from a fixed array compiled into this library instead of a
// caller-provided buffer.  The caller still passes every input and output.
//
// The array lives in device global memory on every GPU that loads the library
// and stays allocated until the process exits.  Its device address is looked
// up once per device with cudaGetSymbolAddress (the host-side name of a
// __device__ variable is not a device address).
#include <mutex>

#include "attention_host.h"
#include "common.cuh"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (set up on first use).
int scratch_address(void **out) {
  int dev = 0;
  PKV_CUDA_CHECK(cudaGetDevice(&dev));
  PKV_REQUIRE(dev >= 0 && dev < kMaxDevices, PKV_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
    PKV_REQUIRE(e == cudaSuccess && p, PKV_ERR_CUDA,
                "cudaGetSymbolAddress of the static attention scratch: %s",
                cudaGetErrorString(e));
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_decode_attn_static(const void *q_rot, const void *k_cache,
                                      const void *v_cache, int32_t num_blocks,
                                      const int32_t *block_tables, int32_t bt_stride,
                                      const int32_t *seq_lens, const float *attn_bias,
                                      int32_t bias_stride, int32_t B, int32_t Hq, int32_t Hkv,
                                      int32_t d, float scale, int32_t num_parts, void *out,
                                      int32_t dtype, int32_t flags, int32_t *dev_err_flag,
                                      void *stream) {
  pkv::clear_error();
  PKV_REQUIRE(!(flags & PKV_ATTN_SEPARATE_MERGE), PKV_ERR_INVALID_ARG,
              "the static-scratch call always merges in the attention kernel");
  if (B == 0) return PKV_OK;
  size_t need = 0;
  // (pkv_attn_workspace_bytes also checks the shapes, so Hq / Hkv is valid
  // below; it needs a part count, so a default one is sized after it)
  int rc = pkv_attn_workspace_bytes(B, Hq, Hkv, d, num_parts > 0 ? num_parts : 1, &need);
  if (rc != PKV_OK) return rc;
  if (num_parts <= 0) {
    // the same default as pkv_decode_attn_split: it depends on the group size
    rc = pkv::default_parts(d, dtype, flags, Hq / Hkv, &num_parts);
    if (rc != PKV_OK) return rc;
    rc = pkv_attn_workspace_bytes(B, Hq, Hkv, d, num_parts, &need);
    if (rc != PKV_OK) return rc;
  }
  PKV_REQUIRE(need <= kStaticScratchBytes, PKV_ERR_UNSUPPORTED,
              "this call needs %zu bytes of scratch, more than the %zu-byte static array "
              "(use pkv_decode_attn_split with a caller-provided workspace)",
              need, kStaticScratchBytes);
  void *scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != PKV_OK) return rc;
  // The kernel reads nothing of its scratch before writing it except the merge
  // counters, which it expects at zero and leaves at zero.  An earlier call
  // with another layout (other B, heads or parts), or one that gave up a wait,
  // can leave non-zero words where this call's counters sit: clear them.
  PKV_CUDA_CHECK(cudaMemsetAsync(scratch, 0, pkv::workspace_counter_bytes(B, Hq, Hkv, d,
                                                                          num_parts),
                                 static_cast<cudaStream_t>(stream)));
  return pkv_decode_attn_split(q_rot, k_cache, v_cache, num_blocks, block_tables, bt_stride,
                               seq_lens, attn_bias, bias_stride, B, Hq, Hkv, d, scale, num_parts,
                               scratch, need, out, dtype, flags, dev_err_flag, stream);
}
