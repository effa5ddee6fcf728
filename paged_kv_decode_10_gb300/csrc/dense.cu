// The dense right-padded batch that paging replaces, kept as a comparator:
// helexa issue 121 -- slice 1's assemble_batch (right-pad every sequence's
// KV to the batch maximum and concatenate the rows) and slice 3a's
// extract_row (a row's prefix plus its lockstep decode columns, without the
// padding gap, back into a contiguous per-sequence snapshot); a join or leave
// re-batches by extracting every surviving row and assembling again.
//
// Both are token copies between caches in the block layout
// [blocks, Hkv, 16, d]: a snapshot is one sequence's blocks, a dense batch row
// b owns blocks [b * cap/16, (b+1) * cap/16).  Token t, head g of a buffer at
// block offset base lives at row ((base + t/16) * Hkv + g) * 16 + t%16.
#include <cstdint>

#include "common.cuh"

namespace pkv {
namespace {

struct CopyJob {
  const uint4 *k_src, *v_src;   // null: write zeros
  uint4 *k_dst, *v_dst;
  int32_t src_token, dst_token, count, pad;
};

constexpr int kJobsPerLaunch = 72;   // keeps the parameter block under 4 KB

struct CopyJobs {
  CopyJob job[kJobsPerLaunch];
};

// blockIdx.y = job.  threadIdx.x = (head, 16-byte chunk) of one token,
// threadIdx.y picks one of the block's tokens; blocks stride over the tokens.
// Token indices fit in 32 bits (checked by the callers).
__global__ void __launch_bounds__(1024) token_copy_kernel(const __grid_constant__ CopyJobs jobs,
                                                          int Hkv, int chunks) {
  const CopyJob &j = jobs.job[blockIdx.y];
  const int g = threadIdx.x / chunks, c = threadIdx.x - g * chunks;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  for (int i = blockIdx.x * blockDim.y + threadIdx.y; i < j.count; i += gridDim.x * blockDim.y) {
    const int td = j.dst_token + i;
    const size_t dst = ((static_cast<size_t>(td / kBlockTokens) * Hkv + g) * kBlockTokens +
                        td % kBlockTokens) * chunks + c;
    if (j.k_src) {
      const int ts = j.src_token + i;
      const size_t src = ((static_cast<size_t>(ts / kBlockTokens) * Hkv + g) * kBlockTokens +
                          ts % kBlockTokens) * chunks + c;
      j.k_dst[dst] = j.k_src[src];
      j.v_dst[dst] = j.v_src[src];
    } else {
      j.k_dst[dst] = zero;
      j.v_dst[dst] = zero;
    }
  }
}

int run_jobs(const CopyJob *all, int n, int Hkv, int d, int dtype, cudaStream_t s) {
  const int chunks = d * static_cast<int>(dtype_size(dtype)) / 16;
  const int per_tok = Hkv * chunks;
  PKV_REQUIRE(per_tok <= 1024, PKV_ERR_UNSUPPORTED, "Hkv * d too large for the copy kernel");
  const int tpb = per_tok >= 256 ? 1 : 256 / per_tok;   // tokens per block
  for (int j0 = 0; j0 < n; j0 += kJobsPerLaunch) {
    CopyJobs batch;
    const int m = n - j0 < kJobsPerLaunch ? n - j0 : kJobsPerLaunch;
    int most = 0;
    for (int i = 0; i < m; ++i) {
      batch.job[i] = all[j0 + i];
      if (all[j0 + i].count > most) most = all[j0 + i].count;
    }
    if (most == 0) continue;
    int gx = (most + tpb - 1) / tpb;
    if (gx > 4096) gx = 4096;
    token_copy_kernel<<<dim3(gx, m), dim3(per_tok, tpb), 0, s>>>(batch, Hkv, chunks);
    PKV_LAUNCH_CHECK("token_copy_kernel");
  }
  return PKV_OK;
}

int check_common(int Hkv, int d, int dtype, int cap) {
  PKV_REQUIRE(dtype_ok(dtype), PKV_ERR_UNSUPPORTED, "dtype %d", dtype);
  PKV_REQUIRE(Hkv > 0 && d > 0 && d * static_cast<int>(dtype_size(dtype)) % 16 == 0,
              PKV_ERR_UNSUPPORTED, "head_dim * sizeof(dtype) must be a multiple of 16");
  PKV_REQUIRE(cap > 0 && cap % kBlockTokens == 0, PKV_ERR_INVALID_ARG,
              "cap %d must be a positive multiple of 16", cap);
  return PKV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_dense_assemble(const void *const *k_snaps, const void *const *v_snaps,
                                  const int32_t *lens, int32_t B, int32_t padded_len,
                                  void *k_dense, void *v_dense, int32_t cap, int32_t Hkv,
                                  int32_t d, int32_t dtype, void *stream) {
  clear_error();
  int rc = check_common(Hkv, d, dtype, cap);
  if (rc != PKV_OK) return rc;
  PKV_REQUIRE(B >= 0 && padded_len >= 0 && padded_len <= cap, PKV_ERR_INVALID_ARG,
              "bad B or padded_len");
  if (B == 0) return PKV_OK;
  PKV_REQUIRE(k_snaps && v_snaps && lens && k_dense && v_dense, PKV_ERR_INVALID_ARG,
              "NULL pointer");
  PKV_REQUIRE(aligned16(k_dense) && aligned16(v_dense), PKV_ERR_INVALID_ARG,
              "dense caches must be 16-byte aligned");
  PKV_REQUIRE(static_cast<int64_t>(B) * cap < (int64_t{1} << 31), PKV_ERR_UNSUPPORTED,
              "dense batch too large");
  CopyJob *jobs = new CopyJob[2 * static_cast<size_t>(B)];
  int n = 0;
  for (int b = 0; b < B; ++b) {
    if (lens[b] < 0 || lens[b] > padded_len || (lens[b] > 0 && !(k_snaps[b] && v_snaps[b])) ||
        (lens[b] > 0 && !(aligned16(k_snaps[b]) && aligned16(v_snaps[b])))) {
      delete[] jobs;
      return fail(PKV_ERR_INVALID_ARG, "row %d: length %d outside [0, padded_len=%d] or bad "
                  "snapshot pointer", b, lens[b], padded_len);
    }
    const int64_t row0 = static_cast<int64_t>(b) * cap;   // first token of the dense row
    uint4 *kd = static_cast<uint4 *>(k_dense), *vd = static_cast<uint4 *>(v_dense);
    if (lens[b] > 0)
      jobs[n++] = CopyJob{static_cast<const uint4 *>(k_snaps[b]),
                          static_cast<const uint4 *>(v_snaps[b]), kd, vd, 0,
                          static_cast<int32_t>(row0), lens[b], 0};
    if (padded_len > lens[b])   // the padding gap holds zeros (finite under the mask)
      jobs[n++] = CopyJob{nullptr, nullptr, kd, vd, 0, static_cast<int32_t>(row0 + lens[b]),
                          padded_len - lens[b], 0};
  }
  rc = run_jobs(jobs, n, Hkv, d, dtype, static_cast<cudaStream_t>(stream));
  delete[] jobs;
  return rc;
}

extern "C" int pkv_dense_extract(const void *k_dense, const void *v_dense, int32_t cap,
                                 const int32_t *rows, const int32_t *prefix_lens, int32_t n_rows,
                                 int32_t padded_len, int32_t steps, void *const *k_snaps,
                                 void *const *v_snaps, int32_t Hkv, int32_t d, int32_t dtype,
                                 void *stream) {
  clear_error();
  int rc = check_common(Hkv, d, dtype, cap);
  if (rc != PKV_OK) return rc;
  PKV_REQUIRE(n_rows >= 0 && padded_len >= 0 && steps >= 0 &&
                  static_cast<int64_t>(padded_len) + steps <= cap,
              PKV_ERR_INVALID_ARG, "bad n_rows, padded_len or steps");
  if (n_rows == 0) return PKV_OK;
  PKV_REQUIRE(k_dense && v_dense && rows && prefix_lens && k_snaps && v_snaps,
              PKV_ERR_INVALID_ARG, "NULL pointer");
  CopyJob *jobs = new CopyJob[2 * static_cast<size_t>(n_rows)];
  int n = 0;
  const uint4 *kd = static_cast<const uint4 *>(k_dense), *vd = static_cast<const uint4 *>(v_dense);
  for (int i = 0; i < n_rows; ++i) {
    const int r = rows[i], pre = prefix_lens[i];
    if (r < 0 || static_cast<int64_t>(r + 1) * cap >= (int64_t{1} << 31) || pre < 0 ||
        pre > padded_len || !k_snaps[i] || !v_snaps[i] ||
        !aligned16(k_snaps[i]) || !aligned16(v_snaps[i])) {
      delete[] jobs;
      return fail(PKV_ERR_INVALID_ARG, "extract %d: bad row %d, prefix %d or snapshot", i, r, pre);
    }
    const int32_t row0 = r * cap;
    uint4 *ks = static_cast<uint4 *>(k_snaps[i]), *vs = static_cast<uint4 *>(v_snaps[i]);
    if (pre > 0) jobs[n++] = CopyJob{kd, vd, ks, vs, row0, 0, pre, 0};
    if (steps > 0) jobs[n++] = CopyJob{kd, vd, ks, vs, row0 + padded_len, pre, steps, 0};
  }
  rc = run_jobs(jobs, n, Hkv, d, dtype, static_cast<cudaStream_t>(stream));
  delete[] jobs;
  return rc;
}
