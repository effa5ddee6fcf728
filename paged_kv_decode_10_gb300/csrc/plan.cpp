// Host-planned partition of the split-KV attention kernel (pkv_plan_parts).
//
// The kernel balances, over its num_parts CTAs, the pages of the (row, KV
// head) units plus a fixed cost A per unit boundary: a unit of n > 0 pages is
// n + A consecutive positions, the first A without a page, units laid end to
// end in row-major order, and part c owns positions
// [floor(c*P/C), floor((c+1)*P/C)).  This file states that partition on the
// host, from the metadata a0 has just written, so that a CTA can start from
// its record instead of scanning every row length and then reading its first
// block ids.  The rule for which rows count (valid lengths) and the cost A are
// the kernel's; the kernel can verify a plan (PKV_ATTN_CHECK_PLAN).
#include <cstdint>
#include <vector>

#include "attention_host.h"
#include "status.h"

namespace {
constexpr int32_t kBlock = PKV_BLOCK_SIZE;

// Pages of a row of length L, or 0 for a length the kernel treats as invalid.
int64_t row_pages(int32_t L, int32_t bt_stride, int32_t bias_stride) {
  const bool ok = L >= 0 && static_cast<int64_t>(L) <= static_cast<int64_t>(bt_stride) * kBlock &&
                  (bias_stride <= 0 || L <= bias_stride);
  return ok ? (static_cast<int64_t>(L) + kBlock - 1) / kBlock : 0;
}
}  // namespace

extern "C" int pkv_plan_parts(const int32_t *seq_lens, int32_t B, int32_t Hkv, int32_t d,
                              const int32_t *block_tables, int32_t bt_stride,
                              int32_t bias_stride, int32_t num_parts, int32_t *plan) {
  pkv::clear_error();
  PKV_REQUIRE(plan && (B == 0 || (seq_lens && block_tables)), PKV_ERR_INVALID_ARG,
              "NULL pointer");
  PKV_REQUIRE(B >= 0 && Hkv > 0 && bt_stride > 0 && num_parts > 0, PKV_ERR_INVALID_ARG,
              "bad sizes (B %d, Hkv %d, bt_stride %d, num_parts %d)", B, Hkv, bt_stride,
              num_parts);
  PKV_REQUIRE(d == 64 || d == 128, PKV_ERR_UNSUPPORTED, "head_dim %d", d);
  const int64_t A = pkv::seg_cost(d);
  const int64_t C = num_parts;
  // positions per KV head before each row (prefix sums of n_b + A)
  std::vector<int64_t> rowoff(static_cast<size_t>(B) + 1, 0);
  for (int32_t b = 0; b < B; ++b) {
    const int64_t n = row_pages(seq_lens[b], bt_stride, bias_stride);
    rowoff[b + 1] = rowoff[b] + (n > 0 ? n + A : 0);
  }
  const int64_t P = rowoff[B] * Hkv;
  PKV_REQUIRE(rowoff[B] < (int64_t(1) << 31), PKV_ERR_UNSUPPORTED, "too many positions");
  int32_t b = 0;   // the part starts advance monotonically: one walk over the rows
  for (int64_t c = 0; c < C; ++c) {
    int32_t *r = plan + c * PKV_PLAN_INTS;
    for (int i = 0; i < PKV_PLAN_INTS; ++i) r[i] = (i >= 8) ? -1 : 0;
    r[0] = -1;
    r[4] = static_cast<int32_t>(static_cast<uint64_t>(P) & 0xffffffffu);
    r[5] = static_cast<int32_t>(static_cast<uint64_t>(P) >> 32);
    const int64_t start = P * c / C, end = P * (c + 1) / C;
    if (start >= end) continue;
    while (b < B && start >= rowoff[b + 1] * Hkv) ++b;   // the row whose positions hold start
    if (b >= B) continue;                               // (not reached: start < P)
    const int64_t n = rowoff[b + 1] - rowoff[b] - A;     // pages of row b (> 0)
    r[0] = b;
    r[1] = static_cast<int32_t>(rowoff[b]);
    r[2] = seq_lens[b];
    r[3] = b + 1 < B ? seq_lens[b + 1] : 0;
    const int64_t g = (start - rowoff[b] * Hkv) / (n + A);   // KV head of the first unit
    const int64_t off = rowoff[b] * Hkv + g * (n + A);       // its first position
    const int64_t j0 = start - off - A > 0 ? start - off - A : 0;
    const int64_t j1 = end - off - A < n ? end - off - A : n;
    const int32_t *table = block_tables + static_cast<int64_t>(b) * bt_stride;
    for (int64_t i = 0; i < 32 && j0 + i < j1; ++i) r[8 + i] = table[j0 + i];
  }
  return PKV_OK;
}
