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
#include <cstring>
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
  // One merged walk over the parts and the units, without divisions: part
  // starts floor(P*c/C) advance by P/C plus a carry from the remainders, and
  // the unit cursor (row b, KV head g, first position off) moves forward to the
  // unit holding each start.
  const int64_t q0 = P / C, r0 = P % C;
  int64_t start = 0, rem = 0;
  int32_t b = 0, g = 0;
  while (b < B && rowoff[b + 1] == rowoff[b]) ++b;          // first row with pages
  int64_t off = b < B ? rowoff[b] * Hkv : 0;
  int64_t n = b < B ? rowoff[b + 1] - rowoff[b] - A : 0;     // its pages
  for (int64_t c = 0; c < C; ++c) {
    rem += r0;
    const int64_t end = start + q0 + (rem >= C ? 1 : 0);
    if (rem >= C) rem -= C;
    int32_t *r = plan + c * PKV_PLAN_INTS;
    r[0] = -1;
    r[1] = r[2] = r[3] = r[6] = r[7] = 0;
    r[4] = static_cast<int32_t>(static_cast<uint64_t>(P) & 0xffffffffu);
    r[5] = static_cast<int32_t>(static_cast<uint64_t>(P) >> 32);
    if (start < end) {
      while (start >= off + n + A) {   // the unit holding `start` (start < P: it exists)
        off += n + A;
        if (++g == Hkv) {
          g = 0;
          for (++b; b < B && rowoff[b + 1] == rowoff[b]; ++b) {
          }
          n = rowoff[b + 1] - rowoff[b] - A;
        }
      }
      r[0] = b;
      r[1] = static_cast<int32_t>(rowoff[b]);
      r[2] = seq_lens[b];
      r[3] = b + 1 < B ? seq_lens[b + 1] : 0;
      const int64_t j0 = start - off - A > 0 ? start - off - A : 0;
      const int64_t j1 = end - off - A < n ? end - off - A : n;
      // the ids of the segment's pages; entries past its last page are left as
      // they are (nothing reads them)
      constexpr int kIds = PKV_PLAN_INTS - 8;
      const int64_t m = j1 - j0 < kIds ? j1 - j0 : kIds;
      const int32_t *ids = block_tables + static_cast<int64_t>(b) * bt_stride + j0;
      if (m == kIds) {
        for (int i = 0; i < kIds; ++i) r[8 + i] = ids[i];   // (a fixed-size copy vectorises)
      } else {
        for (int64_t i = 0; i < m; ++i) r[8 + i] = ids[i];
      }
    }
    start = end;
  }
  return PKV_OK;
}
