// Host block allocator for the paged KV cache.
//
// "neurogrid releases" v0.7.0, Paged KV Cache: the cache grows in fixed
// 16-token blocks taken on demand, a block allocator hands blocks out and takes
// them back in constant time, and every sequence has its own block table.
// v0.8.0: kv_len = position + 1.  The policy (LIFO free stack,
// smallest free sequence id on join, lazy block at position % 16 == 0, atomic
// failure) is stated in pkv.h.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <new>
#include <queue>
#include <vector>

#include "status.h"

struct pkv_alloc {
  int32_t num_blocks = 0;
  int32_t max_seqs = 0;
  int32_t max_blocks_per_seq = 0;
  std::vector<int32_t> free_stack;       // bottom .. top; capacity num_blocks
  std::vector<int32_t> tables;           // [max_seqs * max_blocks_per_seq]
  std::vector<int32_t> n_blocks;         // per sequence id
  std::vector<int32_t> lengths;          // per sequence id
  std::vector<uint8_t> live;             // per sequence id
  std::vector<uint32_t> stamp;           // per sequence id, duplicate detection
  std::vector<int32_t> generation;       // per sequence id, joins so far (ids are reused)
  uint32_t epoch = 0;
  std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_ids;

  int32_t *table(int32_t sid) {
    return tables.data() + static_cast<size_t>(sid) * static_cast<size_t>(max_blocks_per_seq);
  }
  const int32_t *table(int32_t sid) const {
    return tables.data() + static_cast<size_t>(sid) * static_cast<size_t>(max_blocks_per_seq);
  }
  bool is_live(int32_t sid) const { return sid >= 0 && sid < max_seqs && live[sid]; }
};

namespace {
constexpr int32_t kBlock = PKV_BLOCK_SIZE;
inline int64_t blocks_for(int64_t tokens) { return (tokens + kBlock - 1) / kBlock; }
}  // namespace

extern "C" int pkv_alloc_create(int32_t num_blocks, int32_t block_size, int32_t max_seqs,
                                int32_t max_blocks_per_seq, const int32_t *initial_free,
                                pkv_alloc **out) {
  pkv::clear_error();
  PKV_REQUIRE(out, PKV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  PKV_REQUIRE(block_size == kBlock, PKV_ERR_UNSUPPORTED, "block_size must be %d", kBlock);
  PKV_REQUIRE(num_blocks > 0 && max_seqs > 0 && max_blocks_per_seq > 0, PKV_ERR_INVALID_ARG,
              "num_blocks, max_seqs and max_blocks_per_seq must be positive");
  PKV_REQUIRE(static_cast<int64_t>(max_seqs) * max_blocks_per_seq <= (int64_t(1) << 31),
              PKV_ERR_INVALID_ARG, "max_seqs * max_blocks_per_seq too large");
  pkv_alloc *a = new (std::nothrow) pkv_alloc();
  PKV_REQUIRE(a, PKV_ERR_INVALID_ARG, "out of host memory");
  try {
    a->num_blocks = num_blocks;
    a->max_seqs = max_seqs;
    a->max_blocks_per_seq = max_blocks_per_seq;
    a->free_stack.resize(num_blocks);
    if (initial_free) {
      std::vector<uint8_t> seen(num_blocks, 0);
      for (int32_t i = 0; i < num_blocks; ++i) {
        int32_t b = initial_free[i];
        if (b < 0 || b >= num_blocks || seen[b]) {
          delete a;
          return pkv::fail(PKV_ERR_INVALID_ARG,
                           "initial_free is not a permutation of 0..%d (entry %d = %d)",
                           num_blocks - 1, i, b);
        }
        seen[b] = 1;
        a->free_stack[i] = b;
      }
    } else {
      for (int32_t i = 0; i < num_blocks; ++i) a->free_stack[i] = i;
    }
    a->tables.assign(static_cast<size_t>(max_seqs) * max_blocks_per_seq, -1);
    a->n_blocks.assign(max_seqs, 0);
    a->lengths.assign(max_seqs, 0);
    a->live.assign(max_seqs, 0);
    a->stamp.assign(max_seqs, 0);
    a->generation.assign(max_seqs, 0);
    for (int32_t i = 0; i < max_seqs; ++i) a->free_ids.push(i);
  } catch (...) {
    delete a;
    return pkv::fail(PKV_ERR_INVALID_ARG, "out of host memory");
  }
  *out = a;
  return PKV_OK;
}

extern "C" void pkv_alloc_destroy(pkv_alloc *a) { delete a; }

extern "C" int pkv_seq_join(pkv_alloc *a, int32_t prefix_len, int32_t *seq_id) {
  pkv::clear_error();
  PKV_REQUIRE(a && seq_id, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(prefix_len >= 0, PKV_ERR_INVALID_ARG, "prefix_len < 0");
  PKV_REQUIRE(!a->free_ids.empty(), PKV_ERR_INVALID_ARG, "all %d sequence ids are live",
              a->max_seqs);
  const int64_t need = blocks_for(prefix_len);
  PKV_REQUIRE(need <= a->max_blocks_per_seq, PKV_ERR_INVALID_ARG,
              "prefix of %d tokens needs %lld blocks > max_blocks_per_seq %d", prefix_len,
              (long long)need, a->max_blocks_per_seq);
  PKV_REQUIRE(need <= static_cast<int64_t>(a->free_stack.size()), PKV_ERR_OUT_OF_BLOCKS,
              "join needs %lld blocks, %zu free", (long long)need, a->free_stack.size());
  const int32_t sid = a->free_ids.top();
  a->free_ids.pop();
  int32_t *t = a->table(sid);
  for (int64_t j = 0; j < need; ++j) {
    t[j] = a->free_stack.back();
    a->free_stack.pop_back();
  }
  a->n_blocks[sid] = static_cast<int32_t>(need);
  a->lengths[sid] = prefix_len;
  a->live[sid] = 1;
  ++a->generation[sid];
  *seq_id = sid;
  return PKV_OK;
}

extern "C" int pkv_seq_leave(pkv_alloc *a, int32_t seq_id) {
  pkv::clear_error();
  PKV_REQUIRE(a, PKV_ERR_INVALID_ARG, "NULL allocator");
  PKV_REQUIRE(a->is_live(seq_id), PKV_ERR_UNKNOWN_SEQ, "sequence %d is not live", seq_id);
  const int32_t *t = a->table(seq_id);
  for (int32_t j = 0; j < a->n_blocks[seq_id]; ++j) a->free_stack.push_back(t[j]);
  a->n_blocks[seq_id] = 0;
  a->lengths[seq_id] = 0;
  a->live[seq_id] = 0;
  a->free_ids.push(seq_id);
  return PKV_OK;
}

namespace {

// a0 for one step (pkv_prepare_step).  With row_state, block_tables is a
// buffer an earlier call wrote with the same row_state, and only the entries
// that differ from what it holds are written.
int prepare_step_impl(pkv_alloc *a, const int32_t *seq_ids, int32_t B, int32_t *positions,
                      int64_t *slot_mapping, int32_t *seq_lens, int32_t *block_tables,
                      int32_t bt_stride, int32_t *row_state) {
  PKV_REQUIRE(a, PKV_ERR_INVALID_ARG, "NULL allocator");
  PKV_REQUIRE(B >= 0, PKV_ERR_INVALID_ARG, "B < 0");
  if (B == 0) return PKV_OK;
  PKV_REQUIRE(seq_ids && positions && slot_mapping && seq_lens && block_tables,
              PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(bt_stride > 0, PKV_ERR_INVALID_ARG, "bt_stride must be positive");
  // Validate everything before changing any state.
  if (++a->epoch == 0) {
    std::fill(a->stamp.begin(), a->stamp.end(), 0u);
    a->epoch = 1;
  }
  int64_t need = 0;
  const int32_t width = bt_stride < a->max_blocks_per_seq ? bt_stride : a->max_blocks_per_seq;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t s = seq_ids[b];
    PKV_REQUIRE(a->is_live(s), PKV_ERR_UNKNOWN_SEQ, "row %d: sequence %d is not live", b, s);
    PKV_REQUIRE(a->stamp[s] != a->epoch, PKV_ERR_INVALID_ARG,
                "sequence %d listed twice in one step", s);
    a->stamp[s] = a->epoch;
    const int64_t len = a->lengths[s];
    PKV_REQUIRE(blocks_for(len + 1) <= width, PKV_ERR_INVALID_ARG,
                "sequence %d would need %lld blocks > %d", s, (long long)blocks_for(len + 1),
                width);
    if (len % kBlock == 0) ++need;
  }
  PKV_REQUIRE(need <= static_cast<int64_t>(a->free_stack.size()), PKV_ERR_OUT_OF_BLOCKS,
              "step needs %lld new blocks, %zu free", (long long)need, a->free_stack.size());
  for (int32_t b = 0; b < B; ++b) {
    const int32_t s = seq_ids[b];
    const int32_t pos = a->lengths[s];
    int32_t *t = a->table(s);
    if (pos % kBlock == 0) {
      t[a->n_blocks[s]++] = a->free_stack.back();
      a->free_stack.pop_back();
    }
    positions[b] = pos;
    slot_mapping[b] = static_cast<int64_t>(t[pos / kBlock]) * kBlock + pos % kBlock;
    a->lengths[s] = pos + 1;
    seq_lens[b] = pos + 1;
    int32_t *row = block_tables + static_cast<size_t>(b) * bt_stride;
    const int32_t n = a->n_blocks[s];
    if (!row_state) {
      std::memcpy(row, t, sizeof(int32_t) * n);
      for (int32_t j = n; j < bt_stride; ++j) row[j] = -1;
      continue;
    }
    // row_state[3b..3b+2]: sequence id, its join generation, entries held
    int32_t *rs = row_state + 3 * static_cast<size_t>(b);
    const bool same = rs[0] == s && rs[1] == a->generation[s] && rs[2] >= 0 && rs[2] <= n;
    if (same) {
      // the same sequence as last time in this buffer: its table only grew
      std::memcpy(row + rs[2], t + rs[2], sizeof(int32_t) * (n - rs[2]));
    } else {
      std::memcpy(row, t, sizeof(int32_t) * n);
      const int32_t held = (rs[2] >= 0 && rs[2] <= bt_stride && rs[0] >= 0) ? rs[2] : bt_stride;
      for (int32_t j = n; j < held; ++j) row[j] = -1;
    }
    rs[0] = s;
    rs[1] = a->generation[s];
    rs[2] = n;
  }
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_prepare_step(pkv_alloc *a, const int32_t *seq_ids, int32_t B,
                                int32_t *positions, int64_t *slot_mapping,
                                int32_t *seq_lens, int32_t *block_tables,
                                int32_t bt_stride) {
  pkv::clear_error();
  return prepare_step_impl(a, seq_ids, B, positions, slot_mapping, seq_lens, block_tables,
                           bt_stride, nullptr);
}

extern "C" int pkv_prepare_step_cached(pkv_alloc *a, const int32_t *seq_ids, int32_t B,
                                       int32_t *positions, int64_t *slot_mapping,
                                       int32_t *seq_lens, int32_t *block_tables,
                                       int32_t bt_stride, int32_t *row_state) {
  pkv::clear_error();
  PKV_REQUIRE(row_state, PKV_ERR_INVALID_ARG, "NULL row_state");
  return prepare_step_impl(a, seq_ids, B, positions, slot_mapping, seq_lens, block_tables,
                           bt_stride, row_state);
}

extern "C" int pkv_seqs_join(pkv_alloc *a, const int32_t *prefix_lens, int32_t n,
                             int32_t *seq_ids, int32_t *positions, int64_t *slot_mapping) {
  pkv::clear_error();
  PKV_REQUIRE(a && n >= 0, PKV_ERR_INVALID_ARG, "NULL allocator or n < 0");
  if (n == 0) return PKV_OK;
  PKV_REQUIRE(prefix_lens && seq_ids, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(!positions == !slot_mapping, PKV_ERR_INVALID_ARG,
              "give both positions and slot_mapping, or neither");
  // validate the whole batch before changing anything
  PKV_REQUIRE(static_cast<size_t>(n) <= a->free_ids.size(), PKV_ERR_INVALID_ARG,
              "%d joins but only %zu free sequence ids", n, a->free_ids.size());
  int64_t need = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t L = prefix_lens[i];
    PKV_REQUIRE(L >= 0, PKV_ERR_INVALID_ARG, "joiner %d: prefix_len %d < 0", i, L);
    PKV_REQUIRE(blocks_for(L) <= a->max_blocks_per_seq, PKV_ERR_INVALID_ARG,
                "joiner %d: prefix of %d tokens needs %lld blocks > max_blocks_per_seq %d", i,
                L, (long long)blocks_for(L), a->max_blocks_per_seq);
    need += blocks_for(L);
  }
  PKV_REQUIRE(need <= static_cast<int64_t>(a->free_stack.size()), PKV_ERR_OUT_OF_BLOCKS,
              "joins need %lld blocks, %zu free", (long long)need, a->free_stack.size());
  int64_t k = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int rc = pkv_seq_join(a, prefix_lens[i], &seq_ids[i]);   // cannot fail now
    if (rc != PKV_OK) return rc;
    if (!positions) continue;
    const int32_t *t = a->table(seq_ids[i]);
    for (int32_t p = 0; p < prefix_lens[i]; ++p, ++k) {
      positions[k] = p;
      slot_mapping[k] = static_cast<int64_t>(t[p / kBlock]) * kBlock + p % kBlock;
    }
  }
  return PKV_OK;
}

extern "C" int pkv_seqs_leave(pkv_alloc *a, const int32_t *seq_ids, int32_t n) {
  pkv::clear_error();
  PKV_REQUIRE(a && n >= 0, PKV_ERR_INVALID_ARG, "NULL allocator or n < 0");
  if (n == 0) return PKV_OK;
  PKV_REQUIRE(seq_ids, PKV_ERR_INVALID_ARG, "NULL seq_ids");
  if (++a->epoch == 0) {
    std::fill(a->stamp.begin(), a->stamp.end(), 0u);
    a->epoch = 1;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = seq_ids[i];
    PKV_REQUIRE(a->is_live(s), PKV_ERR_UNKNOWN_SEQ, "sequence %d is not live", s);
    PKV_REQUIRE(a->stamp[s] != a->epoch, PKV_ERR_INVALID_ARG, "sequence %d listed twice", s);
    a->stamp[s] = a->epoch;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int rc = pkv_seq_leave(a, seq_ids[i]);
    if (rc != PKV_OK) return rc;
  }
  return PKV_OK;
}

extern "C" int pkv_seq_len(const pkv_alloc *a, int32_t seq_id, int32_t *len) {
  pkv::clear_error();
  PKV_REQUIRE(a && len, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->is_live(seq_id), PKV_ERR_UNKNOWN_SEQ, "sequence %d is not live", seq_id);
  *len = a->lengths[seq_id];
  return PKV_OK;
}

extern "C" int pkv_seq_blocks(const pkv_alloc *a, int32_t seq_id, int32_t *out, int32_t cap,
                              int32_t *n) {
  pkv::clear_error();
  PKV_REQUIRE(a && n, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(a->is_live(seq_id), PKV_ERR_UNKNOWN_SEQ, "sequence %d is not live", seq_id);
  const int32_t nb = a->n_blocks[seq_id];
  *n = nb;
  if (out) {
    const int32_t *t = a->table(seq_id);
    for (int32_t j = 0; j < nb && j < cap; ++j) out[j] = t[j];
  }
  return PKV_OK;
}

extern "C" int pkv_seq_slots(const pkv_alloc *a, int32_t seq_id, int32_t start, int32_t count,
                             int32_t *positions, int64_t *slot_mapping) {
  pkv::clear_error();
  PKV_REQUIRE(a, PKV_ERR_INVALID_ARG, "NULL allocator");
  PKV_REQUIRE(a->is_live(seq_id), PKV_ERR_UNKNOWN_SEQ, "sequence %d is not live", seq_id);
  PKV_REQUIRE(start >= 0 && count >= 0, PKV_ERR_INVALID_ARG, "negative start or count");
  const int32_t len = a->lengths[seq_id];
  PKV_REQUIRE(static_cast<int64_t>(start) + count <= len, PKV_ERR_INVALID_ARG,
              "tokens [%d, %d) exceed the sequence length %d", start, start + count, len);
  if (count == 0) return PKV_OK;
  PKV_REQUIRE(positions && slot_mapping, PKV_ERR_INVALID_ARG, "NULL output");
  const int32_t *t = a->table(seq_id);
  for (int32_t i = 0; i < count; ++i) {
    const int32_t p = start + i;
    positions[i] = p;
    slot_mapping[i] = static_cast<int64_t>(t[p / kBlock]) * kBlock + p % kBlock;
  }
  return PKV_OK;
}

extern "C" int pkv_pool_blocks(uint64_t budget_bytes, int32_t n_layers, int32_t Hkv, int32_t d,
                               int32_t dtype, int32_t *num_blocks) {
  pkv::clear_error();
  PKV_REQUIRE(num_blocks, PKV_ERR_INVALID_ARG, "NULL output");
  PKV_REQUIRE(n_layers > 0 && Hkv > 0 && d > 0, PKV_ERR_INVALID_ARG, "non-positive size");
  PKV_REQUIRE(dtype == PKV_F32 || dtype == PKV_BF16, PKV_ERR_UNSUPPORTED, "dtype %d", dtype);
  // one block = 16 tokens of K and of V, all KV heads, every layer
  const uint64_t per_block = static_cast<uint64_t>(n_layers) * 2u * static_cast<uint64_t>(Hkv) *
                             kBlock * static_cast<uint64_t>(d) * (dtype == PKV_BF16 ? 2u : 4u);
  const uint64_t n = budget_bytes / per_block;
  *num_blocks = n > static_cast<uint64_t>(INT32_MAX) ? INT32_MAX : static_cast<int32_t>(n);
  return PKV_OK;
}

extern "C" int pkv_num_free(const pkv_alloc *a, int32_t *n) {
  pkv::clear_error();
  PKV_REQUIRE(a && n, PKV_ERR_INVALID_ARG, "NULL argument");
  *n = static_cast<int32_t>(a->free_stack.size());
  return PKV_OK;
}

extern "C" int pkv_alloc_dump(const pkv_alloc *a, int32_t *free_stack, int32_t cap,
                              int32_t *n) {
  pkv::clear_error();
  PKV_REQUIRE(a && n, PKV_ERR_INVALID_ARG, "NULL argument");
  const int32_t sz = static_cast<int32_t>(a->free_stack.size());
  *n = sz;
  if (free_stack)
    for (int32_t i = 0; i < sz && i < cap; ++i) free_stack[i] = a->free_stack[i];
  return PKV_OK;
}
