// Native serving loop (pkv_server): continuous batching with one host call per
// step.
//
// helexa issue 121, slice 3b: the engine admits joiners, prefills them,
// rebatches and decodes every live sequence in lockstep; a sequence that
// leaves frees its row.  "neurogrid releases" v0.7.0: the KV cache is paged,
// so admitting or retiring a sequence only edits block tables (O(1) block
// allocator) and no KV moves; v0.8.0: the decode step is replayed as one CUDA
// graph that reads positions and lengths from buffers the host wrote, with no
// device-to-host copy.  Here a joiner takes over the row of a sequence that
// left, so the batch keeps B rows and two captured graphs (one per pinned
// metadata buffer, used alternately) serve every step.  The server allocates
// no device memory: every buffer is the caller's.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "attention_host.h"
#include "status.h"

namespace {

size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// Packed metadata of one step: slot_mapping int64 [B], positions int32 [B],
// seq_lens int32 [B], block tables int32 [B, bt_stride] (16-byte aligned),
// plan int32 [num_parts, PKV_PLAN_INTS] (16-byte aligned).
struct MetaLayout {
  size_t slots, pos, lens, tables, plan, bytes;
  MetaLayout(int32_t B, int32_t bt, int32_t parts) {
    slots = 0;
    pos = 8 * static_cast<size_t>(B);
    lens = pos + 4 * static_cast<size_t>(B);
    tables = align16(lens + 4 * static_cast<size_t>(B));
    plan = align16(tables + 4 * static_cast<size_t>(B) * bt);
    bytes = plan + 4 * static_cast<size_t>(PKV_PLAN_INTS) * parts;
  }
};

#define SERVER_CUDA(expr)                                                             \
  do {                                                                                \
    cudaError_t _e = (expr);                                                          \
    if (_e != cudaSuccess)                                                            \
      return ::pkv::fail(PKV_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(_e));      \
  } while (0)

}  // namespace

struct pkv_server {
  pkv_step_args step;                 // device buffers; metadata pointers set per graph
  pkv_alloc *alloc = nullptr;
  int32_t B = 0, bt = 0, parts = 0, max_prefix = 0;
  std::vector<int32_t> rows;          // row -> live sequence id
  std::vector<int32_t> row_state[2];  // pkv_prepare_step_cached state per metadata buffer
  unsigned char *meta[2] = {};        // pinned host metadata buffers
  int32_t *pre_pos[2] = {};           // pinned joiner prefix positions
  int64_t *pre_slot[2] = {};          // pinned joiner prefix slots
  void *pre_pos_dev[2] = {}, *pre_slot_dev[2] = {};   // their mapped addresses
  cudaGraphExec_t graph[2] = {};
  cudaEvent_t meta_done[2] = {}, prefix_done[2] = {};
  bool meta_used[2] = {}, prefix_used[2] = {};
  int turn = 0;
  std::vector<int32_t> scratch_ids, new_ids;
  bool broken = false;

  ~pkv_server() {
    for (int t = 0; t < 2; ++t) {
      if (graph[t]) cudaGraphExecDestroy(graph[t]);
      if (meta_done[t]) cudaEventDestroy(meta_done[t]);
      if (prefix_done[t]) cudaEventDestroy(prefix_done[t]);
    }
  }
};

extern "C" size_t pkv_server_meta_bytes(int32_t B, int32_t bt_stride, int32_t num_parts) {
  if (B < 0 || bt_stride < 0 || num_parts < 0) return 0;
  return MetaLayout(B, bt_stride, num_parts).bytes;
}

// Joiner prefix buffer: positions int32 [max], then (16-byte aligned) slots int64 [max].
extern "C" size_t pkv_server_prefix_bytes(int32_t max_prefix_tokens) {
  if (max_prefix_tokens < 0) return 0;
  return align16(4 * static_cast<size_t>(max_prefix_tokens)) +
         8 * static_cast<size_t>(max_prefix_tokens);
}

namespace {

int mapped(void *host, void **dev) {
  SERVER_CUDA(cudaHostGetDevicePointer(dev, host, 0));
  return PKV_OK;
}

int create(const pkv_server_desc *d, pkv_server *s) {
  const pkv_step_args &a = d->step;
  PKV_REQUIRE(d->alloc && d->rows && a.B > 0 && a.num_parts > 0 && a.bt_stride > 0,
              PKV_ERR_INVALID_ARG, "server needs an allocator, rows, B > 0, num_parts > 0");
  PKV_REQUIRE(!a.attn_bias, PKV_ERR_UNSUPPORTED, "the server decodes without a bias");
  PKV_REQUIRE(d->max_prefix_tokens >= 0, PKV_ERR_INVALID_ARG, "max_prefix_tokens < 0");
  for (int t = 0; t < 2; ++t)
    PKV_REQUIRE(d->meta_host[t] && (d->max_prefix_tokens == 0 || d->prefix_host[t]),
                PKV_ERR_INVALID_ARG, "NULL host buffer");
  s->step = a;
  s->alloc = d->alloc;
  s->B = a.B;
  s->bt = a.bt_stride;
  s->parts = a.num_parts;
  s->max_prefix = d->max_prefix_tokens;
  s->rows.assign(d->rows, d->rows + a.B);
  s->scratch_ids.resize(a.B);
  s->new_ids.resize(a.B);
  const MetaLayout L(s->B, s->bt, s->parts);
  for (int t = 0; t < 2; ++t) {
    s->row_state[t].assign(3 * static_cast<size_t>(s->B), -1);
    s->meta[t] = static_cast<unsigned char *>(d->meta_host[t]);
    PKV_REQUIRE((reinterpret_cast<uintptr_t>(s->meta[t]) & 15) == 0, PKV_ERR_INVALID_ARG,
                "meta_host must be 16-byte aligned");
    if (s->max_prefix > 0) {
      s->pre_pos[t] = static_cast<int32_t *>(d->prefix_host[t]);
      s->pre_slot[t] = reinterpret_cast<int64_t *>(static_cast<unsigned char *>(d->prefix_host[t]) +
                                                   align16(4 * static_cast<size_t>(s->max_prefix)));
      int rc = mapped(s->pre_pos[t], &s->pre_pos_dev[t]);
      if (rc != PKV_OK) return rc;
      rc = mapped(s->pre_slot[t], &s->pre_slot_dev[t]);
      if (rc != PKV_OK) return rc;
    }
    SERVER_CUDA(cudaEventCreateWithFlags(&s->meta_done[t], cudaEventDisableTiming));
    SERVER_CUDA(cudaEventCreateWithFlags(&s->prefix_done[t], cudaEventDisableTiming));
  }
  // one graph per metadata buffer: the step's kernels read that buffer in place
  cudaStream_t cs;
  SERVER_CUDA(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
  int rc = PKV_OK;
  for (int t = 0; t < 2 && rc == PKV_OK; ++t) {
    void *dev = nullptr;
    rc = mapped(s->meta[t], &dev);
    if (rc != PKV_OK) break;
    unsigned char *m = static_cast<unsigned char *>(dev);
    pkv_step_args g = s->step;
    g.slot_mapping = reinterpret_cast<const int64_t *>(m + L.slots);
    g.positions = reinterpret_cast<const int32_t *>(m + L.pos);
    g.seq_lens = reinterpret_cast<const int32_t *>(m + L.lens);
    g.block_tables = reinterpret_cast<const int32_t *>(m + L.tables);
    g.plan = reinterpret_cast<const int32_t *>(m + L.plan);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
      rc = pkv::fail(PKV_ERR_CUDA, "begin capture: %s", cudaGetErrorString(e));
      break;
    }
    rc = pkv_decode_step(&g, cs);
    const cudaError_t e2 = cudaStreamEndCapture(cs, &graph);   // ends the capture either way
    if (rc == PKV_OK && e2 != cudaSuccess)
      rc = pkv::fail(PKV_ERR_CUDA, "step capture: %s", cudaGetErrorString(e2));
    if (rc == PKV_OK) {
      e = cudaGraphInstantiate(&s->graph[t], graph, 0);
      if (e != cudaSuccess) rc = pkv::fail(PKV_ERR_CUDA, "instantiate: %s", cudaGetErrorString(e));
    }
    if (graph) cudaGraphDestroy(graph);
  }
  cudaStreamDestroy(cs);
  return rc;
}

}  // namespace

extern "C" int pkv_server_create(const pkv_server_desc *desc, pkv_server **out) {
  pkv::clear_error();
  PKV_REQUIRE(desc && out, PKV_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  pkv_server *s = new (std::nothrow) pkv_server();
  PKV_REQUIRE(s, PKV_ERR_INVALID_ARG, "out of host memory");
  int rc;
  try {
    rc = create(desc, s);
  } catch (...) {
    rc = pkv::fail(PKV_ERR_INVALID_ARG, "out of host memory");
  }
  if (rc != PKV_OK) {
    delete s;
    return rc;
  }
  *out = s;
  return PKV_OK;
}

extern "C" int pkv_server_step(pkv_server *s, const int32_t *leave_rows,
                               const int32_t *prefix_lens, int32_t n, const void *prefix_k,
                               const void *prefix_v, const void *q, const void *k, const void *v,
                               void *stream) {
  pkv::clear_error();
  PKV_REQUIRE(s, PKV_ERR_INVALID_ARG, "NULL server");
  PKV_REQUIRE(!s->broken, PKV_ERR_INVALID_ARG, "an earlier step failed part way: rebuild the server");
  PKV_REQUIRE(n >= 0 && n <= s->B && (n == 0 || (leave_rows && prefix_lens)), PKV_ERR_INVALID_ARG,
              "bad leave/join lists");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const pkv_step_args &a = s->step;
  const int t = s->turn;
  const size_t el = a.dtype == PKV_BF16 ? 2 : 4;
  if (n > 0) {
    // ---- rebatch: the leaving rows' sequences retire, joiners take the rows
    int64_t total = 0;
    for (int32_t i = 0; i < n; ++i) {
      const int32_t r = leave_rows[i];
      PKV_REQUIRE(r >= 0 && r < s->B, PKV_ERR_INVALID_ARG, "leave row %d out of range", r);
      PKV_REQUIRE(prefix_lens[i] >= 0, PKV_ERR_INVALID_ARG, "prefix_lens[%d] < 0", i);
      s->scratch_ids[i] = s->rows[r];
      total += prefix_lens[i];
    }
    PKV_REQUIRE(total <= s->max_prefix, PKV_ERR_INVALID_ARG,
                "joiners bring %lld prefix tokens > max_prefix_tokens %d", (long long)total,
                s->max_prefix);
    PKV_REQUIRE(total == 0 || (prefix_k && prefix_v), PKV_ERR_INVALID_ARG, "NULL prefix K/V");
    int rc = pkv_seqs_leave(s->alloc, s->scratch_ids.data(), n);   // checks distinct, live
    if (rc != PKV_OK) return rc;
    // the prefill two steps back read this prefix buffer
    if (s->prefix_used[t]) SERVER_CUDA(cudaEventSynchronize(s->prefix_done[t]));
    rc = pkv_seqs_join(s->alloc, prefix_lens, n, s->new_ids.data(),
                       total > 0 ? s->pre_pos[t] : nullptr, total > 0 ? s->pre_slot[t] : nullptr);
    if (rc != PKV_OK) {
      s->broken = true;   // the rows' old sequences are gone
      return rc;
    }
    for (int32_t i = 0; i < n; ++i) s->rows[leave_rows[i]] = s->new_ids[i];
    if (total > 0) {
      rc = pkv_prefill_kv(prefix_k, prefix_v, static_cast<const int32_t *>(s->pre_pos_dev[t]),
                          static_cast<const int64_t *>(s->pre_slot_dev[t]), a.k_cache, a.v_cache,
                          static_cast<int32_t>(total), a.Hkv, a.d, a.num_blocks, a.rope_base,
                          a.dtype, a.dev_err_flag, stream);
      if (rc != PKV_OK) {
        s->broken = true;
        return rc;
      }
      SERVER_CUDA(cudaEventRecord(s->prefix_done[t], st));
      s->prefix_used[t] = true;
    }
  }
  // ---- the step's new tokens into the graph's input buffers
  const size_t qb = static_cast<size_t>(s->B) * a.Hq * a.d * el;
  const size_t kb = static_cast<size_t>(s->B) * a.Hkv * a.d * el;
  if (q && q != a.q)
    SERVER_CUDA(cudaMemcpyAsync(const_cast<void *>(a.q), q, qb, cudaMemcpyDeviceToDevice, st));
  if (k && k != a.k)
    SERVER_CUDA(cudaMemcpyAsync(const_cast<void *>(a.k), k, kb, cudaMemcpyDeviceToDevice, st));
  if (v && v != a.v)
    SERVER_CUDA(cudaMemcpyAsync(const_cast<void *>(a.v), v, kb, cudaMemcpyDeviceToDevice, st));
  // ---- a0 and the plan into this turn's metadata buffer (the graph two
  // steps back read it), then the captured step
  if (s->meta_used[t]) SERVER_CUDA(cudaEventSynchronize(s->meta_done[t]));
  const MetaLayout L(s->B, s->bt, s->parts);
  unsigned char *m = s->meta[t];
  int32_t *lens = reinterpret_cast<int32_t *>(m + L.lens);
  int32_t *tables = reinterpret_cast<int32_t *>(m + L.tables);
  int rc = pkv_prepare_step_cached(s->alloc, s->rows.data(), s->B,
                                   reinterpret_cast<int32_t *>(m + L.pos),
                                   reinterpret_cast<int64_t *>(m + L.slots), lens, tables, s->bt,
                                   s->row_state[t].data());
  if (rc != PKV_OK) {
    if (n > 0) s->broken = true;
    return rc;
  }
  rc = pkv_plan_parts(lens, s->B, a.Hkv, a.d, tables, s->bt, 0, s->parts,
                      reinterpret_cast<int32_t *>(m + L.plan));
  if (rc != PKV_OK) {
    s->broken = true;
    return rc;
  }
  SERVER_CUDA(cudaGraphLaunch(s->graph[t], st));
  SERVER_CUDA(cudaEventRecord(s->meta_done[t], st));
  s->meta_used[t] = true;
  s->turn ^= 1;
  return PKV_OK;
}

extern "C" int pkv_server_rows(const pkv_server *s, int32_t *rows) {
  pkv::clear_error();
  PKV_REQUIRE(s && rows, PKV_ERR_INVALID_ARG, "NULL argument");
  std::memcpy(rows, s->rows.data(), sizeof(int32_t) * s->rows.size());
  return PKV_OK;
}

extern "C" void pkv_server_destroy(pkv_server *s) { delete s; }
