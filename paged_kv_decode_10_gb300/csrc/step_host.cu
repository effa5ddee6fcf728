// The decode step from host buffers (pkv_decode_step_host) and its captured
// form (pkv_step_graph_*): the inputs staged to the device by copies, or read
// in place over the CPU-GPU link through their mapped addresses, then the
// step's kernels (pkv_decode_step), then the output copied back or written in
// place.  Host code only: the kernels are the attention and RoPE/append ones.
#include <cuda_runtime.h>

#include <mutex>
#include <new>

#include "attention_host.h"
#include "common.cuh"

using namespace pkv;

namespace {

// Device addresses of page-locked host buffers, remembered per (device, host
// pointer): a step from host buffers looks up the same buffers every time.
int mapped_address(const void *host, void **dev_ptr) {
  struct Entry {
    const void *host;
    void *dev;
    int device;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int used = 0, next = 0;
  int device = 0;
  PKV_CUDA_CHECK(cudaGetDevice(&device));
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
      if (cache[i].host == host && cache[i].device == device) {
        *dev_ptr = cache[i].dev;
        return PKV_OK;
      }
  }
  PKV_CUDA_CHECK(cudaHostGetDevicePointer(dev_ptr, const_cast<void *>(host), 0));
  std::lock_guard<std::mutex> lock(mu);
  const int slot = used < 32 ? used++ : (next++ % 32);
  cache[slot] = Entry{host, *dev_ptr, device};
  return PKV_OK;
}

// Everything pkv_decode_step_host does except the final wait: the inputs
// copied to the device, the step and the output copied back; or, in place, the
// step's kernels pointed at the mapped addresses of the host inputs and of the
// host output.
int enqueue_host_step(const pkv_step_args *dev, const pkv_step_host_io *host, cudaStream_t s) {
  PKV_REQUIRE(dev && host, PKV_ERR_INVALID_ARG, "NULL argument");
  PKV_REQUIRE(host->q && host->k && host->v && host->positions && host->slot_mapping &&
                  host->seq_lens && host->block_tables && host->out,
              PKV_ERR_INVALID_ARG, "NULL host buffer");
  const int rc0 = check_shapes(dev->B, dev->Hq, dev->Hkv, dev->d, dev->dtype);
  if (rc0 != PKV_OK) return rc0;
  const size_t el = dtype_size(dev->dtype);
  const size_t B = static_cast<size_t>(dev->B);
  const size_t qb = B * dev->Hq * dev->d * el, kb = B * dev->Hkv * dev->d * el;
  if (host->flags & PKV_HOST_IN_PLACE) {
    // inputs read and the result written in place over the CPU-GPU link
    pkv_step_args a = *dev;
    void *m[9] = {};
    const void *h[9] = {host->q, host->k, host->v, host->positions, host->slot_mapping,
                        host->seq_lens, host->block_tables, host->out, host->plan};
    for (int i = 0; i < 9; ++i) {
      if (!h[i]) continue;   // (only the plan is optional)
      const int rc = mapped_address(h[i], &m[i]);
      if (rc != PKV_OK) return rc;
    }
    a.plan = static_cast<const int32_t *>(m[8]);
    a.q = m[0];
    a.k = m[1];
    a.v = m[2];
    a.positions = static_cast<const int32_t *>(m[3]);
    a.slot_mapping = static_cast<const int64_t *>(m[4]);
    a.seq_lens = static_cast<const int32_t *>(m[5]);
    a.block_tables = static_cast<const int32_t *>(m[6]);
    a.out = m[7];
    return pkv_decode_step(&a, s);
  }
  PKV_CUDA_CHECK(cudaMemcpyAsync(const_cast<void *>(dev->q), host->q, qb, cudaMemcpyHostToDevice, s));
  PKV_CUDA_CHECK(cudaMemcpyAsync(const_cast<void *>(dev->k), host->k, kb, cudaMemcpyHostToDevice, s));
  PKV_CUDA_CHECK(cudaMemcpyAsync(const_cast<void *>(dev->v), host->v, kb, cudaMemcpyHostToDevice, s));
  PKV_CUDA_CHECK(cudaMemcpyAsync(const_cast<int32_t *>(dev->positions), host->positions,
                                 B * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  PKV_CUDA_CHECK(cudaMemcpyAsync(const_cast<int64_t *>(dev->slot_mapping), host->slot_mapping,
                                 B * sizeof(int64_t), cudaMemcpyHostToDevice, s));
  PKV_CUDA_CHECK(cudaMemcpyAsync(const_cast<int32_t *>(dev->seq_lens), host->seq_lens,
                                 B * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  PKV_CUDA_CHECK(cudaMemcpyAsync(const_cast<int32_t *>(dev->block_tables), host->block_tables,
                                 B * dev->bt_stride * sizeof(int32_t), cudaMemcpyHostToDevice, s));
  pkv_step_args a = *dev;
  if (host->plan) {
    PKV_REQUIRE(dev->plan && dev->num_parts > 0, PKV_ERR_INVALID_ARG,
                "a host plan needs dev->plan (device buffer) and dev->num_parts");
    PKV_CUDA_CHECK(cudaMemcpyAsync(const_cast<int32_t *>(dev->plan), host->plan,
                                   static_cast<size_t>(dev->num_parts) * PKV_PLAN_INTS *
                                       sizeof(int32_t),
                                   cudaMemcpyHostToDevice, s));
  } else {
    a.plan = nullptr;
  }
  const int rc = pkv_decode_step(&a, s);
  if (rc != PKV_OK) return rc;
  PKV_CUDA_CHECK(cudaMemcpyAsync(host->out, dev->out, qb, cudaMemcpyDeviceToHost, s));
  return PKV_OK;
}

}  // namespace

extern "C" int pkv_decode_step_host(const pkv_step_args *dev, const pkv_step_host_io *host,
                                    void *stream) {
  clear_error();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rc = enqueue_host_step(dev, host, s);
  if (rc != PKV_OK) return rc;
  PKV_CUDA_CHECK(cudaStreamSynchronize(s));
  return PKV_OK;
}

struct pkv_step_graph {
  cudaGraphExec_t exec;
  cudaEvent_t done;   // recorded after every pkv_step_graph_enqueue
};

extern "C" int pkv_step_graph_create(const pkv_step_args *dev, const pkv_step_host_io *host,
                                     pkv_step_graph **out) {
  clear_error();
  PKV_REQUIRE(dev && host && out, PKV_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  // resolve what the step would look up on its first call, outside the capture
  pkv_step_args a = *dev;
  if (a.num_parts <= 0 && a.B > 0) {
    int rc = check_shapes(a.B, a.Hq, a.Hkv, a.d, a.dtype);
    if (rc != PKV_OK) return rc;
    rc = default_parts(a.d, a.dtype, a.flags, a.Hq / a.Hkv, &a.num_parts);
    if (rc != PKV_OK) return rc;
  }
  cudaStream_t cs;
  PKV_CUDA_CHECK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
  cudaGraph_t graph = nullptr;
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal);
  int rc = PKV_OK;
  if (e == cudaSuccess) {
    rc = enqueue_host_step(&a, host, cs);
    const cudaError_t e2 = cudaStreamEndCapture(cs, &graph);   // ends the capture either way
    if (rc == PKV_OK && e2 != cudaSuccess) e = e2;
  }
  cudaStreamDestroy(cs);
  if (rc != PKV_OK) {
    if (graph) cudaGraphDestroy(graph);
    return rc;
  }
  PKV_REQUIRE(e == cudaSuccess, PKV_ERR_CUDA, "step capture failed: %s", cudaGetErrorString(e));
  cudaGraphExec_t exec = nullptr;
  e = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  PKV_REQUIRE(e == cudaSuccess, PKV_ERR_CUDA, "graph instantiation failed: %s",
              cudaGetErrorString(e));
  cudaEvent_t done = nullptr;
  e = cudaEventCreateWithFlags(&done, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    cudaGraphExecDestroy(exec);
    return fail(PKV_ERR_CUDA, "event creation failed: %s", cudaGetErrorString(e));
  }
  pkv_step_graph *g = new (std::nothrow) pkv_step_graph{exec, done};
  if (!g) {
    cudaEventDestroy(done);
    cudaGraphExecDestroy(exec);
    return fail(PKV_ERR_CUDA, "out of host memory");
  }
  *out = g;
  return PKV_OK;
}

extern "C" int pkv_step_graph_launch(pkv_step_graph *g, void *stream) {
  clear_error();
  PKV_REQUIRE(g, PKV_ERR_INVALID_ARG, "NULL graph");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PKV_CUDA_CHECK(cudaGraphLaunch(g->exec, s));
  PKV_CUDA_CHECK(cudaStreamSynchronize(s));
  return PKV_OK;
}

extern "C" int pkv_step_graph_enqueue(pkv_step_graph *g, void *stream) {
  clear_error();
  PKV_REQUIRE(g, PKV_ERR_INVALID_ARG, "NULL graph");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PKV_CUDA_CHECK(cudaGraphLaunch(g->exec, s));
  PKV_CUDA_CHECK(cudaEventRecord(g->done, s));
  return PKV_OK;
}

extern "C" int pkv_step_graph_wait(pkv_step_graph *g) {
  clear_error();
  PKV_REQUIRE(g, PKV_ERR_INVALID_ARG, "NULL graph");
  PKV_CUDA_CHECK(cudaEventSynchronize(g->done));
  return PKV_OK;
}

extern "C" void pkv_step_graph_destroy(pkv_step_graph *g) {
  if (!g) return;
  cudaEventDestroy(g->done);
  cudaGraphExecDestroy(g->exec);
  delete g;
}
