// kvs_graph.cu -- a whole multi-layer decode step as one CUDA graph.
//
// Source: realizar 0.8.5, src/cuda/executor/layers/reduces.rs and
// batched_forward.rs (graph capture with a thread-local capture mode, the
// capture always ended, the eager path kept for when capture fails), and
// aprender-serve 0.70.2, src/gguf/cuda/forward_qwen35_cuda_graph.rs (module
// doc: one graph launch replays every layer of the step; per-token inputs
// such as the position live at fixed device addresses that the host rewrites
// before each replay, and the K/V row is scattered at the device position).
//
// Here the graph holds one kvs_decode_step per layer -- scatter + split-K
// attention, one kernel each, chained with programmatic dependent launch --
// over caller-owned, fixed device buffers.  A memset node ahead of the first
// layer writes a fresh value into the workspace epoch at every replay
// (kvs_step_graph_launch sets it): the epoch is part of the tag the step
// kernel's completion counters carry, so no replay can take counts left by
// an earlier replay that gave up on a wait for its own, although the tag
// arguments of the captured launches are frozen.

#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "kvs_launch.h"
#include "kvsdecode.h"

struct kvs_step_graph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t epoch_node = nullptr;  // memset of the workspace epoch
  cudaMemsetParams epoch = {};
  std::mutex mu;  // one launch at a time updates the node and launches
  int layers = 0;
};

namespace {

// Puts a memset of the workspace epoch word (4 bytes at the workspace base)
// ahead of every root node of the captured graph.
bool add_epoch_node(cudaGraph_t g, void *workspace, cudaGraphNode_t *node,
                    cudaMemsetParams *params) {
  size_t n = 0;
  if (cudaGraphGetRootNodes(g, nullptr, &n) != cudaSuccess || n == 0) return false;
  std::vector<cudaGraphNode_t> roots(n);
  if (cudaGraphGetRootNodes(g, roots.data(), &n) != cudaSuccess) return false;
  cudaMemsetParams p = {};
  p.dst = workspace;
  p.pitch = 0;
  p.value = kvs::fresh_tag();
  p.elementSize = 4;
  p.width = 1;
  p.height = 1;
  if (cudaGraphAddMemsetNode(node, g, nullptr, 0, &p) != cudaSuccess) return false;
  for (size_t i = 0; i < n; ++i)
    if (cudaGraphAddDependencies(g, node, &roots[i], nullptr, 1) != cudaSuccess) return false;
  *params = p;
  return true;
}

// Captures what `body` enqueues on `s` (thread-local mode, the capture
// always ended), puts the epoch memset ahead of it and instantiates it into
// a new handle.  On any error nothing is kept and the status is returned.
template <class Body>
int capture_step_graph(cudaStream_t s, void *workspace, int layers, Body body,
                       kvs_step_graph **graph) {
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  const int rc = body();
  cudaGraph_t g = nullptr;
  const cudaError_t end = cudaStreamEndCapture(s, &g);  // always end the capture
  if (rc != KVS_OK || end != cudaSuccess || g == nullptr) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return rc != KVS_OK ? rc : KVS_ERR_LAUNCH;
  }
  cudaGraphNode_t epoch_node = nullptr;
  cudaMemsetParams epoch = {};
  if (!add_epoch_node(g, workspace, &epoch_node, &epoch)) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  kvs_step_graph *h = new (std::nothrow) kvs_step_graph;
  if (!h) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(g);
    return KVS_ERR_LAUNCH;
  }
  h->graph = g;
  h->exec = exec;
  h->epoch_node = epoch_node;
  h->epoch = epoch;
  h->layers = layers;
  *graph = h;
  return KVS_OK;
}

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Offsets of kvs_step_graph_io_layout (see the header).
void step_io_offsets(int layers, int M, int H, int Hkv, int D, size_t *off) {
  const size_t qo = (size_t)M * H * D * sizeof(float);
  const size_t kv = (size_t)M * Hkv * D * sizeof(float);
  size_t at = 0;
  for (int l = 0; l < layers; ++l) {
    off[3 * l + 0] = at;
    at += round256(qo);
    off[3 * l + 1] = at;
    at += round256(kv);
    off[3 * l + 2] = at;
    at += round256(kv);
  }
  off[3 * layers] = at;  // positions
  at += round256((size_t)M * sizeof(int32_t));
  for (int l = 0; l < layers; ++l) {
    off[3 * layers + 1 + l] = at;
    at += round256(qo);
  }
  off[4 * layers + 1] = at;
}

}  // namespace

extern "C" {

int kvs_step_graph_create(int layers, const float *const *q, const float *const *k_rows,
                          const float *const *v_rows, const int32_t *positions,
                          float *const *k_cache, float *const *v_cache, float *const *out,
                          int M, int num_heads, int num_kv_heads, int head_dim, int max_len,
                          int chunk_size, void *workspace, size_t workspace_bytes,
                          int *d_status, kvs_stream_t stream, kvs_step_graph **graph) {
  if (!graph) return KVS_ERR_NULL;
  *graph = nullptr;
  if (layers < 1 || M < 1 || chunk_size < 0) return KVS_ERR_DIMS;
  if (!q || !k_rows || !v_rows || !k_cache || !v_cache || !out) return KVS_ERR_NULL;
  if (!stream) return KVS_ERR_DIMS;  // the legacy default stream cannot be captured
  // Validate every layer's pointers and configure the kernel before capturing.
  for (int l = 0; l < layers; ++l) {
    if (!q[l] || !k_rows[l] || !v_rows[l] || !k_cache[l] || !v_cache[l] || !out[l])
      return KVS_ERR_NULL;
  }
  const int chunk = chunk_size > 0 ? chunk_size
                                   : kvs_choose_chunk_size(M, num_kv_heads, head_dim, max_len, 0);
  if (chunk <= 0) return -chunk;
  int rc = kvs_prepare(num_heads, num_kv_heads, head_dim);
  if (rc != KVS_OK) return rc;
  // A layer after the first follows another layer of the step, which writes
  // neither the positions nor a cache row below a position: its kernel may
  // read those before its dependency wait (SeqArgs::early).
  return capture_step_graph(
      reinterpret_cast<cudaStream_t>(stream), workspace, layers,
      [&]() {
        int r = KVS_OK;
        for (int l = 0; l < layers && r == KVS_OK; ++l)
          r = kvs::decode_step(q[l], k_rows[l], v_rows[l], positions, k_cache[l], v_cache[l],
                               out[l], M, num_heads, num_kv_heads, head_dim, max_len, chunk,
                               workspace, workspace_bytes, d_status, stream, l > 0);
        return r;
      },
      graph);
}

int kvs_step_graph_io_layout(int layers, int M, int num_heads, int num_kv_heads, int head_dim,
                             size_t *offsets) {
  if (layers < 1 || M < 1 || num_heads < 1 || num_kv_heads < 1 || head_dim < 1)
    return KVS_ERR_DIMS;
  if (!offsets) return KVS_ERR_NULL;
  step_io_offsets(layers, M, num_heads, num_kv_heads, head_dim, offsets);
  return KVS_OK;
}

int kvs_step_graph_create_host_io(int layers, void *host_io, void *io, size_t io_bytes,
                                  float *const *k_cache, float *const *v_cache, int M,
                                  int num_heads, int num_kv_heads, int head_dim, int max_len,
                                  int chunk_size, void *workspace, size_t workspace_bytes,
                                  int *d_status, kvs_stream_t stream, kvs_step_graph **graph) {
  if (!graph) return KVS_ERR_NULL;
  *graph = nullptr;
  if (layers < 1 || M < 1 || chunk_size < 0 || num_heads < 1 || num_kv_heads < 1 ||
      head_dim < 1)
    return KVS_ERR_DIMS;
  if (!host_io || !io || !k_cache || !v_cache) return KVS_ERR_NULL;
  if (!stream) return KVS_ERR_DIMS;  // the legacy default stream cannot be captured
  if ((reinterpret_cast<uintptr_t>(io) & 255u) != 0) return KVS_ERR_ALIGN;
  for (int l = 0; l < layers; ++l)
    if (!k_cache[l] || !v_cache[l]) return KVS_ERR_NULL;
  std::vector<size_t> off(4 * (size_t)layers + 2);
  step_io_offsets(layers, M, num_heads, num_kv_heads, head_dim, off.data());
  const size_t in_end = off[3 * layers + 1], total = off[4 * layers + 1];
  if (io_bytes < total) return KVS_ERR_WORKSPACE;
  // The copies are kernels of this library reading and writing the host
  // buffer over the host link: it must be pinned memory the GPU can address
  // (a copy engine's copy from pageable memory cannot be part of a graph).
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, host_io) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_UNSUPPORTED;
  }
  if (pa.type != cudaMemoryTypeHost || pa.devicePointer == nullptr ||
      (reinterpret_cast<uintptr_t>(pa.devicePointer) & 15u) != 0)
    return KVS_ERR_UNSUPPORTED;
  unsigned char *mapped = static_cast<unsigned char *>(pa.devicePointer);
  unsigned char *base = static_cast<unsigned char *>(io);
  const int chunk = chunk_size > 0 ? chunk_size
                                   : kvs_choose_chunk_size(M, num_kv_heads, head_dim, max_len, 0);
  if (chunk <= 0) return -chunk;
  int rc = kvs_prepare(num_heads, num_kv_heads, head_dim);
  if (rc != KVS_OK) return rc;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int32_t *pos = reinterpret_cast<const int32_t *>(base + off[3 * layers]);
  return capture_step_graph(
      s, workspace, layers,
      [&]() {
        // every layer's inputs and the positions, in one copy
        int r = kvs::launch_io_copy(mapped, base, in_end, s);
        for (int l = 0; l < layers && r == KVS_OK; ++l)
          r = kvs::decode_step(reinterpret_cast<const float *>(base + off[3 * l]),
                               reinterpret_cast<const float *>(base + off[3 * l + 1]),
                               reinterpret_cast<const float *>(base + off[3 * l + 2]), pos,
                               k_cache[l], v_cache[l],
                               reinterpret_cast<float *>(base + off[3 * layers + 1 + l]), M,
                               num_heads, num_kv_heads, head_dim, max_len, chunk, workspace,
                               workspace_bytes, d_status, stream, l > 0);
        // every layer's out, in one copy
        if (r == KVS_OK) r = kvs::launch_io_copy(base + in_end, mapped + in_end, total - in_end, s);
        return r;
      },
      graph);
}

int kvs_step_graph_launch(kvs_step_graph *graph, kvs_stream_t stream) {
  if (!graph || !graph->exec) return KVS_ERR_NULL;
  std::lock_guard<std::mutex> lk(graph->mu);
  cudaMemsetParams p = graph->epoch;
  p.value = kvs::fresh_tag();  // this replay's epoch
  if (cudaGraphExecMemsetNodeSetParams(graph->exec, graph->epoch_node, &p) != cudaSuccess ||
      cudaGraphLaunch(graph->exec, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  return KVS_OK;
}

int kvs_step_graph_destroy(kvs_step_graph *graph) {
  if (!graph) return KVS_OK;
  if (graph->exec) cudaGraphExecDestroy(graph->exec);
  if (graph->graph) cudaGraphDestroy(graph->graph);
  delete graph;
  return KVS_OK;
}

}  // extern "C"
