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

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  // A layer after the first follows another layer of the step, which writes
  // neither the positions nor a cache row below a position: its kernel may
  // read those before its dependency wait (SeqArgs::early).
  for (int l = 0; l < layers && rc == KVS_OK; ++l)
    rc = kvs::decode_step(q[l], k_rows[l], v_rows[l], positions, k_cache[l], v_cache[l], out[l],
                          M, num_heads, num_kv_heads, head_dim, max_len, chunk, workspace,
                          workspace_bytes, d_status, stream, l > 0);
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
