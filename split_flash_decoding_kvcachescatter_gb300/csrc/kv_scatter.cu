// kv_scatter.cu -- writes each sequence's new K and V row into its KV cache
// at the sequence's position, for all M sequences and both caches in one
// launch.
//
// Source: realizar 0.8.5, src/cuda/executor/head_dim.rs,
// flash_decoding_attention_into, "Step 1: Scatter K/V to caches" -- the
// pages launch one (num_kv_heads x head_dim) kernel per sequence and per
// cache (2*M launches) with the host position as an argument; here the
// position is read on the device (aprender-serve 0.70.2,
// src/gguf/cuda/forward_qwen35_cuda_graph.rs, module doc: the K/V row is
// scattered at *io.pos) and one launch covers everything.
//
// Work: 2*M*Hkv*D floats read and written.  It is launch-latency bound; each
// thread moves one float4 (coalesced 16-byte loads and stores).  It is
// launched with programmatic stream serialisation, so its launch overlaps the
// tail of the previous kernel in the stream.

#include "kvs_device.cuh"
#include "kvs_launch.h"

namespace kvs {

__global__ void __launch_bounds__(256)
    kv_scatter_kernel(const float4 *__restrict__ k_rows,
                      const float4 *__restrict__ v_rows,
                      const int32_t *__restrict__ positions,
                      float4 *__restrict__ k_cache, float4 *__restrict__ v_cache,
                      int M, int Hkv, int D4, int max_len, int *d_status) {
  // the caches may still be read by the preceding kernel in the stream
  grid_dependency_wait();
  allow_dependent_launch();
  const int64_t per_cache = (int64_t)M * Hkv * D4;  // float4s per cache
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= 2 * per_cache) return;
  const bool is_v = idx >= per_cache;
  const int64_t e = is_v ? idx - per_cache : idx;  // within [M][Hkv][D4]
  const int d4 = (int)(e % D4);
  const int64_t ig = e / D4;  // i * Hkv + g
  const int i = (int)(ig / Hkv);
  const int p = __ldca(positions + i);
  if (p < 0 || p >= max_len) {
    if (!is_v && d4 == 0 && ig % Hkv == 0) record_status(d_status, KVS_ERR_POSITION);
    return;
  }
  const int64_t dst = (ig * max_len + p) * D4 + d4;
  if (is_v)
    v_cache[dst] = __ldcg(v_rows + e);
  else
    k_cache[dst] = __ldcg(k_rows + e);
}

int launch_kv_scatter(const float *k_rows, const float *v_rows,
                      const int32_t *positions, float *k_cache, float *v_cache,
                      int M, int Hkv, int D, int max_len, int *d_status,
                      cudaStream_t stream) {
  const int D4 = D / 4;
  const int64_t total = 2ll * M * Hkv * D4;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  static bool carveout_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64 && !carveout_set[dev]) {
    // the same L1/shared split as the attention kernels that follow it
    cudaFuncSetAttribute(kv_scatter_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    carveout_set[dev] = true;
  }
  const cudaError_t e = launch_pdl(
      kv_scatter_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
      reinterpret_cast<const float4 *>(k_rows), reinterpret_cast<const float4 *>(v_rows),
      positions, reinterpret_cast<float4 *>(k_cache), reinterpret_cast<float4 *>(v_cache), M,
      Hkv, D4, max_len, d_status);
  return e == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

}  // namespace kvs
