// argmax.cu -- batched greedy token selection: for each of M logit rows,
// the index of the largest logit, in one launch.
//
// Source: realizar 0.8.5, src/cuda/executor/reduces.rs, gpu_argmax (PAR-062,
// PAR-068) and batched_gpu_argmax (PMAT-045): a two-pass reduction (blocks
// find local (max, index) pairs, one block reduces those) run for M rows with
// one synchronisation, so only the token IDs leave the GPU.
//
// GB300 design: one thread-block cluster of CS blocks per row (a row of a
// 152,064-entry vocabulary is 608 KB).  Block r reduces an equal slice of
// the row with 16-byte loads; the CS block results meet over distributed
// shared memory after one cluster barrier, so the second pass needs neither
// a second launch nor a global buffer.  All M rows go in one launch: the
// pages launch 2*M kernels.
//
// Order: a larger value wins; equal values go to the smaller index; NaN is
// never chosen (it is read as -inf); a row with nothing above -inf gives 0.

#include <cstdint>
#include <mutex>

#include "kvs_device.cuh"
#include "kvs_launch.h"
#include "kvsdecode.h"

namespace kvs {

namespace {

constexpr int kArgmaxThreads = 512;
constexpr int kArgmaxMaxDevices = 64;

struct Best {
  float v;
  int i;
};

__device__ __forceinline__ Best better(Best a, Best b) {
  return (b.v > a.v || (b.v == a.v && b.i < a.i)) ? b : a;
}

__device__ __forceinline__ void take(Best &b, float x, int i) {
  const float v = (x == x) ? x : neg_inf_f();
  if (v > b.v || (v == b.v && i < b.i)) {
    b.v = v;
    b.i = i;
  }
}

__device__ __forceinline__ Best warp_best(Best b) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    Best c;
    c.v = __shfl_xor_sync(0xffffffffu, b.v, o);
    c.i = __shfl_xor_sync(0xffffffffu, b.i, o);
    b = better(b, c);
  }
  return b;
}

// grid (CS, rows), clusters of (CS, 1, 1); rows >= gridDim.y loop.
__global__ void __launch_bounds__(kArgmaxThreads)
    argmax_cluster_kernel(const float *__restrict__ logits, int M, int V, int32_t *ids) {
  __shared__ Best s_warp[kArgmaxThreads / 32];
  __shared__ float s_v;
  __shared__ int s_i;
  const int t = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const int cs = (int)gridDim.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0) && (V % 4 == 0);
  grid_dependency_wait();
  allow_dependent_launch();
  for (int row = blockIdx.y; row < M; row += gridDim.y) {  // same trip count in a cluster
    const float *x = logits + (size_t)row * V;
    Best b{neg_inf_f(), 0x7fffffff};
    if (vec) {
      const int V4 = V / 4;
      const int a = (int)((long long)V4 * rank / cs);
      const int e = (int)((long long)V4 * (rank + 1) / cs);
      const float4 *x4 = reinterpret_cast<const float4 *>(x);
      int k = a + t;
      for (; k + 3 * kArgmaxThreads < e; k += 4 * kArgmaxThreads) {  // four loads in flight
        float4 f[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) f[u] = __ldcs(x4 + k + u * kArgmaxThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i0 = 4 * (k + u * kArgmaxThreads);
          take(b, f[u].x, i0);
          take(b, f[u].y, i0 + 1);
          take(b, f[u].z, i0 + 2);
          take(b, f[u].w, i0 + 3);
        }
      }
      for (; k < e; k += kArgmaxThreads) {
        const float4 f = __ldcs(x4 + k);
        take(b, f.x, 4 * k);
        take(b, f.y, 4 * k + 1);
        take(b, f.z, 4 * k + 2);
        take(b, f.w, 4 * k + 3);
      }
    } else {
      const int a = (int)((long long)V * rank / cs);
      const int e = (int)((long long)V * (rank + 1) / cs);
      for (int k = a + t; k < e; k += kArgmaxThreads) take(b, __ldcs(x + k), k);
    }
    b = warp_best(b);
    if ((t & 31) == 0) s_warp[t >> 5] = b;
    __syncthreads();
    if (t < 32) {
      Best c = (t < kArgmaxThreads / 32) ? s_warp[t] : Best{neg_inf_f(), 0x7fffffff};
      c = warp_best(c);
      if (t == 0) {
        s_v = c.v;
        s_i = c.i;
      }
    }
    cluster_sync_all();  // every block's (max, index) is in its shared memory
    if (rank == 0 && t < 32) {
      Best c{neg_inf_f(), 0x7fffffff};
      if (t < cs) {
        c.v = ld_dsmem_f32(dsmem_addr(&s_v, t));
        c.i = ld_dsmem_s32(dsmem_addr(&s_i, t));
      }
      c = warp_best(c);
      if (t == 0) ids[row] = (c.i == 0x7fffffff) ? 0 : c.i;
    }
    cluster_sync_all();  // block 0 has read them: they may be overwritten
  }
}

struct ArgmaxInfo {
  int max_size = 0;
  int active[5] = {0};
  bool configured = false;
};

const ArgmaxInfo *argmax_info(int dev) {
  static ArgmaxInfo info[kArgmaxMaxDevices];
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (!info[dev].configured) {
    int top = 16;
    if (cudaFuncSetAttribute(argmax_cluster_kernel,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
      cudaGetLastError();
      top = 8;
    }
    ArgmaxInfo rec;
    for (int k = 0, cs = 1; cs <= top; ++k, cs <<= 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, argmax_cluster_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      if (n <= 0) break;
      rec.active[k] = n;
      rec.max_size = cs;
    }
    if (rec.max_size < 1) return nullptr;
    rec.configured = true;
    info[dev] = rec;
  }
  return &info[dev];
}

}  // namespace

int launch_argmax(const float *logits, int M, int V, int32_t *ids, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kArgmaxMaxDevices)
    return KVS_ERR_LAUNCH;
  const ArgmaxInfo *ai = argmax_info(dev);
  if (!ai) return KVS_ERR_LAUNCH;
  // Largest cluster size whose clusters for all M rows are resident at once
  // (one wave), and no slice under 16 KB.
  int cs = ai->max_size, k = 0;
  while ((1 << k) < cs) ++k;
  while (cs > 1 && ((long long)M > ai->active[k] || (long long)V * 4 / cs < (16 << 10))) {
    cs >>= 1;
    --k;
  }
  const int rows = M < 65535 ? M : 65535;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, rows, 1);
  cfg.blockDim = dim3(kArgmaxThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, argmax_cluster_kernel, logits, M, V, ids);
  if (e != cudaSuccess) {
    cudaGetLastError();  // leave no stale error for the caller's next check
    return KVS_ERR_LAUNCH;
  }
  return KVS_OK;
}

}  // namespace kvs
