// kvs_launch.h -- internal interface between the C-ABI layer (kvs_api.cu)
// and the kernel launchers.  Not installed; not part of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace kvs {

// Workspace layout of the chunk partials, shared by the chunk and reduce
// kernels.  For sequence i, query head h, chunk c (n_max = ceil(Lmax / C)):
//   acc [((i*H + h)*n_max + c)*D + d]   weighted-V accumulator, float32
//   ml  [((i*H + h)*n_max + c)*2 + 0]   running max of the scores (log2 units)
//   ml  [((i*H + h)*n_max + c)*2 + 1]   running sum exp2(s - max)
struct PartialLayout {
  int64_t n_max;
  size_t acc_bytes;  // offset of ml
  size_t total_bytes;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline PartialLayout partial_layout(int M, int H, int D, int max_len,
                                    int chunk) {
  PartialLayout p;
  p.n_max = ((int64_t)max_len + chunk - 1) / chunk;
  const size_t slots = (size_t)M * (size_t)H * (size_t)p.n_max;
  p.acc_bytes = align_up(slots * (size_t)D * sizeof(float), 256);
  p.total_bytes = p.acc_bytes + align_up(slots * 2 * sizeof(float), 256);
  return p;
}

int launch_kv_scatter(const float *k_rows, const float *v_rows,
                      const int32_t *positions, float *k_cache, float *v_cache,
                      int M, int Hkv, int D, int max_len, int *d_status,
                      cudaStream_t stream);

int launch_fd_chunks(const float *q, const float *k_cache, const float *v_cache,
                     const int32_t *positions, int M, int H, int Hkv, int D,
                     int max_len, int chunk, void *workspace, int *d_status,
                     cudaStream_t stream);

int launch_fd_reduce(const int32_t *positions, float *out, int M, int H, int D,
                     int max_len, int chunk, const void *workspace,
                     int *d_status, cudaStream_t stream);

// Number of SMs of the current device (cached per device); <= 0 on error.
int device_sm_count();

}  // namespace kvs
