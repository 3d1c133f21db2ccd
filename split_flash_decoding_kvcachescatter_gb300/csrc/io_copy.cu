// io_copy.cu -- moves the inputs and the result of a host-buffer decode step
// (kvs_decode_step_host_io) between pinned host memory and the device with
// the SMs' own loads and stores, instead of a copy engine.
//
// Why: a decode step moves well under a megabyte each way (8B-class batch:
// 786 KB in, 524 KB out).  Measured on GB300 (same box, same inputs), that
// step with its two copies on copy engines took 185.9 us against 164 us
// without copies; with this kernel doing both, 171.9 us.  Pinned host memory
// is addressable from the GPU over the host link, and a grid of blocks that
// each keep a few 16-byte words in flight moves it at far more than one copy
// engine's rate; the copy is one more launch in the stream, chained to its
// neighbours with programmatic dependent launch.

#include <algorithm>

#include "kvs_device.cuh"
#include "kvs_launch.h"

namespace kvs {

namespace {

constexpr int kIoThreads = 256;
constexpr int kIoPerThread = 4;  // 16-byte words a thread keeps in flight

// dst[0, bytes) = src[0, bytes); src and dst 16-byte aligned.
__global__ void __launch_bounds__(kIoThreads)
    io_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, size_t n16,
                   const unsigned char *__restrict__ src_tail,
                   unsigned char *__restrict__ dst_tail, int tail_bytes) {
  // The source may be written, and the destination read, by the preceding
  // kernel in the stream: wait for it.  The kernel that follows reads what
  // this one writes, so it is let in only once every word is written (it
  // cannot see a partial copy through any cache), and the loads are
  // coherent (.cg): the source is not read-only while this grid is resident.
  grid_dependency_wait();
  const size_t stride = (size_t)gridDim.x * kIoThreads * kIoPerThread;
  for (size_t e0 = (size_t)blockIdx.x * kIoThreads * kIoPerThread + threadIdx.x; e0 < n16;
       e0 += stride) {
    uint4 w[kIoPerThread];
#pragma unroll
    for (int u = 0; u < kIoPerThread; ++u) {
      const size_t e = e0 + (size_t)u * kIoThreads;
      if (e < n16) w[u] = __ldcg(src + e);
    }
#pragma unroll
    for (int u = 0; u < kIoPerThread; ++u) {
      const size_t e = e0 + (size_t)u * kIoThreads;
      if (e < n16) dst[e] = w[u];
    }
  }
  if (blockIdx.x == 0 && (int)threadIdx.x < tail_bytes)
    dst_tail[threadIdx.x] = __ldcg(src_tail + threadIdx.x);
  allow_dependent_launch();
}

}  // namespace

int launch_io_copy(const void *src, void *dst, size_t bytes, cudaStream_t stream) {
  const size_t n16 = bytes / 16;
  const int tail = (int)(bytes % 16);
  const int sms = device_sm_count();
  if (sms <= 0) return KVS_ERR_LAUNCH;
  const size_t per_block = (size_t)kIoThreads * kIoPerThread;
  const size_t want = std::max<size_t>(1, (n16 + per_block - 1) / per_block);
  const unsigned blocks = (unsigned)std::min<size_t>(want, (size_t)sms * 4);
  const unsigned char *s = static_cast<const unsigned char *>(src);
  unsigned char *d = static_cast<unsigned char *>(dst);
  const cudaError_t e = launch_pdl(io_copy_kernel, dim3(blocks), dim3(kIoThreads), 0, stream,
                                   reinterpret_cast<const uint4 *>(s),
                                   reinterpret_cast<uint4 *>(d), n16, s + n16 * 16,
                                   d + n16 * 16, tail);
  return e == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

}  // namespace kvs
