// kvs_launch.h -- internal interface between the C-ABI layer (kvs_api.cu)
// and the kernel launchers.  Not installed; not part of the C ABI.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kvsdecode.h"

namespace kvs {

// Upper bound on the step kernel's persistent grid (GB300: 152 SMs x 2).
constexpr int kMaxChunkBlocks = 1024;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace of kvs_flash_decode / kvs_decode_step.
//   header  256 bytes: a u32 epoch at offset 0 (changed by any call that
//           gives up on a bounded wait; part of the counters' tag, so that
//           counts such a call left behind never match a later call, even a
//           replayed CUDA graph whose tag argument is frozen), the rest
//           reserved
//   done    u64 [M*Hkv]: rows of (i, g) whose partial is written (counters
//           carry the tag of the call that last used them, so the buffer
//           needs no initialisation)
//   ml      float2 [slots][G]: (running max in log2 units, running sum)
//   acc     float  [slots][G][D]: unnormalised weighted-V accumulator
// A partial slot belongs to one run of consecutive chunks of one (i, g):
//   slot i*Hkv + g          the run that starts at chunk 0 of (i, g)
//   slot M*Hkv + b          block b's first run, when it starts inside (i, g)
// so slots = M*Hkv + kMaxChunkBlocks, independent of max_len and chunk size.
struct WsLayout {
  size_t off_done, off_ml, off_acc, total;
  int64_t slots;
};

inline WsLayout ws_layout(int M, int Hkv, int G, int D) {
  WsLayout l;
  l.slots = (int64_t)M * Hkv + kMaxChunkBlocks;
  l.off_done = 256;
  l.off_ml = align_up(l.off_done + (size_t)M * Hkv * 8, 256);
  l.off_acc = align_up(l.off_ml + (size_t)l.slots * G * 8, 256);
  l.total = align_up(l.off_acc + (size_t)l.slots * G * D * 4, 256);
  return l;
}

struct WsView {
  unsigned *epoch;
  unsigned long long *done;
  float2 *ml;
  float *acc;
};

inline WsView workspace_view(void *base, int M, int Hkv, int G, int D) {
  const WsLayout l = ws_layout(M, Hkv, G, D);
  unsigned char *p = static_cast<unsigned char *>(base);
  return WsView{reinterpret_cast<unsigned *>(p), reinterpret_cast<unsigned long long *>(p + l.off_done),
                reinterpret_cast<float2 *>(p + l.off_ml), reinterpret_cast<float *>(p + l.off_acc)};
}

// Launch with programmatic stream serialisation: the kernel may start while
// its predecessor in the stream finishes; every kernel of this library
// executes griddepcontrol.wait before it touches global memory, so results
// are those of plain stream order.  Because the kernel is resident while its
// predecessor may still be writing, it never reads through the read-only
// (ld.global.nc) path data that a preceding kernel can write: those loads are
// coherent (.ca or .cg), or bulk copies through L2.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
  // a refused launch also sets the runtime's last error: clear it, so that
  // the caller's next CUDA error check does not report it a second time
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

// The sequences of one call: positions, and optionally a cache slot per
// sequence (slots == nullptr: slot i, num_slots == M) and a finished flag
// per sequence (done == nullptr: none).  All device pointers.
struct SeqArgs {
  const int32_t *positions;
  const int32_t *slots;
  const uint8_t *done;
  int max_len;
  int num_slots;
  // The kernel preceding this launch in the stream writes neither the
  // positions, slots and finished flags nor any cache row below a sequence's
  // position (a layer of a step graph after the first): the cluster kernel
  // then reads them, and starts streaming those rows, before its dependency
  // wait.  The persistent kernel ignores it.
  bool early = false;
};

// kvs_decode_step with SeqArgs::early set as given (the step graph's
// layers after the first); validation and dispatch are the same.
int decode_step(const float *q, const float *k_rows, const float *v_rows,
                const int32_t *positions, float *k_cache, float *v_cache, float *out, int M,
                int num_heads, int num_kv_heads, int head_dim, int max_len, int chunk_size,
                void *workspace, size_t workspace_bytes, int *d_status, kvs_stream_t stream,
                bool early);

int launch_kv_scatter(const float *k_rows, const float *v_rows, const int32_t *positions,
                      float *k_cache, float *v_cache, int M, int Hkv, int D, int max_len,
                      int *d_status, cudaStream_t stream);

// One launch of the step kernel: split-K attention over the caches; with
// k_rows/v_rows non-null the scatter of those rows is done in the same launch.
int launch_fd_step(const float *q, float *k_cache, float *v_cache, const SeqArgs &seqs,
                   const float *k_rows, const float *v_rows, float *out, int M, int H, int Hkv,
                   int D, int chunk, void *workspace, int *d_status, cudaStream_t stream);

// One launch of the cluster kernel (one thread-block cluster per (sequence,
// kv head), partials merged in distributed shared memory; no workspace).
// Requires M * Hkv <= kMaxClusterPairs.
constexpr long long kMaxClusterPairs = 65535;
int launch_fd_cluster(const float *q, float *k_cache, float *v_cache, const SeqArgs &seqs,
                      const float *k_rows, const float *v_rows, float *out, int M, int H, int Hkv,
                      int D, int *d_status, cudaStream_t stream);

// Sets the cluster kernel's attributes for (H / Hkv, D) on the current device.
int prepare_cluster_kernel(int H, int Hkv, int D);

// 1 if the automatic schedule should run this shape on the cluster kernel
// (current device; configures the kernel on first use), else 0.
int cluster_auto_ok(int M, int H, int Hkv, int D, int max_len);

// One launch of the batched argmax (ids[m] = argmax of logits row m).
int launch_argmax(const float *logits, int M, int V, int32_t *ids, cudaStream_t stream);

// The tensor-core prefill attention (q, k, v, out [H][S][D]): a pack launch
// (FP16 tiles into the workspace) and the attention launch.
size_t prefill_workspace_bytes(int H, int S, int D);
int launch_prefill(const float *q, const float *k, const float *v, float *out, int H, int S, int D,
                   int causal, void *workspace, int *d_status, cudaStream_t stream);

// Sets the step kernel's attributes for (H / Hkv, D) on the current device
// (done on first use anyway; a stream capture calls it beforehand).
int prepare_step_kernel(int H, int Hkv, int D);

// Number of SMs of the current device (cached per device); <= 0 on error.
int device_sm_count();

// dst[0, bytes) = src[0, bytes) by a kernel (the SMs' loads and stores), for
// a host buffer the GPU can address; src and dst 16-byte aligned.
int launch_io_copy(const void *src, void *dst, size_t bytes, cudaStream_t stream);

// A fresh nonzero 32-bit value for every call (a process-wide counter): the
// per-launch tag of the step kernel's workspace counters, and the workspace
// epoch a step graph writes at each replay.
unsigned fresh_tag();

// True while kvs_set_wait_limit_ns has lowered the wait bound of the current
// device: launches then take the kernels' polling wait variant, which reads
// the bound at run time (kvs_device.cuh).
bool poll_waits();

// Each translation unit that has pipeline waits keeps its own copy of the
// wait bound (kvs_device.cuh); these set it on the current device.
int set_wait_limit_step(uint64_t ns);
int set_wait_limit_cluster(uint64_t ns);
int set_wait_limit_prefill(uint64_t ns);

}  // namespace kvs
