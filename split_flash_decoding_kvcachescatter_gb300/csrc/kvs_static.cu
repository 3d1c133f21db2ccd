// kvs_static.cu -- kvs_flash_decode_static: split-K decode attention whose
// scratch (the chunk partials) lives in a fixed buffer inside this library
// instead of a caller-provided workspace.
//
// Why it exists: some callers cannot allocate device memory at the point
// where they run attention -- for example code that runs under a strict
// memory budget that forbids cudaMalloc after start-up, plug-in hosts that
// hand out streams and tensors but no allocator, or runtimes whose own
// allocator must not be re-entered from this call.  For them this entry point
// takes only inputs and outputs and allocates nothing: no cudaMalloc, no
// cudaFree, no allocating library routine.
//
// The buffer is a file-scope __device__ array of KVS_STATIC_WORKSPACE_BYTES.
// Every GPU on which this library's device code is loaded holds it until
// the process exits.  Host code cannot use the array's name as a device
// address (on the host it names a stand-in object), so the first call on each
// device looks up the real address with cudaGetSymbolAddress while that
// device is current, and caches it.  CUDA loads device code lazily, so that
// lookup is also when the device commits the buffer; a device that cannot
// provide it makes the call return KVS_ERR_MEMORY.  The cached address
// belongs to the device's primary context: it is not valid after that
// context is destroyed (cudaDeviceReset).

#include <cstdint>
#include <mutex>

#include "kvs_launch.h"
#include "kvsdecode.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[KVS_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {nullptr};

// Device address of g_static_workspace on the current device (looked up once
// per device) in *addr.  Returns KVS_OK, KVS_ERR_MEMORY when the device could
// not provide the buffer, or KVS_ERR_LAUNCH for any other failure.
int static_workspace_address(void **addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // reset the error state so later CUDA calls do not see it
      return e == cudaErrorMemoryAllocation ? KVS_ERR_MEMORY : KVS_ERR_LAUNCH;
    }
    g_addr[dev] = p;
  }
  *addr = g_addr[dev];
  return KVS_OK;
}

}  // namespace

extern "C" int kvs_flash_decode_static(const float *q, const float *k_cache,
                                       const float *v_cache, const int32_t *positions,
                                       float *out, int M, int num_heads, int num_kv_heads,
                                       int head_dim, int max_len, int chunk_size,
                                       int *d_status, kvs_stream_t stream) {
  // Same shape rules as kvs_flash_decode; an invalid shape sizes to 0 bytes.
  if (M == 0) return kvs_flash_decode(q, k_cache, v_cache, positions, out, M, num_heads,
                                      num_kv_heads, head_dim, max_len, chunk_size, nullptr,
                                      0, d_status, stream);
  const size_t need = kvs_flash_decode_workspace_bytes(M, num_heads, num_kv_heads, head_dim,
                                                       max_len, chunk_size);
  if (need == 0)  // invalid arguments: let the regular entry report which
    return kvs_flash_decode(q, k_cache, v_cache, positions, out, M, num_heads, num_kv_heads,
                            head_dim, max_len, chunk_size, nullptr, 0, d_status, stream);
  if (need > (size_t)KVS_STATIC_WORKSPACE_BYTES) return KVS_ERR_WORKSPACE;
  void *ws = nullptr;
  const int rc = static_workspace_address(&ws);
  if (rc != KVS_OK) return rc;
  // The partials need no initial value: every slot the reduce reads is
  // written by the chunk kernel of the same call.
  return kvs_flash_decode(q, k_cache, v_cache, positions, out, M, num_heads, num_kv_heads,
                          head_dim, max_len, chunk_size, ws, (size_t)KVS_STATIC_WORKSPACE_BYTES,
                          d_status, stream);
}
