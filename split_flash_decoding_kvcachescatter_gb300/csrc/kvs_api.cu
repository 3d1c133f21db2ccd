// kvs_api.cu -- the C ABI (include/kvsdecode.h): argument validation on the
// host, the chunk-size rule, workspace sizing, and dispatch to the kernel
// launchers.  Nothing here allocates, frees or synchronises.

#include <atomic>
#include <cstdint>
#include <mutex>

#include "kvs_launch.h"
#include "kvsdecode.h"

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool head_dim_supported(int D) { return D == 64 || D == 128; }

// Shape checks shared by the attention entry points (no pointers).
int check_attention_shape(int M, int H, int Hkv, int D, int max_len, int chunk) {
  if (M < 0 || H < 1 || Hkv < 1 || max_len < 1 || chunk < 0) return KVS_ERR_DIMS;
  if (H % Hkv != 0) return KVS_ERR_DIMS;
  if (!head_dim_supported(D)) return KVS_ERR_UNSUPPORTED;
  if (H / Hkv > 8) return KVS_ERR_UNSUPPORTED;
  if ((int64_t)M * H > 0x7fffffffll) return KVS_ERR_DIMS;
  return KVS_OK;
}

// Kernel schedule (kvs_set_schedule); process-wide.
std::atomic<int> g_schedule{KVS_SCHEDULE_AUTO};

// Wait bound of each device (kvs_set_wait_limit_ns), as last set.
constexpr int kMaxLimitDevices = 64;
std::mutex g_limit_mu;
std::atomic<uint64_t> g_limit[kMaxLimitDevices] = {};
struct LimitInit {
  LimitInit() {
    for (auto &x : g_limit) x.store(KVS_WAIT_LIMIT_DEFAULT_NS);
  }
} g_limit_init;

// Upper bound of the K/V bytes of one step above which the automatic
// schedule never considers the cluster kernel (checked before any device
// query).
constexpr long long kClusterAutoBytes = 64ll << 20;

bool use_cluster(int M, int H, int Hkv, int D, int max_len) {
  const long long pairs = (long long)M * Hkv;
  if (pairs > kvs::kMaxClusterPairs) return false;
  switch (g_schedule.load(std::memory_order_relaxed)) {
    case KVS_SCHEDULE_PERSISTENT: return false;
    case KVS_SCHEDULE_CLUSTER: return true;
    default:
      if (pairs * max_len * D * 8 > kClusterAutoBytes) return false;
      return kvs::cluster_auto_ok(M, H, Hkv, D, max_len) != 0;
  }
}

// The attention launch of kvs_flash_decode (k_rows == nullptr) and
// kvs_decode_step, on the schedule in force.
int launch_attention(const float *q, float *k_cache, float *v_cache, const kvs::SeqArgs &seqs,
                     const float *k_rows, const float *v_rows, float *out, int M, int H, int Hkv,
                     int D, int chunk, void *workspace, int *d_status, cudaStream_t stream) {
  if (use_cluster(M, H, Hkv, D, seqs.max_len))
    return kvs::launch_fd_cluster(q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, H, Hkv, D,
                                  d_status, stream);
  return kvs::launch_fd_step(q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, H, Hkv, D, chunk,
                             workspace, d_status, stream);
}

// chunk_size == 0 -> the library rule on the current device.
int resolve_chunk(int M, int Hkv, int D, int max_len, int chunk) {
  if (chunk > 0) return chunk;
  return kvs_choose_chunk_size(M, Hkv, D, max_len, 0);
}

}  // namespace

bool kvs::poll_waits() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxLimitDevices) {
    cudaGetLastError();
    return false;
  }
  return g_limit[dev].load(std::memory_order_relaxed) < KVS_WAIT_LIMIT_DEFAULT_NS;
}

extern "C" {

const char *kvs_strerror(int status) {
  switch (status) {
    case KVS_OK: return "ok";
    case KVS_ERR_NULL: return "a required pointer is NULL";
    case KVS_ERR_DIMS: return "invalid dimensions";
    case KVS_ERR_UNSUPPORTED: return "unsupported head_dim or query-head group";
    case KVS_ERR_ALIGN: return "pointer not aligned (16 bytes for tensors, 256 for workspace)";
    case KVS_ERR_WORKSPACE: return "workspace missing or too small";
    case KVS_ERR_LAUNCH: return "CUDA launch or device query failed";
    case KVS_ERR_POSITION: return "a position is outside [0, max_len)";
    case KVS_ERR_TIMEOUT: return "a bounded device pipeline wait expired";
    case KVS_ERR_SLOT: return "a cache slot is outside [0, num_slots)";
    case KVS_ERR_MEMORY: return "the device could not provide the library's own buffer";
    default: return "unknown kvs status";
  }
}

int kvs_kv_scatter(const float *k_rows, const float *v_rows, const int32_t *positions,
                   float *k_cache, float *v_cache, int M, int num_kv_heads, int head_dim,
                   int max_len, int *d_status, kvs_stream_t stream) {
  if (M < 0 || num_kv_heads < 1 || max_len < 1) return KVS_ERR_DIMS;
  if (!head_dim_supported(head_dim)) return KVS_ERR_UNSUPPORTED;
  if (M == 0) return KVS_OK;
  if (!k_rows || !v_rows || !positions || !k_cache || !v_cache) return KVS_ERR_NULL;
  if (!aligned(k_rows, 16) || !aligned(v_rows, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(positions, 4))
    return KVS_ERR_ALIGN;
  return kvs::launch_kv_scatter(k_rows, v_rows, positions, k_cache, v_cache, M, num_kv_heads,
                                head_dim, max_len, d_status,
                                reinterpret_cast<cudaStream_t>(stream));
}

int kvs_choose_chunk_size(int M, int num_kv_heads, int head_dim, int max_len, int num_sms) {
  if (M < 1 || num_kv_heads < 1 || max_len < 1) return -KVS_ERR_DIMS;
  if (!head_dim_supported(head_dim)) return -KVS_ERR_UNSUPPORTED;
  const int sms = num_sms > 0 ? num_sms : kvs::device_sm_count();
  if (sms <= 0) return -KVS_ERR_LAUNCH;
  // Chunks are the scheduling atoms of the persistent chunk kernel: a block's
  // range starts and ends on chunk boundaries, so the chunk size is the
  // granularity of the load balance (a block holds its 1/P share of the live
  // rows to within one chunk).  Partials are kept per run of chunks, so small
  // chunks cost no extra partial traffic.  Aim for about 1/128 of a block's
  // share of a full cache, as a power of two in [16, 64].
  const int64_t blocks = 2ll * sms;
  const int64_t share = (int64_t)M * num_kv_heads * max_len / blocks;
  int c = 16;
  while (c < 64 && 2ll * c * 128 <= share) c <<= 1;
  return c;
}

size_t kvs_flash_decode_workspace_bytes(int M, int num_heads, int num_kv_heads, int head_dim,
                                        int max_len, int chunk_size) {
  if (check_attention_shape(M, num_heads, num_kv_heads, head_dim, max_len, chunk_size) != KVS_OK)
    return 0;
  if (M == 0) return 0;
  // The partials are kept per run of chunks (see kvs_launch.h), so the size
  // depends on neither max_len nor the chunk size.
  return kvs::ws_layout(M, num_kv_heads, num_heads / num_kv_heads, head_dim).total;
}

// Pointer and workspace checks shared by the attention entry points.
static int check_attention_buffers(const float *q, const float *k_cache, const float *v_cache,
                                   const int32_t *positions, const float *out, int M,
                                   int num_heads, int num_kv_heads, int head_dim,
                                   const void *workspace, size_t workspace_bytes) {
  if (!q || !k_cache || !v_cache || !positions || !out) return KVS_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(positions, 4))
    return KVS_ERR_ALIGN;
  if (!workspace) return KVS_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KVS_ERR_ALIGN;
  if (workspace_bytes < kvs::ws_layout(M, num_kv_heads, num_heads / num_kv_heads, head_dim).total)
    return KVS_ERR_WORKSPACE;
  return KVS_OK;
}

int kvs_flash_decode(const float *q, const float *k_cache, const float *v_cache,
                     const int32_t *positions, float *out, int M, int num_heads,
                     int num_kv_heads, int head_dim, int max_len, int chunk_size,
                     void *workspace, size_t workspace_bytes, int *d_status,
                     kvs_stream_t stream) {
  int rc = check_attention_shape(M, num_heads, num_kv_heads, head_dim, max_len, chunk_size);
  if (rc != KVS_OK) return rc;
  if (M == 0) return KVS_OK;
  rc = check_attention_buffers(q, k_cache, v_cache, positions, out, M, num_heads, num_kv_heads,
                               head_dim, workspace, workspace_bytes);
  if (rc != KVS_OK) return rc;
  const int chunk = resolve_chunk(M, num_kv_heads, head_dim, max_len, chunk_size);
  if (chunk <= 0) return -chunk;
  // the caches are only read when no new rows are passed
  const kvs::SeqArgs seqs{positions, nullptr, nullptr, max_len, M};
  return launch_attention(q, const_cast<float *>(k_cache), const_cast<float *>(v_cache), seqs,
                          nullptr, nullptr, out, M, num_heads, num_kv_heads, head_dim, chunk,
                          workspace, d_status, reinterpret_cast<cudaStream_t>(stream));
}

int kvs_decode_step(const float *q, const float *k_rows, const float *v_rows,
                    const int32_t *positions, float *k_cache, float *v_cache, float *out, int M,
                    int num_heads, int num_kv_heads, int head_dim, int max_len, int chunk_size,
                    void *workspace, size_t workspace_bytes, int *d_status,
                    kvs_stream_t stream) {
  return kvs::decode_step(q, k_rows, v_rows, positions, k_cache, v_cache, out, M, num_heads,
                          num_kv_heads, head_dim, max_len, chunk_size, workspace,
                          workspace_bytes, d_status, stream, false);
}

}  // extern "C"

int kvs::decode_step(const float *q, const float *k_rows, const float *v_rows,
                     const int32_t *positions, float *k_cache, float *v_cache, float *out, int M,
                     int num_heads, int num_kv_heads, int head_dim, int max_len, int chunk_size,
                     void *workspace, size_t workspace_bytes, int *d_status,
                     kvs_stream_t stream, bool early) {
  int rc = check_attention_shape(M, num_heads, num_kv_heads, head_dim, max_len, chunk_size);
  if (rc != KVS_OK) return rc;
  if (M == 0) return KVS_OK;
  if (!k_rows || !v_rows) return KVS_ERR_NULL;
  if (!aligned(k_rows, 16) || !aligned(v_rows, 16)) return KVS_ERR_ALIGN;
  rc = check_attention_buffers(q, k_cache, v_cache, positions, out, M, num_heads, num_kv_heads,
                               head_dim, workspace, workspace_bytes);
  if (rc != KVS_OK) return rc;
  const int chunk = resolve_chunk(M, num_kv_heads, head_dim, max_len, chunk_size);
  if (chunk <= 0) return -chunk;
  kvs::SeqArgs seqs{positions, nullptr, nullptr, max_len, M};
  seqs.early = early;
  return launch_attention(q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, num_heads,
                          num_kv_heads, head_dim, chunk, workspace, d_status,
                          reinterpret_cast<cudaStream_t>(stream));
}

extern "C" {

namespace {

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Offsets of the device copies in the io buffer of kvs_decode_step_host:
// q, k_rows, v_rows, positions, out, each 256-byte aligned.
struct IoLayout {
  size_t q, k, v, pos, out, total;
};

IoLayout io_layout(int M, int num_heads, int num_kv_heads, int head_dim) {
  const size_t qo = (size_t)M * num_heads * head_dim * sizeof(float);
  const size_t kv = (size_t)M * num_kv_heads * head_dim * sizeof(float);
  IoLayout L;
  L.q = 0;
  L.k = L.q + round256(qo);
  L.v = L.k + round256(kv);
  L.pos = L.v + round256(kv);
  L.out = L.pos + round256((size_t)M * sizeof(int32_t));
  L.total = L.out + round256(qo);
  return L;
}

}  // namespace

size_t kvs_step_io_bytes(int M, int num_heads, int num_kv_heads, int head_dim) {
  if (M < 1 || num_heads < 1 || num_kv_heads < 1 || head_dim < 1) return 0;
  return io_layout(M, num_heads, num_kv_heads, head_dim).total;
}

int kvs_decode_step_host(const float *q, const float *k_rows, const float *v_rows,
                         const int32_t *positions, float *k_cache, float *v_cache, float *out,
                         int M, int num_heads, int num_kv_heads, int head_dim, int max_len,
                         int chunk_size, void *io, size_t io_bytes, void *workspace,
                         size_t workspace_bytes, int *d_status, kvs_stream_t stream) {
  int rc = check_attention_shape(M, num_heads, num_kv_heads, head_dim, max_len, chunk_size);
  if (rc != KVS_OK) return rc;
  if (M == 0) return KVS_OK;
  if (!q || !k_rows || !v_rows || !positions || !out || !io) return KVS_ERR_NULL;
  if (!aligned(io, 256)) return KVS_ERR_ALIGN;
  const IoLayout L = io_layout(M, num_heads, num_kv_heads, head_dim);
  if (io_bytes < L.total) return KVS_ERR_WORKSPACE;
  unsigned char *base = static_cast<unsigned char *>(io);
  float *dq = reinterpret_cast<float *>(base + L.q);
  float *dk = reinterpret_cast<float *>(base + L.k);
  float *dv = reinterpret_cast<float *>(base + L.v);
  int32_t *dpos = reinterpret_cast<int32_t *>(base + L.pos);
  float *dout = reinterpret_cast<float *>(base + L.out);
  rc = check_attention_buffers(dq, k_cache, v_cache, dpos, dout, M, num_heads, num_kv_heads,
                               head_dim, workspace, workspace_bytes);
  if (rc != KVS_OK) return rc;
  const int chunk = resolve_chunk(M, num_kv_heads, head_dim, max_len, chunk_size);
  if (chunk <= 0) return -chunk;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t qo = (size_t)M * num_heads * head_dim * sizeof(float);
  const size_t kv = (size_t)M * num_kv_heads * head_dim * sizeof(float);
  if (cudaMemcpyAsync(dpos, positions, (size_t)M * sizeof(int32_t), cudaMemcpyHostToDevice,
                      st) != cudaSuccess ||
      cudaMemcpyAsync(dq, q, qo, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(dk, k_rows, kv, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(dv, v_rows, kv, cudaMemcpyHostToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  const kvs::SeqArgs seqs{dpos, nullptr, nullptr, max_len, M};
  rc = launch_attention(dq, k_cache, v_cache, seqs, dk, dv, dout, M, num_heads, num_kv_heads,
                        head_dim, chunk, workspace, d_status, st);
  if (rc != KVS_OK) return rc;
  if (cudaMemcpyAsync(out, dout, qo, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  return KVS_OK;
}

int kvs_step_io_layout(int M, int num_heads, int num_kv_heads, int head_dim, size_t *offsets) {
  if (M < 1 || num_heads < 1 || num_kv_heads < 1 || head_dim < 1) return KVS_ERR_DIMS;
  if (!offsets) return KVS_ERR_NULL;
  const IoLayout L = io_layout(M, num_heads, num_kv_heads, head_dim);
  offsets[0] = L.q;
  offsets[1] = L.k;
  offsets[2] = L.v;
  offsets[3] = L.pos;
  offsets[4] = L.out;
  offsets[5] = L.total;
  return KVS_OK;
}

int kvs_decode_step_host_io(void *host_io, float *k_cache, float *v_cache, int M, int num_heads,
                            int num_kv_heads, int head_dim, int max_len, int chunk_size, void *io,
                            size_t io_bytes, void *workspace, size_t workspace_bytes,
                            int *d_status, kvs_stream_t stream) {
  int rc = check_attention_shape(M, num_heads, num_kv_heads, head_dim, max_len, chunk_size);
  if (rc != KVS_OK) return rc;
  if (M == 0) return KVS_OK;
  if (!host_io || !io) return KVS_ERR_NULL;
  if (!aligned(io, 256)) return KVS_ERR_ALIGN;
  const IoLayout L = io_layout(M, num_heads, num_kv_heads, head_dim);
  if (io_bytes < L.total) return KVS_ERR_WORKSPACE;
  unsigned char *base = static_cast<unsigned char *>(io);
  float *dq = reinterpret_cast<float *>(base + L.q);
  float *dk = reinterpret_cast<float *>(base + L.k);
  float *dv = reinterpret_cast<float *>(base + L.v);
  int32_t *dpos = reinterpret_cast<int32_t *>(base + L.pos);
  float *dout = reinterpret_cast<float *>(base + L.out);
  rc = check_attention_buffers(dq, k_cache, v_cache, dpos, dout, M, num_heads, num_kv_heads,
                               head_dim, workspace, workspace_bytes);
  if (rc != KVS_OK) return rc;
  const int chunk = resolve_chunk(M, num_kv_heads, head_dim, max_len, chunk_size);
  if (chunk <= 0) return -chunk;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t qo = (size_t)M * num_heads * head_dim * sizeof(float);
  unsigned char *host = static_cast<unsigned char *>(host_io);
  // the inputs (q, k_rows, v_rows, positions and the padding between them)
  // in one copy
  const size_t in_bytes = L.pos + (size_t)M * sizeof(int32_t);
  // Pinned host memory the GPU can address is moved by the library's copy
  // kernel; any other host memory by a copy engine.
  cudaPointerAttributes pa;
  unsigned char *mapped = nullptr;
  if (cudaPointerGetAttributes(&pa, host_io) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
      pa.devicePointer != nullptr && aligned(pa.devicePointer, 16))
    mapped = static_cast<unsigned char *>(pa.devicePointer);
  else
    cudaGetLastError();
  if (mapped) {
    rc = kvs::launch_io_copy(mapped, base, in_bytes, st);
    if (rc != KVS_OK) return rc;
  } else if (cudaMemcpyAsync(base, host, in_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  const kvs::SeqArgs seqs{dpos, nullptr, nullptr, max_len, M};
  rc = launch_attention(dq, k_cache, v_cache, seqs, dk, dv, dout, M, num_heads, num_kv_heads,
                        head_dim, chunk, workspace, d_status, st);
  if (rc != KVS_OK) return rc;
  if (mapped) return kvs::launch_io_copy(dout, mapped + L.out, qo, st);
  if (cudaMemcpyAsync(host + L.out, dout, qo, cudaMemcpyDeviceToHost, st) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  return KVS_OK;
}

int kvs_decode_step_slots(const float *q, const float *k_rows, const float *v_rows,
                          const int32_t *positions, const int32_t *slots, const uint8_t *done,
                          float *k_pool, float *v_pool, int num_slots, float *out, int M,
                          int num_heads, int num_kv_heads, int head_dim, int max_len,
                          int chunk_size, void *workspace, size_t workspace_bytes,
                          int *d_status, kvs_stream_t stream) {
  int rc = check_attention_shape(M, num_heads, num_kv_heads, head_dim, max_len, chunk_size);
  if (rc != KVS_OK) return rc;
  if (num_slots < 1 || (!slots && num_slots < M)) return KVS_ERR_DIMS;
  if (M == 0) return KVS_OK;
  if ((k_rows == nullptr) != (v_rows == nullptr)) return KVS_ERR_NULL;
  if (k_rows && (!aligned(k_rows, 16) || !aligned(v_rows, 16))) return KVS_ERR_ALIGN;
  if (slots && !aligned(slots, 4)) return KVS_ERR_ALIGN;
  rc = check_attention_buffers(q, k_pool, v_pool, positions, out, M, num_heads, num_kv_heads,
                               head_dim, workspace, workspace_bytes);
  if (rc != KVS_OK) return rc;
  const int chunk = resolve_chunk(M, num_kv_heads, head_dim, max_len, chunk_size);
  if (chunk <= 0) return -chunk;
  const kvs::SeqArgs seqs{positions, slots, done, max_len, num_slots};
  return launch_attention(q, k_pool, v_pool, seqs, k_rows, v_rows, out, M, num_heads,
                          num_kv_heads, head_dim, chunk, workspace, d_status,
                          reinterpret_cast<cudaStream_t>(stream));
}

int kvs_argmax(const float *logits, int M, int vocab_size, int32_t *token_ids,
               kvs_stream_t stream) {
  if (M < 0 || vocab_size < 1) return KVS_ERR_DIMS;
  if (M == 0) return KVS_OK;
  if (!logits || !token_ids) return KVS_ERR_NULL;
  if (!aligned(logits, 4) || !aligned(token_ids, 4)) return KVS_ERR_ALIGN;
  return kvs::launch_argmax(logits, M, vocab_size, token_ids,
                            reinterpret_cast<cudaStream_t>(stream));
}

size_t kvs_prefill_workspace_bytes(int num_heads, int seq_len, int head_dim) {
  if (num_heads < 1 || seq_len < 1 || num_heads > 65535 || (int64_t)seq_len > 65535ll * 128 ||
      !head_dim_supported(head_dim))
    return 0;
  return kvs::prefill_workspace_bytes(num_heads, seq_len, head_dim);
}

int kvs_prefill_attention(const float *q, const float *k, const float *v, float *out,
                          int num_heads, int seq_len, int head_dim, int causal, void *workspace,
                          size_t workspace_bytes, int *d_status, kvs_stream_t stream) {
  if (num_heads < 0 || seq_len < 0) return KVS_ERR_DIMS;
  if (!head_dim_supported(head_dim)) return KVS_ERR_UNSUPPORTED;
  if ((int64_t)num_heads > 65535 || (int64_t)seq_len > 65535ll * 128) return KVS_ERR_DIMS;
  if (num_heads == 0 || seq_len == 0) return KVS_OK;
  if (!q || !k || !v || !out) return KVS_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return KVS_ERR_ALIGN;
  if (!workspace) return KVS_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KVS_ERR_ALIGN;
  if (workspace_bytes < kvs::prefill_workspace_bytes(num_heads, seq_len, head_dim))
    return KVS_ERR_WORKSPACE;
  return kvs::launch_prefill(q, k, v, out, num_heads, seq_len, head_dim, causal ? 1 : 0,
                             workspace, d_status, reinterpret_cast<cudaStream_t>(stream));
}

int kvs_set_schedule(int schedule) {
  if (schedule != KVS_SCHEDULE_AUTO && schedule != KVS_SCHEDULE_PERSISTENT &&
      schedule != KVS_SCHEDULE_CLUSTER)
    return -KVS_ERR_DIMS;
  return g_schedule.exchange(schedule);
}

int kvs_get_schedule(void) { return g_schedule.load(); }

int kvs_set_wait_limit_ns(uint64_t ns, uint64_t *previous) {
  if (ns > KVS_WAIT_LIMIT_DEFAULT_NS) return KVS_ERR_DIMS;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxLimitDevices) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lk(g_limit_mu);
  int rc = kvs::set_wait_limit_step(ns);
  if (rc == KVS_OK) rc = kvs::set_wait_limit_cluster(ns);
  if (rc == KVS_OK) rc = kvs::set_wait_limit_prefill(ns);
  if (rc != KVS_OK) return rc;
  if (previous) *previous = g_limit[dev].load();
  g_limit[dev].store(ns);
  return KVS_OK;
}

int kvs_schedule_for(int M, int num_heads, int num_kv_heads, int head_dim, int max_len) {
  const int rc = check_attention_shape(M, num_heads, num_kv_heads, head_dim, max_len, 0);
  if (rc != KVS_OK) return -rc;
  if (M < 1) return -KVS_ERR_DIMS;
  return use_cluster(M, num_heads, num_kv_heads, head_dim, max_len) ? KVS_SCHEDULE_CLUSTER
                                                                    : KVS_SCHEDULE_PERSISTENT;
}

int kvs_prepare(int num_heads, int num_kv_heads, int head_dim) {
  if (num_heads < 1 || num_kv_heads < 1 || num_heads % num_kv_heads != 0) return KVS_ERR_DIMS;
  if (!head_dim_supported(head_dim)) return KVS_ERR_UNSUPPORTED;
  if (num_heads / num_kv_heads > 8) return KVS_ERR_UNSUPPORTED;
  const int rc = kvs::prepare_step_kernel(num_heads, num_kv_heads, head_dim);
  if (rc != KVS_OK) return rc;
  return kvs::prepare_cluster_kernel(num_heads, num_kv_heads, head_dim);
}

}  // extern "C"
