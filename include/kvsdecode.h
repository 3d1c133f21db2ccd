/*
 * kvsdecode.h -- C ABI of the GB300 (sm_103a) batched decode-step attention
 * library: KV-cache scatter followed by split-K ("flash decoding") softmax
 * attention under grouped-query attention.
 *
 * Source of the operations: realizar 0.8.5, src/cuda/executor/head_dim.rs,
 * `flash_decoding_attention_into` (PAR-118) -- doc comment (layouts; the KV
 * cache is cut into chunks processed in parallel, whose partial results are
 * merged with softmax rescaling), "Step 1: Scatter K/V to caches", "Update
 * cache lengths" (a sequence at position p attends rows 0..p), "Step 3:
 * Compute max chunks needed" (ceil(seq_len / chunk)), "Step 4" (chunk
 * kernel), "Step 5" (reduce kernel).  The device-resident position follows
 * aprender-serve 0.70.2, src/gguf/cuda/forward_qwen35_cuda_graph.rs, module
 * doc table (the K/V row is "scattered at *io.pos", read on the device).
 *
 * Conventions shared by every entry point
 *   - All tensors are float32, C-contiguous, in DEVICE memory owned by the
 *     caller; positions are int32 in device memory.  (kvs_decode_step_host
 *     is the exception: its inputs and result are in host memory.)  The
 *     library never allocates, frees or synchronises; it does not keep
 *     pointers after a call returns.
 *   - Layouts (M sequences, H = num_heads query heads, Hkv = num_kv_heads,
 *     G = H / Hkv, D = head_dim, Lmax = max_len):
 *         q, out              [M][H][D]
 *         k_rows, v_rows      [M][Hkv][D]          (this step's new rows)
 *         k_cache, v_cache    [M][Hkv][Lmax][D]    (sequence stride Hkv*Lmax*D)
 *         positions           [M]                  (int32)
 *     Query head h reads kv head h / G (contiguous groups).  The softmax
 *     scale is 1/sqrt(D).
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream) and returns; kernels run asynchronously.
 *     Ordering between calls is the stream's.  kvs_kv_scatter must be
 *     ordered before kvs_flash_decode of the same layer: attention includes
 *     row p, the row the scatter writes.
 *   - Return value: KVS_OK, or a kvs_status code.  Argument errors are
 *     detected on the host BEFORE anything is enqueued.  KVS_ERR_LAUNCH
 *     carries a CUDA launch failure.
 *   - d_status (nullable): a device int the caller zeroes.  Kernels record
 *     the first device-detected error there (atomic compare-and-swap from
 *     0): KVS_ERR_POSITION for a position outside [0, Lmax) (that sequence
 *     is skipped; the scatter writes nothing for it and its attention
 *     output rows are NaN), KVS_ERR_TIMEOUT if an internal pipeline wait
 *     exceeded its bound (the kernel returns instead of hanging; outputs
 *     of that call are undefined, nothing outside them is written, and the
 *     context stays usable).
 *   - State: a call keeps nothing of its arguments.  Two process-wide
 *     settings do apply to every call: the kernel schedule
 *     (kvs_set_schedule; which attention kernel a call runs) and, per
 *     device, the wait bound (kvs_set_wait_limit_ns).  A change made on
 *     one host thread applies to the calls that other threads make from
 *     then on.  Otherwise the entry points may be called from several host
 *     threads on different streams (with separate workspaces).
 */
#ifndef KVSDECODE_H
#define KVSDECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvs_status {
  KVS_OK = 0,
  KVS_ERR_NULL = 1,        /* a required pointer is NULL */
  KVS_ERR_DIMS = 2,        /* M < 0, H % Hkv != 0, sizes < 1, chunk_size < 0 */
  KVS_ERR_UNSUPPORTED = 3, /* head_dim not 64 or 128, or H / Hkv > 8 */
  KVS_ERR_ALIGN = 4,       /* a tensor pointer is not 16-byte aligned */
  KVS_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than required */
  KVS_ERR_LAUNCH = 6,      /* CUDA reported a launch or device-query error */
  KVS_ERR_POSITION = 7,    /* device: a position outside [0, max_len) */
  KVS_ERR_TIMEOUT = 8,     /* device: a bounded pipeline wait expired */
  KVS_ERR_SLOT = 9,        /* device: a cache slot outside [0, num_slots) */
  KVS_ERR_MEMORY = 10      /* the device could not provide memory the library
                              itself holds (kvs_flash_decode_static) */
} kvs_status;

/* A cudaStream_t, passed as an opaque pointer so this header needs no CUDA
 * include. */
typedef void *kvs_stream_t;

/*
 * kvs_kv_scatter -- "Step 1: Scatter K/V to caches" of
 * flash_decoding_attention_into, done for all M sequences, both K and V,
 * in ONE launch (the pages launch it twice per sequence).
 *
 * For every sequence i with 0 <= p = positions[i] < max_len and every kv
 * head g:  k_cache[i][g][p][:] = k_rows[i][g][:],  v_cache likewise.
 * No other cache byte is touched; the copy is bit-exact.
 *
 *   k_rows, v_rows    in   [M][Hkv][D] float32, device, 16-byte aligned
 *   positions         in   [M] int32, device
 *   k_cache, v_cache  out  [M][Hkv][Lmax][D] float32, device, 16-byte aligned
 *   M >= 0 (0: nothing enqueued), num_kv_heads >= 1, head_dim in {64, 128},
 *   max_len >= 1.
 * Errors: NULL, DIMS, UNSUPPORTED, ALIGN, LAUNCH on the host; POSITION via
 * d_status.
 */
int kvs_kv_scatter(const float *k_rows, const float *v_rows,
                   const int32_t *positions, float *k_cache, float *v_cache,
                   int M, int num_kv_heads, int head_dim, int max_len,
                   int *d_status, kvs_stream_t stream);

/*
 * kvs_choose_chunk_size -- the chunk size used when a caller passes
 * chunk_size = 0 (the pages fix one compile-time FLASH_DECODE_CHUNK_SIZE).
 *
 * On the pages the chunk size also fixes the split count: a sequence of L
 * rows gets ceil(L / chunk) chunks, each one block of the chunk kernel.
 * Here the split is made separately: the persistent kernel cuts the live
 * rows of the whole batch, read from the device positions at run time,
 * into equal columns, one per resident block (2 per SM), so the number of
 * pieces a sequence is split into follows from its length and the batch,
 * whatever the chunk size.  Chunks are only the granule of that cut: a
 * block's range starts and ends on chunk boundaries, and partials are kept
 * per run of chunks, not per chunk.  So the rule depends on the SM count
 * and the cache size (not on positions, which the host does not read).
 * With r = M * num_kv_heads * max_len / (2 * SMs) cache rows per block
 * (integer division) it returns 16 for r < 4096, 32 for r < 8192, else 64.
 * Returns a chunk size in rows (>= 1), or a negative kvs_status.
 *   num_sms > 0: use that SM count; num_sms <= 0: query the current device.
 */
int kvs_choose_chunk_size(int M, int num_kv_heads, int head_dim, int max_len,
                          int num_sms);

/*
 * kvs_flash_decode_workspace_bytes -- size of the scratch buffer that
 * kvs_flash_decode needs: the softmax partials (running max, running sum and
 * weighted-V accumulator; the pages' flash_decode_partials buffer), kept
 * for each run of consecutive chunks one block of the chunk kernel handles,
 * plus a small table of the blocks' ranges.  The size depends on M,
 * num_heads, num_kv_heads and head_dim only (max_len and chunk_size are
 * validated, not used).  Returns 0 on invalid arguments.
 */
size_t kvs_flash_decode_workspace_bytes(int M, int num_heads, int num_kv_heads,
                                        int head_dim, int max_len,
                                        int chunk_size);

/*
 * kvs_flash_decode -- "Step 3" to "Step 5" of flash_decoding_attention_into:
 * split-K decode attention over the scattered cache, in one kernel launch.
 *
 * For every sequence i (L = positions[i] + 1) and query head h (kv head
 * g = h / G):  out[i][h][:] = softmax_j( q[i][h] . k_cache[i][g][j] / sqrt(D) )
 * applied to v_cache[i][g][j][:], j = 0..L-1.  Rows j >= L are never read.
 *
 Two schedules compute this (see kvs_set_schedule); both read each K/V
 * row once for all G query heads of its group, and both return the same
 * attention up to float rounding:
 *  - persistent: the cache rows of every (sequence, kv head) are cut into
 *    chunks of chunk_size rows, processed in parallel by a persistent grid;
 *    each chunk yields (running max, running sum, weighted-V accumulator).
 *    Consecutive chunks of one (sequence, kv head) handled by the same
 *    block merge as they stream; the block that completes a (sequence, kv
 *    head) merges its partials with softmax rescaling through the
 *    workspace and writes the output.
 *  - cluster (small steps): one thread-block cluster of up to 16 blocks per
 *    (sequence, kv head); block r takes rows [L*r/CS, L*(r+1)/CS) and the
 *    partials are merged with the same rescaling in distributed shared
 *    memory.  chunk_size and the workspace are validated but not used.
 *
 *   q          in   [M][H][D] float32, device, 16-byte aligned
 *   k_cache,
 *   v_cache    in   [M][Hkv][Lmax][D] float32, device, 16-byte aligned
 *   positions  in   [M] int32, device
 *   out        out  [M][H][D] float32, device, 16-byte aligned
 *   chunk_size      rows per chunk; 0 = kvs_choose_chunk_size
 *   workspace       device scratch of >= kvs_flash_decode_workspace_bytes
 *                   bytes, 256-byte aligned; contents need no initialisation
 *                   and are overwritten; it must not be shared by calls
 *                   that can overlap on the GPU.  Its first 4 bytes are an
 *                   epoch that the completion counters' tags include; a
 *                   call that gives up on a wait (KVS_ERR_TIMEOUT) changes
 *                   it.  A CUDA graph that the caller captures around these
 *                   calls replays the same tags: after a replay that
 *                   reported KVS_ERR_TIMEOUT, zero the workspace before the
 *                   next replay (kvs_step_graph needs nothing: it writes a
 *                   fresh epoch at every replay).
 * Errors: NULL, DIMS, UNSUPPORTED, ALIGN, WORKSPACE, LAUNCH on the host;
 * POSITION, TIMEOUT via d_status.
 */
int kvs_flash_decode(const float *q, const float *k_cache,
                     const float *v_cache, const int32_t *positions,
                     float *out, int M, int num_heads, int num_kv_heads,
                     int head_dim, int max_len, int chunk_size,
                     void *workspace, size_t workspace_bytes, int *d_status,
                     kvs_stream_t stream);

/*
 * kvs_decode_step -- one whole decode step of the attention path: exactly
 * kvs_kv_scatter(k_rows, v_rows, positions, k_cache, v_cache) followed by
 * kvs_flash_decode(q, k_cache, v_cache, positions, out), in ONE kernel
 * launch (the pages' flash_decoding_attention_into, Steps 1-5).  The
 * attention reads row p of every sequence from k_rows / v_rows directly, so
 * it does not wait for the cache write.
 *
 *   k_rows, v_rows    in   [M][Hkv][D] float32, device, 16-byte aligned
 *   k_cache, v_cache  in/out [M][Hkv][Lmax][D]: row p of each sequence is
 *                     written; rows 0..p-1 are read
 *   other arguments, layouts and errors: as kvs_kv_scatter and
 *   kvs_flash_decode (one workspace of kvs_flash_decode_workspace_bytes).
 */
int kvs_decode_step(const float *q, const float *k_rows, const float *v_rows,
                    const int32_t *positions, float *k_cache, float *v_cache,
                    float *out, int M, int num_heads, int num_kv_heads,
                    int head_dim, int max_len, int chunk_size, void *workspace,
                    size_t workspace_bytes, int *d_status, kvs_stream_t stream);

/*
 * kvs_decode_step_host -- kvs_decode_step with the step's inputs and its
 * result in HOST memory: the caller's whole step (host -> device copies of
 * q, k_rows, v_rows and positions, the fused scatter + attention launch, the
 * device -> host copy of out) in one call, all enqueued on `stream` in that
 * order.  The pages' step starts from device tensors; this entry point adds
 * the transfers a host-side caller makes around it.
 *
 *   q          in   [M][H][D] float32, host
 *   k_rows, v_rows  in  [M][Hkv][D] float32, host
 *   positions  in   [M] int32, host
 *   out        out  [M][H][D] float32, host: valid once `stream` has
 *                   reached the end of the call (synchronise it first)
 *   io         device scratch of >= kvs_step_io_bytes(M, H, Hkv, D) bytes,
 *              256-byte aligned, owned by the caller: the device copies of
 *              the inputs and of out; must not be shared by calls that can
 *              overlap on the GPU
 *   k_cache, v_cache, workspace, d_status: device, as kvs_decode_step.
 * Host buffers in pinned memory (cudaHostAlloc / cudaHostRegister) give
 * asynchronous copies, and must then stay untouched until the stream has
 * passed them; pageable host memory works, with copies that block the host.
 * Errors: as kvs_decode_step, plus NULL (a host pointer or io), ALIGN (io),
 * WORKSPACE (io_bytes too small), LAUNCH (a copy could not be enqueued).
 */
size_t kvs_step_io_bytes(int M, int num_heads, int num_kv_heads, int head_dim);

int kvs_decode_step_host(const float *q, const float *k_rows,
                         const float *v_rows, const int32_t *positions,
                         float *k_cache, float *v_cache, float *out, int M,
                         int num_heads, int num_kv_heads, int head_dim,
                         int max_len, int chunk_size, void *io, size_t io_bytes,
                         void *workspace, size_t workspace_bytes,
                         int *d_status, kvs_stream_t stream);

/*
 * kvs_step_io_layout -- where each array sits in a buffer of
 * kvs_step_io_bytes(M, H, Hkv, D) bytes: offsets[0..4] receive the byte
 * offsets of q, k_rows, v_rows, positions and out (each 256-byte aligned,
 * in that order), offsets[5] the total size.  The device io buffer of
 * kvs_decode_step_host and kvs_decode_step_host_io has this layout, and so
 * has the host buffer of kvs_decode_step_host_io.
 *   offsets  out  size_t[6], host
 * Errors: DIMS (a size < 1), NULL.
 */
int kvs_step_io_layout(int M, int num_heads, int num_kv_heads, int head_dim, size_t *offsets);

/*
 * kvs_decode_step_host_io -- kvs_decode_step_host for a caller that keeps
 * the step's inputs and result in ONE host buffer laid out like the device
 * io buffer (kvs_step_io_layout): q, k_rows, v_rows and positions at their
 * offsets go to the device in one host -> device copy (the padding between
 * them included), and out comes back to its offset in one device -> host
 * copy; in between, the fused scatter + attention launch.  All three are
 * enqueued on `stream` in that order.  When host_io is pinned memory the GPU
 * can address (cudaHostAlloc / cudaHostRegister), the two copies are
 * kernels of this library (every SM moves a share over the host link, far
 * faster than one copy engine at these sizes); otherwise they are
 * cudaMemcpyAsync calls, which for pageable memory block the host.
 *
 *   host_io  in/out  host buffer of >= kvs_step_io_bytes bytes with that
 *                    layout; the inputs must stay untouched, and out is
 *                    valid, once `stream` has passed the call
 *   io, k_cache, v_cache, workspace, d_status, other arguments: as
 *   kvs_decode_step_host.
 * Errors: as kvs_decode_step_host.
 */
int kvs_decode_step_host_io(void *host_io, float *k_cache, float *v_cache, int M,
                            int num_heads, int num_kv_heads, int head_dim, int max_len,
                            int chunk_size, void *io, size_t io_bytes, void *workspace,
                            size_t workspace_bytes, int *d_status, kvs_stream_t stream);

/*
 * kvs_decode_step_slots -- kvs_decode_step for a serving batch whose
 * sequences live in arbitrary slots of a cache pool, some of them finished
 * (the pages' "Step 2: Build pointer arrays": a per-sequence cache pointer
 * for non-contiguous slots and mid-batch joins, and PMAT-076: a finished
 * slot gets seq_len 0 so the attention kernels skip it).
 *
 *   k_pool, v_pool  in/out [num_slots][Hkv][Lmax][D] float32, device,
 *                   16-byte aligned: the cache pool
 *   slots           in  [M] int32, device, or NULL (sequence i uses slot i;
 *                   then num_slots >= M): the pool slot of each sequence.
 *                   Slots are indices, so the kernels can check them: one
 *                   outside [0, num_slots) is KVS_ERR_SLOT via d_status, and
 *                   that sequence is neither scattered nor attended (its out
 *                   rows are NaN unless it is finished).  Two sequences must
 *                   not share a slot (they would race).
 *   done            in  [M] uint8, device, or NULL (none finished): nonzero
 *                   marks a finished sequence.  As on the pages, its new
 *                   row is still scattered, but no attention runs for it and
 *                   its out rows are left exactly as they were.
 *   k_rows, v_rows  in  [M][Hkv][D], or both NULL: attention only, no scatter
 *   q, out, positions, chunk_size, workspace, d_status, stream: as
 *   kvs_decode_step (one workspace of kvs_flash_decode_workspace_bytes for
 *   M sequences; the pool size does not change it).
 * Errors: DIMS (also num_slots < 1, or slots NULL with num_slots < M), NULL
 * (one of k_rows / v_rows NULL), ALIGN, UNSUPPORTED, WORKSPACE, LAUNCH on the
 * host; POSITION, SLOT, TIMEOUT via d_status.
 */
int kvs_decode_step_slots(const float *q, const float *k_rows,
                          const float *v_rows, const int32_t *positions,
                          const int32_t *slots, const uint8_t *done,
                          float *k_pool, float *v_pool, int num_slots,
                          float *out, int M, int num_heads, int num_kv_heads,
                          int head_dim, int max_len, int chunk_size,
                          void *workspace, size_t workspace_bytes,
                          int *d_status, kvs_stream_t stream);

/*
 * CUDA graph of a whole multi-layer decode step (the pages' graphed decode:
 * realizar 0.8.5 batched_forward.rs / reduces.rs capture and replay, and
 * aprender-serve 0.70.2 forward_qwen35_cuda_graph.rs, module doc: one graph
 * launch replays every layer; per-token inputs live at fixed device
 * addresses that the host rewrites before each replay).
 *
 * kvs_step_graph_create captures, on `stream` (not the legacy default
 * stream; it must not be capturing already), one kvs_decode_step per layer
 * l = 0..layers-1 with q[l], k_rows[l], v_rows[l], k_cache[l], v_cache[l],
 * out[l] (host arrays of `layers` device pointers) and the shared
 * `positions`, `workspace` (one buffer serves all layers: the layers run in
 * order) and `d_status`.  Capture uses the thread-local mode and is always
 * ended; on any error nothing is kept and the status is returned (the
 * caller can stay on the eager path).  Every pointer is frozen into the
 * graph: update the buffers' contents, never their addresses, between
 * launches.  The graph and its executable are CUDA objects owned by the
 * handle; the library allocates no device memory.
 * Inside the graph, each layer after the first starts before the layer
 * ahead of it has finished: it reads `positions` and streams its cache rows
 * below the positions while that layer runs, and reads q, the new rows and
 * row p only after it.  So no layer's out may overlap `positions` or any
 * layer's caches (the library's own writes, row p of each cache, never
 * overlap what a later layer reads early).
 *
 * kvs_step_graph_launch enqueues the whole step on `stream`.  The graph
 * starts with a 4-byte write of a fresh value to the workspace epoch (see
 * kvs_flash_decode), so a replay after one that timed out is clean.  One
 * handle is launched by one host thread at a time (a lock inside orders
 * concurrent launches).
 * kvs_step_graph_destroy releases the handle (NULL is a no-op).
 */
typedef struct kvs_step_graph kvs_step_graph;

int kvs_step_graph_create(int layers, const float *const *q,
                          const float *const *k_rows,
                          const float *const *v_rows, const int32_t *positions,
                          float *const *k_cache, float *const *v_cache,
                          float *const *out, int M, int num_heads,
                          int num_kv_heads, int head_dim, int max_len,
                          int chunk_size, void *workspace,
                          size_t workspace_bytes, int *d_status,
                          kvs_stream_t stream, kvs_step_graph **graph);

/*
 * kvs_step_graph_io_layout -- the layout of one buffer holding a whole
 * step's inputs and results for kvs_step_graph_create_host_io: the inputs
 * first (q, k_rows, v_rows of layer 0, then of layer 1, ..., then the
 * positions, shared by the layers), then the results (out of layer 0, 1,
 * ...), each array 256-byte aligned, with the shapes of kvs_decode_step.
 *   offsets  out  size_t[4 * layers + 2], host: offsets[3l], [3l + 1],
 *                 [3l + 2] = q, k_rows, v_rows of layer l; [3 layers] =
 *                 positions; [3 layers + 1 + l] = out of layer l (the inputs
 *                 end at [3 layers + 1]); [4 layers + 1] = the total size.
 * Errors: DIMS (a size < 1), NULL.
 */
int kvs_step_graph_io_layout(int layers, int M, int num_heads, int num_kv_heads, int head_dim,
                             size_t *offsets);

/*
 * kvs_step_graph_create_host_io -- kvs_step_graph_create for a step whose
 * per-token inputs and results live in ONE pinned host buffer (the pages'
 * graphed decode: inputs at fixed addresses that the host rewrites before
 * each launch).  The graph copies every layer's inputs and the positions to
 * the device buffer `io` (the same layout) in one copy, runs the layers from
 * there (fused scatter + attention, as kvs_step_graph_create), and copies
 * every layer's out back in one copy.  The copies are kernels of this
 * library moving the bytes over the host link.
 *   host_io   in/out  host buffer of >= the layout's total size, pinned and
 *                     addressable by the GPU (cudaHostAlloc /
 *                     cudaHostRegister; other memory: UNSUPPORTED).  Write
 *                     the inputs before a launch; the outs are valid once
 *                     `stream` has passed it.
 *   io        scratch device buffer of >= the total size, 256-byte aligned
 *   k_cache, v_cache, M, num_heads, num_kv_heads, head_dim, max_len,
 *   chunk_size, workspace, d_status, stream, graph: as kvs_step_graph_create
 *   (k_cache, v_cache: host arrays of `layers` device pointers).
 * Errors: NULL, DIMS, ALIGN (io), WORKSPACE (io_bytes), UNSUPPORTED (host_io
 * not pinned), and those of kvs_step_graph_create.
 */
int kvs_step_graph_create_host_io(int layers, void *host_io, void *io, size_t io_bytes,
                                  float *const *k_cache, float *const *v_cache, int M,
                                  int num_heads, int num_kv_heads, int head_dim, int max_len,
                                  int chunk_size, void *workspace, size_t workspace_bytes,
                                  int *d_status, kvs_stream_t stream, kvs_step_graph **graph);

int kvs_step_graph_launch(kvs_step_graph *graph, kvs_stream_t stream);

int kvs_step_graph_destroy(kvs_step_graph *graph);

/*
 * kvs_flash_decode_static -- kvs_flash_decode for callers that cannot
 * allocate device memory (no counterpart in the pages: they always hand the
 * kernels a preallocated partials buffer).
 *
 * Who needs it: code that may not call cudaMalloc at the point where it runs
 * attention -- a process under a fixed device-memory budget that forbids
 * allocation after start-up, a plug-in host that lends streams and tensors
 * but no allocator, or a runtime whose own allocator must not be re-entered
 * from inside this call.  This entry point takes only inputs and outputs
 * and allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine).
 *
 * Scratch: the chunk partials go to one buffer of KVS_STATIC_WORKSPACE_BYTES
 * compiled into the library as a device array.  Every GPU on which the
 * library's device code is loaded holds that buffer until the process
 * exits.  Problems whose partials need more
 * (kvs_flash_decode_workspace_bytes(...) > KVS_STATIC_WORKSPACE_BYTES)
 * are rejected with KVS_ERR_WORKSPACE before anything is enqueued, whatever
 * kernel the schedule would pick for them (the cluster kernel needs no
 * scratch, but the size rule does not look at the schedule); use
 * kvs_flash_decode with your own workspace for those.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the buffer's device address.  CUDA loads device code lazily, so that
 * first call is also when the device commits the 32 MiB: a caller under a
 * fixed memory budget should make one call at start-up, while it may still
 * allocate.  If the device cannot provide the buffer then, the call returns
 * KVS_ERR_MEMORY (other set-up failures: KVS_ERR_LAUNCH).  Make that first
 * call before any stream capture on that device.  The address is kept for
 * the life of the process: after cudaDeviceReset (or anything else that
 * destroys the device's primary context) do not call this entry point
 * again on that device.
 *
 * Sharing: all calls on a device use the same buffer, which keeps whatever
 * the last call left in it.  Nothing in it has to start at zero (each call
 * writes every partial it later reads), but calls that can overlap on the
 * GPU -- different streams without ordering between them, or different
 * host threads -- race on the buffer and give wrong results.  Order such
 * calls on one stream or with events.
 *
 * Arguments, layouts and the other errors: exactly as kvs_flash_decode.
 */
#define KVS_STATIC_WORKSPACE_BYTES (32u * 1024u * 1024u)

int kvs_flash_decode_static(const float *q, const float *k_cache,
                            const float *v_cache, const int32_t *positions,
                            float *out, int M, int num_heads, int num_kv_heads,
                            int head_dim, int max_len, int chunk_size,
                            int *d_status, kvs_stream_t stream);

/*
 * kvs_argmax -- batched greedy token selection (realizar 0.8.5, reduces.rs,
 * gpu_argmax PAR-062 / batched_gpu_argmax PMAT-045: the token ID with the
 * largest logit for each of M logit vectors, computed on the GPU so that
 * only the IDs need to leave it), in ONE launch for all rows.
 *
 *   logits     in   [M][vocab_size] float32, device, 4-byte aligned
 *                   (16-byte aligned rows are read with 16-byte loads)
 *   token_ids  out  [M] int32, device
 * token_ids[m] is the smallest index j with logits[m][j] equal to the row's
 * largest value; NaN entries are never chosen; a row with no value above
 * -inf gives 0.  The result is enqueued on `stream`; copy it to the host
 * with one cudaMemcpyAsync and one synchronisation for the whole batch.
 * Errors: DIMS (M < 0, vocab_size < 1), NULL, ALIGN, LAUNCH.  M = 0 enqueues
 * nothing.
 */
int kvs_argmax(const float *logits, int M, int vocab_size, int32_t *token_ids,
               kvs_stream_t stream);

/*
 * kvs_prefill_attention -- softmax attention over whole sequences on the
 * tensor cores (realizar 0.8.5, head_dim.rs, tensor_core_attention,
 * PARITY-001.3: FP32 inputs converted to FP16 on the GPU, Q K^T and P V as
 * tensor-core products, FP32 output, optional causal mask).
 *
 *   q, k, v  in   [num_heads][seq_len][head_dim] float32, device, 16-byte aligned
 *   out      out  [num_heads][seq_len][head_dim] float32, device, 16-byte aligned
 * out[h][i] = softmax_j(q[h][i] . k[h][j] / sqrt(head_dim)) v[h][j] over
 * j = 0..seq_len-1, or j = 0..i when causal != 0.  q, k and v are rounded to
 * FP16 (round to nearest even); scores, the softmax and the output
 * accumulate in FP32; the probabilities are rounded to FP16 before the P V
 * product (the row sum adds them in FP32).  head_dim must be 64 or 128; any seq_len >= 1 (the pages require
 * a multiple of 16; here the last tile is masked).
 *   workspace  device scratch of >= kvs_prefill_workspace_bytes bytes,
 *              256-byte aligned: a 4-byte ready flag per tile and a task
 *              counter (3 * num_heads * T + 1 words, T = ceil(seq_len/128),
 *              padded to a multiple of 256 bytes), then q, k and v as FP16
 *              tiles in the tensor-core layout (3 * num_heads * T * 128 *
 *              head_dim * 2 bytes); no initialisation needed (the call
 *              zeroes the flags); must not be shared by calls that can
 *              overlap on the GPU.
 * Enqueued: a memset of the flags, an FP16 pack launch for the tiles needed
 * first, then the attention launch, whose pack warps convert the remaining
 * tiles while it runs.
 * Errors: DIMS (negative sizes, num_heads > 65535, seq_len > 65535 * 128),
 * UNSUPPORTED (head_dim not 64 or 128; more than 2^30 tiles), NULL, ALIGN,
 * WORKSPACE, LAUNCH on the host; TIMEOUT via
 * d_status.  num_heads = 0 or seq_len = 0 enqueues nothing.
 */
size_t kvs_prefill_workspace_bytes(int num_heads, int seq_len, int head_dim);

int kvs_prefill_attention(const float *q, const float *k, const float *v,
                          float *out, int num_heads, int seq_len, int head_dim,
                          int causal, void *workspace, size_t workspace_bytes,
                          int *d_status, kvs_stream_t stream);

/*
 * Kernel schedule of kvs_flash_decode, kvs_decode_step (and so of the
 * graphs and the static entry point), process-wide:
 *   KVS_SCHEDULE_AUTO        (the default) the cluster kernel for steps
 *                            bound by latency rather than bandwidth: the
 *                            K/V bytes of full caches (M * num_kv_heads *
 *                            max_len * head_dim * 8) at most 64 MiB, every
 *                            cluster of the launch resident at once on the
 *                            current device, and each block's slice of a
 *                            full cache at most 512 KiB; else the
 *                            persistent kernel;
 *   KVS_SCHEDULE_PERSISTENT  always the persistent kernel;
 *   KVS_SCHEDULE_CLUSTER     the cluster kernel whenever M * num_kv_heads
 *                            <= 65535.
 * kvs_set_schedule returns the previous schedule, or -KVS_ERR_DIMS for an
 * unknown value (nothing changes).  The schedule is read when a call is
 * made (a captured graph keeps the kernel chosen at capture).
 */
typedef enum kvs_schedule {
  KVS_SCHEDULE_AUTO = 0,
  KVS_SCHEDULE_PERSISTENT = 1,
  KVS_SCHEDULE_CLUSTER = 2
} kvs_schedule;

int kvs_set_schedule(int schedule);
int kvs_get_schedule(void);

/* The kernel a call with these sizes would run on the current device under
 * the schedule in force: KVS_SCHEDULE_PERSISTENT or KVS_SCHEDULE_CLUSTER, or
 * a negative kvs_status (DIMS, UNSUPPORTED).  Without a usable device the
 * automatic schedule answers KVS_SCHEDULE_PERSISTENT. */
int kvs_schedule_for(int M, int num_heads, int num_kv_heads, int head_dim,
                     int max_len);

/*
 * kvs_set_wait_limit_ns -- the bound on each pipeline wait of this
 * library's kernels on the current device (default
 * KVS_WAIT_LIMIT_DEFAULT_NS = 2 s).  A wait that runs past it makes its
 * kernel record KVS_ERR_TIMEOUT in d_status and return instead of waiting
 * on; at the default only a fault could take that long.  Lowering the bound
 * makes waits run out on purpose, so that a caller can test its handling of
 * KVS_ERR_TIMEOUT.  Calls made while the bound is below the default launch
 * a variant of each kernel whose waits poll without sleeping and compare
 * against the bound at every poll (0 ends the first wait that does not find
 * its data ready); calls at the default launch the kernels whose waits
 * sleep in the hardware wait and carry no such test.  A CUDA graph keeps
 * the variant its capture launched: one captured under a lowered bound
 * reads the bound in force at each replay.  Whatever the bound, a block
 * that gives up still lets every copy and tensor-core product it issued
 * finish before it exits (those waits keep 2 s), and leaves the context
 * usable.  The value applies to every host thread's calls on that device;
 * set it back when done.  The call synchronises with the device like
 * cudaMemcpyToSymbol; it must not be made during a stream capture.
 *   ns        0 .. KVS_WAIT_LIMIT_DEFAULT_NS, else KVS_ERR_DIMS
 *   previous  nullable: receives the bound in force before the call
 * Errors: DIMS, LAUNCH.
 */
#define KVS_WAIT_LIMIT_DEFAULT_NS 2000000000ull

int kvs_set_wait_limit_ns(uint64_t ns, uint64_t *previous);

/*
 * kvs_prepare -- sets up, on the current device, both attention kernels
 * for (num_heads, num_kv_heads, head_dim): shared-memory attributes and the
 * largest cluster size the device can co-schedule.  Every entry point does
 * this on first use; call it first when the first attention call will be
 * made under stream capture.  Errors: DIMS, UNSUPPORTED, LAUNCH.
 */
int kvs_prepare(int num_heads, int num_kv_heads, int head_dim);

/* Human-readable name of a kvs_status value (static string). */
const char *kvs_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* KVSDECODE_H */
