// fd_cluster.cu -- the decode-step attention for small steps: one thread-block
// cluster per (sequence, kv head), the split-K partials merged through
// distributed shared memory.
//
// Source: realizar 0.8.5, src/cuda/executor/head_dim.rs,
// flash_decoding_attention_into (PAR-118): doc comment (split the KV cache
// into chunks processed in parallel, then merge the partial results with
// softmax rescaling), "Step 1: Scatter K/V to caches" and "Step 4" / "Step 5"
// (chunk and reduce kernels).
//
// Why a second kernel: when a step moves only a few MB (a small model, short
// caches) the persistent kernel is bound by latency, not bandwidth, and most
// of that latency is its global-memory merge protocol -- partial stores, a
// fence, a counter atomic, then the merging block's loads, each a round trip
// through L2.  Here the CS blocks that share one (i, g) form a cluster:
//  * block r of the cluster streams rows [L*r/CS, L*(r+1)/CS) of (i, g)
//    with the same warp-specialised pipeline and consumer tile as the
//    persistent kernel (bulk async copies into a ring of stages);
//  * each block stores its partial (m, l, acc for the G heads), element by
//    element, into the shared memory of the block that merges each share of
//    the output (distributed shared memory); one cluster barrier makes the
//    stores visible, and each block merges its share from its own shared
//    memory and writes it.  No block reads another's memory, so the blocks
//    may exit after that one barrier.
// No workspace, no atomics, no global round trip between the partials and
// the merge.  The fused scatter works as in the persistent kernel: the last
// block of the cluster writes the new rows, and the stage holding row p
// takes it from the new rows.  Inside a step graph, a layer after the first
// streams its cache rows before its dependency wait (SeqArgs::early).
//
// Every thread of every block arrives at the entry barrier, waits on it
// before its first remote store, and passes the merge barrier on every path
// (the only early exit, a bad position or a finished sequence, is taken by
// the whole cluster before any wait), and every mbarrier wait is bounded in
// time, so a lost copy ends in KVS_ERR_TIMEOUT, never in a hang.

#include <cmath>
#include <mutex>

#include "fd_tile.cuh"
#include "kvs_cluster.cuh"
#include "kvs_device.cuh"
#include "kvs_launch.h"

namespace kvs {

namespace {

constexpr int kMaxClusterDevices = 64;
constexpr int kMaxClusterSize = 16;  // the largest cluster launched

// Block geometry: four consumer warps, two blocks per SM, as in the
// persistent kernel, but each warp folds up to four sub-tiles per stage, the
// most whose ring still fits two blocks per SM.  A block's slice is a few
// dozen to a few hundred rows, so the stages it walks one after another,
// each a chain of shared-memory, shuffle and exponential latencies, set its
// time, not the bytes: more rows per stage means fewer chains.  Measured on
// GB300 (small model layer: M=4, 14 heads over 2 kv heads, head_dim 64):
// 9.6 us a layer with one sub-tile, 8.2 with four; eight consumer warps at
// one block per SM were slower (fewer clusters resident at once), and seven
// consumer warps with two sub-tiles each (two blocks per SM at 128
// registers) no faster than four with four.  The running max is taken with
// shuffles (SHFL_MAX): 185.6 -> 176.5 us for that model's 24-layer step.
template <int D, int G>
constexpr int cluster_nsub() {
  return Geo<D, G, 4, 2, 4, true>::FITS ? 4 : Geo<D, G, 4, 2, 2, true>::FITS ? 2 : 1;
}
template <int D, int G>
using ClusterGeo = Geo<D, G, 4, 2, cluster_nsub<D, G>(), true>;

template <int D, int G, bool kPoll>
__global__ void __launch_bounds__(ClusterGeo<D, G>::THREADS, ClusterGeo<D, G>::MINB)
    fd_cluster_kernel(const float *__restrict__ q, float *k_cache, float *v_cache, SeqMap sm,
                      const float *__restrict__ k_rows, const float *__restrict__ v_rows,
                      float *__restrict__ out, int Hkv, float qscale, int *d_status,
                      int early) {
  using C = ClusterGeo<D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  StageDesc *desc = reinterpret_cast<StageDesc *>(smem + C::OFF_DESC);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::S;
  volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
  // The partials this block merges, written here by every block of the
  // cluster (itself included) before the cluster barrier: element j of this
  // block's share (chunk = E / CS elements) from block r at
  // recv_acc[r * chunk + j], the (m, l) of head h from block r at
  // recv_ml[r * G + h].  They use the q slots of ring stages 1 and 2: the
  // consumer warps of this kernel load q straight into registers, so no
  // copy ever lands in a q slot and nothing else reads them.
  constexpr int E = G * C::LPR;  // output float4s of one (i, g)
  static_assert(C::FITS, "two blocks per SM must fit");
  static_assert(C::S >= 3, "the receive areas need ring stages 1 and 2");
  static_assert(E % kMaxClusterSize == 0, "every cluster size divides the output");
  static_assert(E * 16 <= C::Q_BYTES && kMaxClusterSize * G * 8 <= C::Q_BYTES,
                "the receive areas fit the q slots");
  float4 *recv_acc = reinterpret_cast<float4 *>(smem + C::STAGE_BYTES + 2 * C::KV_BYTES);
  float2 *recv_ml = reinterpret_cast<float2 *>(smem + 2 * C::STAGE_BYTES + 2 * C::KV_BYTES);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // grid (CS, M*Hkv), clusters of (CS, 1, 1): one cluster per (i, g)
  const uint32_t rank = cluster_rank();
  const int ncl = (int)gridDim.x;
  const int ig = blockIdx.y;
  const int i = ig / Hkv;
  const int g = ig - i * Hkv;
  const int H = Hkv * G;
  const bool scatter = (k_rows != nullptr);

  // Every block of the cluster has started once this barrier completes;
  // it is waited on before the first store into another block's memory.
  cluster_arrive_relaxed();
  // The ring's barriers live in shared memory only: set them up while the
  // previous kernel in the stream may still be finishing.
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NW);
    }
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Without `early`, everything below may read what the preceding kernel in
  // the stream writes: wait for it first.  With `early` (a layer of a step
  // graph after the first), positions, slots, finished flags and the cache
  // rows below each position are not written by the preceding kernel, so
  // they are read, and the first stages' cache rows streamed, before the
  // wait; q, the new rows, the caches' row p, the output and the status
  // come after it.
  if (!early) grid_dependency_wait();
  // sequence i (coherent loads: with `early` the preceding kernel may still
  // be resident, and nothing it wrote may be served from a stale L1 line)
  const int p = __ldcg(sm.pos + i);
  const int slot = sm.slot ? __ldcg(sm.slot + i) : i;
  const bool finished = sm.done && __ldcg(sm.done + i) != 0;
  const int err = (p < 0 || p >= sm.max_len)                           ? KVS_ERR_POSITION
                  : (sm.slot && (slot < 0 || slot >= sm.num_slots)) ? KVS_ERR_SLOT
                                                                     : KVS_OK;
  // rows of (i, g): the first row of its cache, and its new row
  const size_t head_base = ((size_t)slot * Hkv + g) * (size_t)sm.max_len;
  const size_t row_src = ((size_t)i * Hkv + g) * D;
  // Step 1, scatter: the block holding row p writes the new rows (a finished
  // sequence too; none for a bad position or slot).  Threads [t0, t0 + nt).
  auto scatter_rows = [&](int t0, int nt) {
    if (!scatter || err != KVS_OK || rank != (uint32_t)(ncl - 1)) return;
    constexpr int D4 = D / 4;
    const size_t dst = (head_base + p) * D4;
    const size_t src = row_src / 4;
    for (int e = (int)threadIdx.x - t0; e < 2 * D4; e += nt) {
      if (e < D4)
        reinterpret_cast<float4 *>(k_cache)[dst + e] =
            __ldcg(reinterpret_cast<const float4 *>(k_rows) + src + e);
      else
        reinterpret_cast<float4 *>(v_cache)[dst + e - D4] =
            __ldcg(reinterpret_cast<const float4 *>(v_rows) + src + e - D4);
    }
  };
  // The whole cluster leaves here (its blocks share i) before any wait on a
  // cluster barrier and before any remote store; it has only arrived at the
  // entry barrier, which no thread then waits on.
  if (err != KVS_OK || finished) {
    grid_dependency_wait();
    scatter_rows(0, C::THREADS);
    if (err != KVS_OK && rank == 0) {
      if (!finished) {  // a finished sequence's output is left as it is
        const float nan = __int_as_float(0x7fc00000);
        float4 *o4 = reinterpret_cast<float4 *>(out) + ((size_t)i * H + (size_t)g * G) * (D / 4);
        for (int e = threadIdx.x; e < G * (D / 4); e += C::THREADS)
          o4[e] = make_float4(nan, nan, nan, nan);
      }
      if (threadIdx.x == 0) record_status(d_status, err);
    }
    return;
  }
  const int L = p + 1;
  const int r0 = (int)((long long)L * rank / ncl);
  const int r1 = (int)((long long)L * (rank + 1) / ncl);

  if (warp == C::NW) {
    // ===================== producer warp (lane 0 issues) ====================
    if (lane != 0) {
      grid_dependency_wait();
      allow_dependent_launch();
    } else {
      const uint64_t pol_stream = policy_evict_first();
      int ok = 1;
      const int nst = (r1 - r0 + C::T - 1) / C::T;  // stages of the block's rows
      // Stage k in two parts: its cache rows (with the descriptor and the
      // barrier's byte count for the whole stage), and what the preceding
      // kernel may write -- the new rows, with the stage holding row p.
      // The byte count keeps the stage incomplete until both parts have
      // landed.  (q goes straight to the consumers' registers.)
      auto issue_cache_part = [&](uint32_t k) {
        const uint32_t s = k % C::S;
        const int rs = r0 + (int)k * C::T;
        const int nrows = min(C::T, r1 - rs);
        StageDesc &dd = desc[s];
        dd.flags = (k == 0 ? kRunStart : 0) | (rs + C::T >= r1 ? kRunEnd : 0);
        dd.nrows = nrows;
        const uint32_t kv_bytes = (uint32_t)nrows * D * 4;
        mbar_arrive_expect_tx(&full[s], 2 * kv_bytes);
        // with the scatter folded in, row L-1 (position p) comes from the new rows
        const bool tail = scatter && (rs + nrows == L);
        const uint32_t cache_bytes = tail ? kv_bytes - D * 4 : kv_bytes;
        if (cache_bytes > 0) {
          unsigned char *stage = smem + s * C::STAGE_BYTES;
          const size_t row0 = (head_base + rs) * D;
          bulk_g2s_hint(stage, k_cache + row0, cache_bytes, &full[s], pol_stream);
          bulk_g2s_hint(stage + C::KV_BYTES, v_cache + row0, cache_bytes, &full[s], pol_stream);
        }
      };
      auto issue_input_part = [&](uint32_t k) {
        const uint32_t s = k % C::S;
        const int rs = r0 + (int)k * C::T;
        const int nrows = min(C::T, r1 - rs);
        unsigned char *stage = smem + s * C::STAGE_BYTES;
        if (scatter && rs + nrows == L) {
          const uint32_t cache_bytes = (uint32_t)(nrows - 1) * D * 4;
          bulk_g2s(stage + cache_bytes, k_rows + row_src, D * 4, &full[s]);
          bulk_g2s(stage + C::KV_BYTES + cache_bytes, v_rows + row_src, D * 4, &full[s]);
        }
      };
      // Every ring slot is fresh for its first use: the first S stages need
      // no wait for a free slot.
      const uint32_t npre = early ? (uint32_t)min(nst, C::S) : 0u;
      for (uint32_t k = 0; k < npre; ++k) issue_cache_part(k);
      grid_dependency_wait();
      allow_dependent_launch();
      for (uint32_t k = 0; k < npre; ++k) issue_input_part(k);
      uint32_t k = npre;
      for (; k < (uint32_t)nst; ++k) {
        const uint32_t s = k % C::S;
        const uint32_t use = k / C::S;
        if (!mbar_wait<kPoll>(&empty[s], (use & 1u) ^ 1u, abort)) {
          ok = 0;
          break;
        }
        issue_cache_part(k);
        issue_input_part(k);
      }
      // Copies of uses below `first_live` have landed: the consumers
      // released those stages before the producer's last successful wait.
      uint32_t first_live = k > (uint32_t)C::S ? k - C::S : 0u;
      if (ok) {  // tell the consumers there is nothing more
        const uint32_t s = k % C::S;
        const uint32_t use = k / C::S;
        if (mbar_wait<kPoll>(&empty[s], (use & 1u) ^ 1u, abort)) {
          desc[s].flags = kNoMore;
          desc[s].nrows = 0;
          mbar_arrive(&full[s]);
          first_live = k + 1 > (uint32_t)C::S ? k + 1 - C::S : 0u;
        } else {
          ok = 0;
        }
      }
      if (!ok) {
        *abort = 1;
        record_status(d_status, KVS_ERR_TIMEOUT);
      }
      // Every copy this block issued lands before the block goes on, also
      // when a consumer warp gave up and no longer waits for it.  (The
      // latest use of each ring slot is in [first_live, k), so each wait is
      // for that use's phase.)
      for (uint32_t j = first_live; j < k; ++j) mbar_wait_drain(&full[j % C::S], (j / C::S) & 1u);
    }
    __syncwarp();
    cluster_wait();  // the split barrier of the kernel entry
  } else {
    // ===================== consumer warps ===================================
    grid_dependency_wait();
    // q of the group, the lane's float4 column, straight from global memory
    // (coherent loads: the preceding kernel may have written it), scaled as
    // the stage math wants it (log2(e)/sqrt(D), base-2 softmax)
    const TileLane<C> tl = tile_lane<C>(smem, warp, lane);
    float4 qv[G];
    {
      const float4 *q4 = reinterpret_cast<const float4 *>(q) +
                         ((size_t)i * H + (size_t)g * G) * C::LPR + tl.li;
      float4 v[G];
#pragma unroll
      for (int h = 0; h < G; ++h) v[h] = __ldcg(q4 + h * C::LPR);
#pragma unroll
      for (int h = 0; h < G; ++h)
        qv[h] = make_float4(v[h].x * qscale, v[h].y * qscale, v[h].z * qscale, v[h].w * qscale);
    }
    allow_dependent_launch();
    scatter_rows(0, C::NW * 32);
    float4 acc[G];
    float m_run[G];
    float l_lane;
    tile_reset<G>(acc, m_run, l_lane);
    for (uint32_t k = 0;; ++k) {
      const uint32_t s = k % C::S;
      const uint32_t use = k / C::S;
      // all lanes of the warp leave together (shuffles follow)
      if (!__all_sync(0xffffffffu, mbar_wait<kPoll>(&full[s], use & 1u, abort))) {
        if (lane == 0) {
          *abort = 1;
          record_status(d_status, KVS_ERR_TIMEOUT);
        }
        break;
      }
      const StageDesc dsc = desc[s];
      if (dsc.flags & kNoMore) break;
      const unsigned char *stage = smem + s * C::STAGE_BYTES;
      tile_consume<C>(tl, stage, dsc.nrows, qv, acc, m_run, l_lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // A block with no rows publishes m = -inf, l = 0, acc = 0.
    tile_publish<C>(tl, acc, m_run, l_lane);
    consumer_sync(C::NW * 32);
    // The block's partial, element by element, into the shared memory of
    // the block that merges it (remote stores: nothing waits for them here),
    // once every block of the cluster has started.
    cluster_wait();
    const int chunk = E / ncl;
    for (int e = threadIdx.x; e < E; e += C::NW * 32) {
      float4 a;
      float mx, lsum;
      merged_warp_states<C>(smem, e, a, mx, lsum);
      const int dst = e / chunk;
      st_dsmem_f4(dsmem_addr(&recv_acc[rank * chunk + (e - dst * chunk)], dst), a);
      if (e % C::LPR == 0) {  // (m, l) of head h to every block merging part of it
        const int h = e / C::LPR;
        const int d_last = (e + C::LPR - 1) / chunk;
        for (int d = dst; d <= d_last; ++d)
          st_dsmem_f2(dsmem_addr(&recv_ml[rank * G + h], d), make_float2(mx, lsum));
      }
    }
  }

  cluster_sync_all();  // every partial is in the shared memory of the block merging it
  if (warp < C::NW) {
    // Block r merges elements [r * chunk, (r + 1) * chunk) from its own
    // shared memory and writes that share of the output.  Element j takes
    // ncl consecutive lanes, lane rr holding block rr's partial; max and
    // sums go over those lanes by shuffles (ncl is a power of two <= 16 and
    // divides E, so an element's lanes lie in one warp and are all active
    // or all idle).
    const int chunk = E / ncl;
    for (int base = warp * 32; base < E; base += C::NW * 32) {
      const int t = base + lane;
      const bool act = t < E;
      const int j = t / ncl;
      const int rr = t - j * ncl;
      const int e = (int)rank * chunk + j;
      const int h = e / C::LPR;
      const float2 ml = act ? recv_ml[rr * G + h] : make_float2(neg_inf(), 0.f);
      const float4 b = act ? recv_acc[rr * chunk + j] : make_float4(0.f, 0.f, 0.f, 0.f);
      float mx = ml.x;
      for (int o = 1; o < ncl; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float w = (ml.x == neg_inf()) ? 0.f : exp2f(ml.x - mx);
      float4 a = make_float4(w * b.x, w * b.y, w * b.z, w * b.w);
      float l = w * ml.y;
      for (int o = 1; o < ncl; o <<= 1) {
        a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
        a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
        a.z += __shfl_xor_sync(0xffffffffu, a.z, o);
        a.w += __shfl_xor_sync(0xffffffffu, a.w, o);
        l += __shfl_xor_sync(0xffffffffu, l, o);
      }
      if (act && rr == 0) {
        const float inv = 1.f / l;
        reinterpret_cast<float4 *>(out)[((size_t)i * H + (size_t)g * G) * C::LPR + e] =
            make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
      }
    }
  }
  // No block reads another's shared memory after the barrier, and every
  // remote store came before it: the blocks may exit now.
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
// Target rows per block: a block's slice should be a few stages, so that the
// cluster's blocks finish together soon after their first copies land.
constexpr int kClusterRowsPerBlock = 32;

constexpr int kClusterSizes = 5;  // 1, 2, 4, 8, 16

struct ClusterInfo {
  int max_size = 0;
  int active[kClusterSizes] = {0};  // clusters of size 2^k resident at once
  bool configured = false;
};

// Cluster size for a cache of max_len rows, given the largest launchable.
inline int cluster_size_for(int max_len, int cs_max) {
  int cs = 1;
  while (cs < cs_max && (long long)cs * kClusterRowsPerBlock < max_len) cs <<= 1;
  return cs;
}

// Configures this instantiation on device `dev` on first use and returns its
// record: the largest cluster size (a power of two <= 16) it can be launched
// with, and how many clusters of each size the device keeps resident.
template <int D, int G>
const ClusterInfo *cluster_info(int dev) {
  using C = ClusterGeo<D, G>;
  static ClusterInfo info[kMaxClusterDevices];
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (!info[dev].configured) {
    auto kern = fd_cluster_kernel<D, G, false>;
    int top = 16;
    // both wait variants have the same shared memory and launch bounds
    for (auto k : {fd_cluster_kernel<D, G, false>, fd_cluster_kernel<D, G, true>}) {
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
          cudaSuccess) {
        cudaGetLastError();
        return nullptr;
      }
      cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
          cudaSuccess) {
        cudaGetLastError();
        top = 8;
      }
    }
    ClusterInfo rec;
    for (int k = 0, cs = 1; cs <= top; ++k, cs <<= 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(cs, 1, 1);
      cfg.blockDim = dim3(C::THREADS, 1, 1);
      cfg.dynamicSmemBytes = C::SMEM_BYTES;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
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

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxClusterDevices) return -1;
  return dev;
}

template <int D, int G>
int launch_cluster_impl(const float *q, float *k_cache, float *v_cache, const SeqArgs &seqs,
                        const float *k_rows, const float *v_rows, float *out, int M, int Hkv,
                        int *d_status, cudaStream_t stream) {
  const int max_len = seqs.max_len;
  using C = ClusterGeo<D, G>;
  const int dev = current_device();
  if (dev < 0) return KVS_ERR_LAUNCH;
  const ClusterInfo *ci = cluster_info<D, G>(dev);
  if (!ci) return KVS_ERR_LAUNCH;
  const long long pairs = (long long)M * Hkv;
  if (pairs > kMaxClusterPairs) return KVS_ERR_UNSUPPORTED;
  const int cs = cluster_size_for(max_len, ci->max_size);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, (unsigned)pairs, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
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
  const float qscale = (float)(1.4426950408889634074 / std::sqrt((double)D));
  const SeqMap sm{seqs.positions, seqs.slots, seqs.done, max_len, seqs.num_slots, Hkv};
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, poll_waits() ? fd_cluster_kernel<D, G, true> : fd_cluster_kernel<D, G, false>, q,
      k_cache, v_cache, sm, k_rows, v_rows, out, Hkv, qscale, d_status, seqs.early ? 1 : 0);
  if (e != cudaSuccess) {
    cudaGetLastError();  // leave no stale error for the caller's next check
    return KVS_ERR_LAUNCH;
  }
  return KVS_OK;
}

template <int D>
int cluster_dispatch(int G, const float *q, float *k_cache, float *v_cache,
                     const SeqArgs &seqs, const float *k_rows, const float *v_rows,
                     float *out, int M, int Hkv, int *d_status, cudaStream_t stream) {
  switch (G) {
#define KVS_CASE(g)                                                                            \
  case g:                                                                                      \
    return launch_cluster_impl<D, g>(q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, Hkv, \
                                     d_status, stream);
    KVS_CASE(1)
    KVS_CASE(2)
    KVS_CASE(3)
    KVS_CASE(4)
    KVS_CASE(5)
    KVS_CASE(6)
    KVS_CASE(7)
    KVS_CASE(8)
#undef KVS_CASE
    default:
      return KVS_ERR_UNSUPPORTED;
  }
}

}  // namespace

int set_wait_limit_cluster(uint64_t ns) {
  if (set_unit_wait_limit(ns) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  return KVS_OK;
}

int prepare_cluster_kernel(int H, int Hkv, int D) {
  const int dev = current_device();
  if (dev < 0) return KVS_ERR_LAUNCH;
  if (Hkv < 1 || H % Hkv != 0) return KVS_ERR_DIMS;
  const int G = H / Hkv;
  const ClusterInfo *ci = nullptr;
  switch (D * 16 + G) {
#define KVS_PREP(d, g)                     \
  case d * 16 + g:                         \
    ci = cluster_info<d, g>(dev);          \
    break;
    KVS_PREP(64, 1) KVS_PREP(64, 2) KVS_PREP(64, 3) KVS_PREP(64, 4)
    KVS_PREP(64, 5) KVS_PREP(64, 6) KVS_PREP(64, 7) KVS_PREP(64, 8)
    KVS_PREP(128, 1) KVS_PREP(128, 2) KVS_PREP(128, 3) KVS_PREP(128, 4)
    KVS_PREP(128, 5) KVS_PREP(128, 6) KVS_PREP(128, 7) KVS_PREP(128, 8)
#undef KVS_PREP
    default:
      return KVS_ERR_UNSUPPORTED;
  }
  return ci ? KVS_OK : KVS_ERR_LAUNCH;
}

// Whether the automatic schedule should take the cluster kernel: every
// cluster of the launch resident at once (one wave), and each block's slice
// of a full cache at most kClusterAutoSliceBytes.  Measured on GB300: the
// cluster kernel wins on a few (sequence, kv head) pairs with short slices
// (a small model's 8 pairs: 12 us against 18 us a layer), and loses once
// its clusters need a second wave.
int cluster_auto_ok(int M, int H, int Hkv, int D, int max_len) {
  constexpr long long kClusterAutoSliceBytes = 512ll << 10;
  const int dev = current_device();
  if (dev < 0 || Hkv < 1 || H % Hkv != 0) return 0;
  const int G = H / Hkv;
  const ClusterInfo *ci = nullptr;
  switch (D * 16 + G) {
#define KVS_INFO(d, g)                     \
  case d * 16 + g:                         \
    ci = cluster_info<d, g>(dev);          \
    break;
    KVS_INFO(64, 1) KVS_INFO(64, 2) KVS_INFO(64, 3) KVS_INFO(64, 4)
    KVS_INFO(64, 5) KVS_INFO(64, 6) KVS_INFO(64, 7) KVS_INFO(64, 8)
    KVS_INFO(128, 1) KVS_INFO(128, 2) KVS_INFO(128, 3) KVS_INFO(128, 4)
    KVS_INFO(128, 5) KVS_INFO(128, 6) KVS_INFO(128, 7) KVS_INFO(128, 8)
#undef KVS_INFO
    default:
      return 0;
  }
  if (!ci) return 0;
  const int cs = cluster_size_for(max_len, ci->max_size);
  int k = 0;
  while ((1 << k) < cs) ++k;
  const long long pairs = (long long)M * Hkv;
  const long long slice_bytes = ((long long)max_len + cs - 1) / cs * D * 8;
  return pairs <= ci->active[k] && slice_bytes <= kClusterAutoSliceBytes;
}

int launch_fd_cluster(const float *q, float *k_cache, float *v_cache, const SeqArgs &seqs,
                      const float *k_rows, const float *v_rows, float *out, int M, int H,
                      int Hkv, int D, int *d_status, cudaStream_t stream) {
  const int G = H / Hkv;
  if (D == 128)
    return cluster_dispatch<128>(G, q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, Hkv,
                                 d_status, stream);
  if (D == 64)
    return cluster_dispatch<64>(G, q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, Hkv,
                                d_status, stream);
  return KVS_ERR_UNSUPPORTED;
}

}  // namespace kvs
