// flash_decode.cu -- the decode-step attention kernel for sm_103a: split-K
// flash decoding in ONE persistent kernel per call (split plan, chunk
// partials, rescaled merge), optionally with the KV-cache scatter of the
// same step folded in.
//
// Source: realizar 0.8.5, src/cuda/executor/head_dim.rs,
// flash_decoding_attention_into (PAR-118): doc comment (split the KV cache
// into chunks processed in parallel, then merge the partial results with
// softmax rescaling), "Step 1: Scatter K/V to caches", "Step 3: Compute max
// chunks needed" (a sequence of length L has ceil(L / chunk) chunks), "Step
// 4" (chunk kernel, one 32-thread block per (query head, sequence, chunk))
// and "Step 5" (reduce kernel, one block per (query head, sequence)).
//
// GB300 design (what differs from the pages):
//  * Scheduling atom = chunk (sequence i, kv head g, chunk c) of `chunk`
//    cache rows, ordered (i, g, c).  One chunk serves all G = H/Hkv query
//    heads of its group, so every K/V byte leaves HBM once per call (the
//    pages' per-query-head blocks read each row G times).
//  * Persistent grid of P blocks (#SMs x blocks per SM).  The live (i, g),
//    in (i, g) order, are laid out in a "cost row" space where (i, g) takes
//    L + cost rows (cost = the fixed price of a run, ~40 KB of K+V rows).
//    That space is cut into P equal columns; block b takes the chunks that
//    start in column b, so blocks get equal rows plus run overheads even when
//    many sequences are short.  Lengths and columns are derived on the device
//    from the device-resident positions.
//  * A block merges consecutive chunks of one (i, g) on the fly (its
//    online-softmax state just continues) and writes one partial per run:
//    the run that starts at chunk 0 of (i, g) owns slot i*Hkv + g; a block's
//    first run, when it starts inside (i, g), owns slot M*Hkv + b.
//  * Merge without a second kernel: every run adds its row count to a
//    per-(i, g) counter; the block whose run completes the L rows of (i, g)
//    merges all of (i, g)'s runs (found from the same column arithmetic) and
//    writes the output.  A (i, g) covered by a single run is written
//    directly.  The counters carry the tag of the call that last used them,
//    so the workspace needs no initialisation, and the merging block resets
//    its counter, so replaying a captured graph (same tag) is safe too.
//  * Scatter folded in (kvs_decode_step): blocks first write the step's new
//    K/V rows into the caches; the attention reads row p of each sequence
//    from the new-row input itself, so no block waits for another.
//  * Warp-specialised block: the producer warp computes the block's range and
//    one of its lanes streams each run's K and V rows (contiguous ranges of the
//    [Lmax][D] layout) and the group's q rows into a ring of shared-memory
//    stages with 1-D bulk asynchronous copies (TMA, cp.async.bulk + mbarrier
//    transaction counts), writing a small descriptor per stage.  NW consumer
//    warps follow the descriptors.  Every wait is bounded in time.
//  * Consumer warp tile: RW rows x G heads.  Lanes split head_dim (one
//    float4 per lane per row); q for the G heads lives in registers,
//    pre-multiplied by log2(e)/sqrt(D) so the softmax runs in base 2.  The
//    RW*G partial dot products are reduced with a transposing butterfly
//    (each shuffle level halves the values a lane holds), leaving one score
//    per lane.  Per tile and head: tile max -> running max, rescale factor,
//    exp2 of the lane's own score, then P.V with float4 reads of V.
//  * Launched with programmatic stream serialisation: it waits
//    (griddepcontrol.wait) before touching global memory, so its launch
//    overlaps the tail of the previous kernel in the stream.
//
// Partial semantics (per query head, run R of rows):
//   m = max_{j in R} s_j,  l = sum exp2(s_j - m),  acc = sum exp2(s_j - m) v_j,
//   s_j = log2(e) q.k_j / sqrt(D).
// Merge: M* = max m,  out = sum 2^(m - M*) acc / sum 2^(m - M*) l.

#include <atomic>
#include <chrono>
#include <cmath>
#include <mutex>

#include "kvs_device.cuh"
#include "kvs_launch.h"
#include "fd_tile.cuh"

namespace kvs {

namespace {

// Fixed price of one run, in bytes of K+V rows: it sets the `cost` rows that
// each (i, g) adds to the balanced split (40 rows at D = 128, 80 at D = 64).
constexpr int kRunCostBytes = 40960;


// ---------------------------------------------------------------------------
// Split plan on the device (warp-cooperative; every lane returns the result)
//
// Work is balanced in a "cost row" space: (i, g) occupies L + cost rows --
// `cost` rows that stand for the fixed price of a run (its start, the merge
// of the warp states, the partial or output write) followed by its L cache
// rows; chunk c of (i, g) starts at cost row V + cost + c*chunk, where V is
// the first cost row of (i, g).  The live (i, g) follow each other in
// (i, g) order.  Sequences with L = 0 occupy nothing.
// ---------------------------------------------------------------------------
struct SplitTotals {
  long long rows;   // sum_i Hkv * (L_i + cost) over live sequences
  long long units;  // sum_i Hkv * ceil(L_i / chunk)
};

__device__ SplitTotals warp_split_totals(const SeqMap &sm, int M, int Hkv, int chunk, int cost,
                                         int lane) {
  long long rows = 0, units = 0;
  for (int i = lane; i < M; i += 32) {
    const int L = sm.len(i);
    if (L > 0) rows += (long long)Hkv * (L + cost);
    units += (long long)Hkv * ((L + chunk - 1) / chunk);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    rows += __shfl_xor_sync(0xffffffffu, rows, o);
    units += __shfl_xor_sync(0xffffffffu, units, o);
  }
  return {rows, units};
}

// a / b for a >= 0, b > 0: a 32-bit division when both fit (the 64-bit one
// is a long instruction sequence, on the path to a block's first copy)
__device__ __forceinline__ long long div_nn(long long a, long long b) {
  if (((a | b) >> 31) == 0) return (long long)((unsigned)a / (unsigned)b);
  return a / b;
}

// A block's share of the plan: the chunks it runs, [ub, ue) -- the first
// chunk that starts at or after cost row t0, and the first at or after t1
// (total_units past the end) -- and, for ub, the (i, g, c) the cost row t0
// falls in with the first cost row of sequence i.  c == n (the chunk count
// of sequence i) means ub is chunk 0 of the (i, g) after (i, g).  One
// warp-cooperative pass over the sequences; every lane returns the result.
struct BlockPlan {
  long long ub, ue;
  int i, g, c;
  long long seq_row0;
};

__device__ BlockPlan warp_block_plan(long long t0, long long t1, const SeqMap &sm, int M,
                                     int Hkv, int chunk, int cost, long long total_units,
                                     int lane) {
  BlockPlan p{total_units, total_units, M, 0, 0, 0};
  bool have0 = false, have1 = false;
  long long row_base = 0, unit_base = 0;
  for (int i0 = 0; i0 < M && !(have0 && have1); i0 += 32) {
    const int i = i0 + lane;
    const int L = (i < M) ? sm.len(i) : 0;
    const int n = (L + chunk - 1) / chunk;
    const long long rows = (L > 0) ? (long long)Hkv * (L + cost) : 0;
    const long long units = (long long)Hkv * n;
    long long rinc = rows, uinc = units;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long a = __shfl_up_sync(0xffffffffu, rinc, o);
      const long long b = __shfl_up_sync(0xffffffffu, uinc, o);
      if (lane >= o) {
        rinc += a;
        uinc += b;
      }
    }
    const long long rexcl = row_base + rinc - rows;  // first cost row of sequence i
    const long long uexcl = unit_base + uinc - units;
    const long long span = (long long)L + cost;  // cost rows of one (i, g)
    // the first chunk of sequence i's rows starting at or after cost row t
    auto chunk_at = [&](long long t, int &g, int &c) {
      const long long off = t - rexcl;
      g = (int)div_nn(off, span);
      const long long r = off - (long long)g * span - cost;  // offset from chunk 0's start
      c = (r <= 0) ? 0 : (int)div_nn(r + chunk - 1, chunk);
      return uexcl + (long long)g * n + c;
    };
    if (!have0) {
      const bool hit = rows > 0 && t0 >= rexcl && t0 < rexcl + rows;
      int g = 0, c = 0;
      long long u = 0;
      if (hit) u = chunk_at(t0, g, c);
      const unsigned ballot = __ballot_sync(0xffffffffu, hit);
      if (ballot) {
        const int src = __ffs(ballot) - 1;
        p.ub = __shfl_sync(0xffffffffu, u, src);
        p.i = i0 + src;
        p.g = __shfl_sync(0xffffffffu, g, src);
        p.c = __shfl_sync(0xffffffffu, c, src);
        p.seq_row0 = __shfl_sync(0xffffffffu, rexcl, src);
        have0 = true;
      }
    }
    if (!have1) {
      const bool hit = rows > 0 && t1 >= rexcl && t1 < rexcl + rows;
      int g = 0, c = 0;
      long long u = 0;
      if (hit) u = chunk_at(t1, g, c);
      const unsigned ballot = __ballot_sync(0xffffffffu, hit);
      if (ballot) {
        p.ue = __shfl_sync(0xffffffffu, u, __ffs(ballot) - 1);
        have1 = true;
      }
    }
    row_base += __shfl_sync(0xffffffffu, rinc, 31);
    unit_base += __shfl_sync(0xffffffffu, uinc, 31);
  }
  return p;
}

// ---------------------------------------------------------------------------
// Columns: block b owns the chunks that start in cost rows [R*b/P, R*(b+1)/P).
// ---------------------------------------------------------------------------
__device__ __forceinline__ long long column_start_row(long long R, int P, int b) {
  return R * b / P;
}

// Column holding cost row r (0 <= r < R): the largest b with R*b/P <= r.
__device__ __forceinline__ int column_of_row(long long r, long long R, int P) {
  const long long c = (r * P + P - 1) / R;
  return (int)(c < P - 1 ? c : P - 1);
}

// Counters tagged with the call that last used them: the value is
// (tag << 32 | count).  A value left by another call (another tag, or
// whatever the workspace held) counts as zero: the first adder of this call
// replaces it with (tag, amount).  Each returns the count before the add.
// Bounded: after 2^20 failed attempts they record KVS_ERR_TIMEOUT and return
// 0xffffffff.  `v` is what an atomicAdd(ctr, amount) returned.
__device__ unsigned resolve_tagged_add(unsigned long long *ctr, unsigned long long v,
                                       unsigned amount, unsigned tag, int *d_status,
                                       unsigned *epoch) {
  for (int attempt = 0; attempt < (1 << 20); ++attempt) {
    if ((unsigned)(v >> 32) == tag) return (unsigned)v;
    const unsigned long long cur = v + amount;
    const unsigned long long mine = ((unsigned long long)tag << 32) | amount;
    const unsigned long long prev = atomicCAS(ctr, cur, mine);
    if (prev == cur) return 0u;
    if ((unsigned)(prev >> 32) == tag)
      v = atomicAdd(ctr, (unsigned long long)amount);
    else
      v = prev - amount;
  }
  record_status(d_status, KVS_ERR_TIMEOUT);
  atomicAdd(epoch, 1u);
  return 0xffffffffu;
}

__device__ __forceinline__ unsigned tagged_add(unsigned long long *ctr, unsigned amount,
                                               unsigned tag, int *d_status, unsigned *epoch) {
  return resolve_tagged_add(ctr, atomicAdd(ctr, (unsigned long long)amount), amount, tag,
                            d_status, epoch);
}

// The tag this launch's counters carry: the host's per-launch tag combined
// with the workspace epoch.  Every block of a launch reads the same epoch
// (nothing changes it unless a block gives up), so every block computes the
// same tag.  A launch that gives up changes the epoch, so the counts it
// leaves can never be taken for a later launch's own, not even by a replayed
// graph, whose host tag is frozen at capture.  Never 0: a reset counter
// holds tag 0.
__device__ __forceinline__ unsigned launch_tag(unsigned host_tag, unsigned epoch) {
  const unsigned t = host_tag ^ (epoch * 0x9E3779B1u);
  return t != 0u ? t : 0x5BD1E995u;
}

// A block gives up the call: stop every role of the block, report it, and
// move the workspace epoch on (see launch_tag).
__device__ __forceinline__ void give_up(volatile int *abort, int *d_status, unsigned *epoch) {
  *abort = 1;
  record_status(d_status, KVS_ERR_TIMEOUT);
  atomicAdd(epoch, 1u);
}


// A run: consecutive chunks of one (i, g) inside a block's range.
struct Run {
  int i, g, c;  // first chunk of the run
  int L, n;     // sequence length, chunks of the sequence
  int units;    // chunks in the run
};

__device__ __forceinline__ Run make_run(int i, int g, int c, long long remaining,
                                        const SeqMap &sm, int chunk) {
  Run r;
  r.i = i;
  r.g = g;
  r.c = c;
  r.L = sm.len(i);
  r.n = (r.L + chunk - 1) / chunk;
  r.units = (int)min((long long)(r.n - c), remaining);
  return r;
}

// The run after `r` (called only while chunks remain): next kv head of the
// sequence, else the next sequence that has rows.  Never reads past M-1; if
// the list ended (it cannot when the piece came from the same positions) the
// run is empty (units = 0), which ends the loops.
__device__ __forceinline__ Run next_run(const Run &r, long long remaining, const SeqMap &sm,
                                        int M, int Hkv, int chunk) {
  if (r.g + 1 < Hkv) return make_run(r.i, r.g + 1, 0, remaining, sm, chunk);
  for (int i = r.i + 1; i < M; ++i) {
    if (sm.len(i) > 0)
      return make_run(i, 0, 0, remaining, sm, chunk);
  }
  Run e = r;
  e.units = 0;
  e.L = 0;
  return e;
}

// ---------------------------------------------------------------------------
// Merge of all runs of one (i, g), by the NW consumer warps of the block
// whose run completed (i, g).  Runs: the one at chunk 0 (slot i*Hkv + g) and,
// for every chunk cc > 0 at which a block's range starts, that block's first
// run (slot M*Hkv + block; of several blocks starting at the same chunk only
// the last has work).  Candidate blocks come in row order, so the runs do
// too and the sums are taken in a fixed order.
//
// One pass with a running maximum, as in the chunk loop itself: each thread
// owns (query head, float4 column) outputs and takes the runs in batches of
// MB, issuing all of a batch's loads -- (m, l) and accumulator -- before it
// uses any, so a batch costs one L2 round trip.
// ---------------------------------------------------------------------------
template <int D, int G, int NW>
__device__ __noinline__ void merge_runs(const WsView &ws, float *out, int i, int g, int M, int Hkv,
                           long long S, int L, long long R, int P, int chunk, int cost,
                           unsigned char *scratch) {
  constexpr int LPR = D / 4;
  constexpr int NT = NW * 32;
  constexpr int NE = (G * LPR + NT - 1) / NT;
  constexpr int MB = merge_batch(G) / NE;  // NE * MB loads in flight per thread
  int *s_list = reinterpret_cast<int *>(scratch);  // [kMergeWindow]
  int *s_n = s_list + kMergeWindow;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int H = Hkv * G;
  const int n = (L + chunk - 1) / chunk;
  const long long c0 = S + cost;  // cost row where chunk 0 of (i, g) starts
  // candidate blocks: those whose range may start at a chunk cc in (0, n)
  const int b_lo = (L >= 2) ? column_of_row(c0 + 1, R, P) : 0;
  const int b_hi = (L >= 2) ? column_of_row(c0 + L - 1, R, P) : -1;
  const int ncand = b_hi - b_lo + 1;
  auto cand_chunk = [&](int j) -> int {  // chunk where block b_lo + j starts, or -1
    const long long r = column_start_row(R, P, b_lo + j) - c0;
    if (r <= 0 || r >= L) return -1;
    const int cc = (int)((r + chunk - 1) / chunk);
    return cc < n ? cc : -1;
  };
  auto run_slot = [&](int j) -> int {  // j = -1: the chunk-0 run; else -1 if not a run
    if (j < 0) return i * Hkv + g;
    const int cc = cand_chunk(j);
    if (cc < 0) return -1;
    if (j + 1 < ncand && cand_chunk(j + 1) == cc) return -1;  // an empty block; the next starts here
    return M * Hkv + b_lo + j;
  };

  const float4 *acc4 = reinterpret_cast<const float4 *>(ws.acc);
  float4 a[NE];
  float mq[NE], lq[NE];
#pragma unroll
  for (int q = 0; q < NE; ++q) {
    a[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    mq[q] = neg_inf();
    lq[q] = 0.f;
  }
  for (int base = -1; base < ncand; base += kMergeWindow) {
    if (t < 32) {  // this window's runs, compacted in order
      const int j = base + t;
      const int sl = (j < ncand) ? run_slot(j) : -1;
      const unsigned ballot = __ballot_sync(0xffffffffu, sl >= 0);
      if (sl >= 0) s_list[__popc(ballot & ((1u << lane) - 1u))] = sl;
      if (lane == 0) *s_n = __popc(ballot);
    }
    consumer_sync(NT);
    const int nb = *s_n;
    for (int r0 = 0; r0 < nb; r0 += MB) {
      const int nr = min(MB, nb - r0);
      float2 ml[NE][MB];
      float4 bb[NE][MB];
#pragma unroll
      for (int q = 0; q < NE; ++q) {
        const int e = min(t + q * NT, G * LPR - 1);  // a spare thread re-reads a valid slot
        const int h = e / LPR;
        const int d4 = e - h * LPR;
#pragma unroll
        for (int j = 0; j < MB; ++j) {
          if (j < nr) {
            const size_t sl = (size_t)s_list[r0 + j] * G + h;
            ml[q][j] = __ldcg(&ws.ml[sl]);
            bb[q][j] = __ldcg(&acc4[sl * LPR + d4]);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < NE; ++q) {
        float mb = mq[q];
#pragma unroll
        for (int j = 0; j < MB; ++j)
          if (j < nr) mb = fmaxf(mb, ml[q][j].x);
        const float sc = (mq[q] == neg_inf()) ? 0.f : exp2f(mq[q] - mb);
        float4 acc = make_float4(a[q].x * sc, a[q].y * sc, a[q].z * sc, a[q].w * sc);
        float l = lq[q] * sc;
#pragma unroll
        for (int j = 0; j < MB; ++j) {
          if (j < nr) {
            const float w = exp2f(ml[q][j].x - mb);
            acc.x = fmaf(w, bb[q][j].x, acc.x);
            acc.y = fmaf(w, bb[q][j].y, acc.y);
            acc.z = fmaf(w, bb[q][j].z, acc.z);
            acc.w = fmaf(w, bb[q][j].w, acc.w);
            l = fmaf(w, ml[q][j].y, l);
          }
        }
        a[q] = acc;
        lq[q] = l;
        mq[q] = mb;
      }
    }
    consumer_sync(NT);  // every thread has read the list before it is rewritten
  }
  float4 *o4 = reinterpret_cast<float4 *>(out) + ((size_t)i * H + (size_t)g * G) * LPR;
#pragma unroll
  for (int q = 0; q < NE; ++q) {
    const int e = t + q * NT;
    if (e < G * LPR) {
      const float inv = 1.f / lq[q];
      o4[e] = make_float4(a[q].x * inv, a[q].y * inv, a[q].z * inv, a[q].w * inv);
    }
  }
}

// ---------------------------------------------------------------------------
// The step kernel (k_rows == nullptr: attention only; else scatter + attention)
// ---------------------------------------------------------------------------
template <int D, int G, bool kPoll>
__global__ void __launch_bounds__(Geo<D, G>::THREADS, 2)
    fd_step_kernel(const float *__restrict__ q, float *k_cache, float *v_cache, SeqMap sm,
                   const float *__restrict__ k_rows, const float *__restrict__ v_rows,
                   float *__restrict__ out, WsView ws, int M, int Hkv, int chunk, float qscale,
                   unsigned host_tag, int *d_status) {
  using C = Geo<D, G>;
  static_assert(C::FITS, "two blocks per SM must fit");
  constexpr int kCost = kRunCostBytes / (8 * D);  // cost rows per (i, g)
  extern __shared__ __align__(128) unsigned char smem[];
  StageDesc *desc = reinterpret_cast<StageDesc *>(smem + C::OFF_DESC);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::S;
  uint64_t *mbar = empty + C::S;  // consumer warps: end-of-run steps
  long long *info = reinterpret_cast<long long *>(smem + C::OFF_INFO);  // R, U, tag
  volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
  volatile int *s_last = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = Hkv * G;
  const int P = gridDim.x;
  const bool scatter = (k_rows != nullptr);

  // Everything below reads inputs a previous kernel may have written, and
  // writes the caches, the workspace and the output a previous kernel may
  // still read.
  grid_dependency_wait();

  // ---- sequences with a bad position or slot: status, and NaN rows unless
  //      finished (a finished sequence's output is left as it is) ----
  for (int i = blockIdx.x; i < M; i += P) {
    const int err = sm.error(i);
    if (err != KVS_OK) {
      if (!sm.finished(i)) {
        const float nan = __int_as_float(0x7fc00000);
        float4 *o4 = reinterpret_cast<float4 *>(out) + (size_t)i * H * (D / 4);
        for (int e = threadIdx.x; e < H * (D / 4); e += C::THREADS)
          o4[e] = make_float4(nan, nan, nan, nan);
      }
      if (threadIdx.x == 0) record_status(d_status, err);
    }
  }
  // ---- Step 1, scatter: this block's share of the new rows (float4 each) ----
  if (scatter) {
    constexpr int D4 = D / 4;
    const long long per_cache = (long long)M * Hkv * D4;
    for (long long e = (long long)blockIdx.x * C::THREADS + threadIdx.x; e < 2 * per_cache;
         e += (long long)P * C::THREADS) {
      const bool is_v = e >= per_cache;
      const long long f = is_v ? e - per_cache : e;
      const long long ig = f / D4;
      const int i = (int)(ig / Hkv);
      if (sm.error(i) != KVS_OK) continue;
      const int p = __ldca(sm.pos + i);
      const size_t dst = sm.row_index(i, (int)(ig - (long long)i * Hkv), p) * D4 + (f - ig * D4);
      if (is_v)
        reinterpret_cast<float4 *>(v_cache)[dst] = __ldcg(reinterpret_cast<const float4 *>(v_rows) + f);
      else
        reinterpret_cast<float4 *>(k_cache)[dst] = __ldcg(reinterpret_cast<const float4 *>(k_rows) + f);
    }
  }

  if (warp == 0) {
    const unsigned epoch = (lane == 0) ? __ldcg(ws.epoch) : 0u;
    const SplitTotals tot = warp_split_totals(sm, M, Hkv, chunk, kCost, lane);
    if (lane == 0) {
      info[0] = tot.rows;
      info[1] = tot.units;
      info[2] = launch_tag(host_tag, epoch);
      for (int s = 0; s < C::S; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], C::NW);
      }
      mbar_init(mbar, C::NW);
      *abort = 0;
      *s_last = 0;
      fence_mbar_init();
    }
  }
  __syncthreads();
  allow_dependent_launch();
  const long long R = info[0], U = info[1];
  const unsigned tag = (unsigned)info[2];
  if (R == 0) return;

  if (warp == C::NW) {
    // ===================== producer warp =================================
    // The whole warp computes this block's range (the split-plan searches are
    // warp-cooperative); lane 0 issues the copies and writes descriptors.
    const uint64_t pol_stream = policy_evict_first();
    uint32_t k = 0;
    int ok = 1;
    const int b = blockIdx.x;
    // cost rows where columns b and b + 1 start: R * b / P with one 64-bit
    // division (R = qP + rem, so R * b / P = q * b + rem * b / P exactly)
    const long long cq = R / P;
    const long long crem = R - cq * P;
    const long long t0 = cq * b + (crem * b) / P;
    const long long t1 = cq * (b + 1) + (crem * (b + 1)) / P;
    const BlockPlan plan = warp_block_plan(t0, t1, sm, M, Hkv, chunk, kCost, U, lane);
    const long long ub = plan.ub, ue = plan.ue;
    if (ub < ue) {
      // (i, g, c) of chunk ub and the first cost row of sequence i
      int pi = plan.i, pg = plan.g, pc = plan.c;
      long long seq_row0 = plan.seq_row0;
      const int Lp = sm.len(pi);
      if (pc == (Lp + chunk - 1) / chunk) {  // chunk 0 of the (i, g) after (i, g)
        pc = 0;
        if (++pg == Hkv) {  // of the next live sequence, which starts where i ends
          pg = 0;
          seq_row0 += (long long)Hkv * (Lp + kCost);
          do {
            ++pi;
          } while (pi < M && sm.len(pi) == 0);
        }
      }
      const long long block_slot = (long long)M * Hkv + b;
      long long remaining = ue - ub;
      Run run = make_run(pi, pg, pc, remaining, sm, chunk);
      int run_seq = run.i;
      while (ok && remaining > 0 && run.units > 0) {
        if (run.i != run_seq) {  // moved to a later sequence: advance its first row
          for (int j = run_seq; j < run.i; ++j) {
            const int Lj = sm.len(j);
            if (Lj > 0) seq_row0 += (long long)Hkv * (Lj + kCost);
          }
          run_seq = run.i;
        }
        const long long slot = (run.c == 0) ? (long long)run.i * Hkv + run.g : block_slot;
        const int r0 = run.c * chunk;
        const int r1 = (int)min((long long)(run.c + run.units) * chunk, (long long)run.L);
        const size_t head_base = sm.row_index(run.i, run.g, 0);
        const size_t row_src = ((size_t)run.i * Hkv + run.g) * D;  // new row of (i, g)
        // k counts the uses issued: a failed wait leaves the loop before
        // the increment, so the drain below sees exactly the issued copies.
        for (int rs = r0, st = 0; rs < r1; rs += C::T, ++st, ++k) {
          if (lane == 0) {
            const uint32_t s = k % C::S;
            const uint32_t use = k / C::S;
            if (!mbar_wait<kPoll>(&empty[s], (use & 1u) ^ 1u, abort)) {
              ok = 0;
            } else {
              const int nrows = min(C::T, r1 - rs);
              StageDesc &dd = desc[s];
              dd.flags = (st == 0 ? kRunStart : 0) | (rs + C::T >= r1 ? kRunEnd : 0);
              dd.nrows = nrows;
              dd.ig = run.i * Hkv + run.g;
              dd.run_rows = r1 - r0;
              dd.L = run.L;
              dd.slot = slot;
              dd.S = seq_row0 + (long long)run.g * (run.L + kCost);
              const uint32_t kv_bytes = (uint32_t)nrows * D * 4;
              const uint32_t bytes = 2 * kv_bytes + (st == 0 ? (uint32_t)C::Q_BYTES : 0u);
              unsigned char *stage = smem + s * C::STAGE_BYTES;
              mbar_arrive_expect_tx(&full[s], bytes);
              const size_t row0 = (head_base + rs) * D;
              // with the scatter folded in, row L-1 (position p) comes from the new rows
              const bool tail = scatter && (rs + nrows == run.L);
              const uint32_t cache_bytes = tail ? kv_bytes - D * 4 : kv_bytes;
              if (cache_bytes > 0) {
                bulk_g2s_hint(stage, k_cache + row0, cache_bytes, &full[s], pol_stream);
                bulk_g2s_hint(stage + C::KV_BYTES, v_cache + row0, cache_bytes, &full[s], pol_stream);
              }
              if (tail) {
                bulk_g2s(stage + cache_bytes, k_rows + row_src, D * 4, &full[s]);
                bulk_g2s(stage + C::KV_BYTES + cache_bytes, v_rows + row_src, D * 4, &full[s]);
              }
              if (st == 0)
                bulk_g2s(stage + 2 * C::KV_BYTES,
                         q + ((size_t)run.i * H + (size_t)run.g * G) * D, C::Q_BYTES, &full[s]);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
        }
        remaining -= run.units;
        if (ok && remaining > 0)
          run = next_run(run, remaining, sm, M, Hkv, chunk);
      }
    }
    if (lane == 0) {
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
      if (!ok) give_up(abort, d_status, ws.epoch);
      // Every copy this block issued lands before the block can exit, also
      // when a consumer warp gave up and no longer waits for it.  (The
      // latest use of each ring slot is in [first_live, k), so each wait is
      // for that use's phase.)
      for (uint32_t j = first_live; j < k; ++j) mbar_wait_drain(&full[j % C::S], (j / C::S) & 1u);
    }
    return;
  }

  // ========================= consumer warps ================================
  const TileLane<C> tl = tile_lane<C>(smem, warp, lane);
  float4 qv[G];
  float4 acc[G];
  float m_run[G];
  float l_lane;
#pragma unroll
  for (int h = 0; h < G; ++h) qv[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  tile_reset<G>(acc, m_run, l_lane);

  uint32_t mphase = 0;
  // Every wait of a consumer warp ends the same way for all its lanes (the
  // lanes go on to full-warp shuffles together, or leave together).  The
  // warp enters this barrier's wait converged (__syncwarp) and every test in
  // the wait is warp-uniform; the polling variant, whose waits are made to
  // run out, also takes the outcome by vote.
  auto consumers_barrier = [&]() -> bool {  // bounded; every consumer warp arrives once
    __syncwarp();
    if (lane == 0) mbar_arrive(mbar);
    bool got = mbar_wait<kPoll>(mbar, mphase, abort);
    if (kPoll) got = __all_sync(0xffffffffu, got);
    if (!got) {
      if (lane == 0) give_up(abort, d_status, ws.epoch);
      return false;
    }
    mphase ^= 1u;
    return true;
  };

  for (uint32_t k = 0;; ++k) {
    const uint32_t s = k % C::S;
    const uint32_t use = k / C::S;
    if (!__all_sync(0xffffffffu, mbar_wait<kPoll>(&full[s], use & 1u, abort))) {
      if (lane == 0) give_up(abort, d_status, ws.epoch);
      return;
    }
    const StageDesc dsc = desc[s];
    if (dsc.flags & kNoMore) break;
    const unsigned char *stage = smem + s * C::STAGE_BYTES;
    if (dsc.flags & kRunStart) tile_load_q<C>(tl, stage, qscale, qv);
    tile_consume<C>(tl, stage, dsc.nrows, qv, acc, m_run, l_lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (!(dsc.flags & kRunEnd)) continue;

    // ---- end of run: merge the NW warp states --------------------------------
    tile_publish<C>(tl, acc, m_run, l_lane);
    if (!consumers_barrier()) return;
    // A run that covers all of (i, g) is the answer; any other run is a
    // partial for the (i, g) merge.
    const bool whole = (dsc.run_rows == dsc.L);
    const int i_seq = dsc.ig / Hkv;
    const int g_kv = dsc.ig - i_seq * Hkv;
    for (int e = threadIdx.x; e < G * C::LPR; e += C::NW * 32) {
      const int h = e / C::LPR;
      const int d4 = e - h * C::LPR;
      float4 a;
      float mx, lsum;
      merged_warp_states<C>(smem, e, a, mx, lsum);
      if (whole) {
        const float inv = 1.f / lsum;
        reinterpret_cast<float4 *>(out)[((size_t)i_seq * H + (size_t)g_kv * G + h) * C::LPR + d4] =
            make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
      } else {
        const size_t sl = (size_t)dsc.slot * G + h;
        __stcg(&reinterpret_cast<float4 *>(ws.acc)[sl * C::LPR + d4], a);
        if (d4 == 0) __stcg(&ws.ml[sl], make_float2(mx, lsum));
      }
    }
    if (!whole) __threadfence();  // partials visible GPU-wide before the count
    if (!consumers_barrier()) return;
    if (!whole) {
      if (threadIdx.x == 0) {
        const unsigned before = tagged_add(ws.done + dsc.ig, (unsigned)dsc.run_rows, tag, d_status,
                                           ws.epoch);
        const bool last = (before != 0xffffffffu && before + (unsigned)dsc.run_rows == (unsigned)dsc.L);
        // Every run of (i, g) has counted: reset the counter (tag 0 is never
        // a call's tag), so a later launch with the same tag -- a replayed
        // CUDA graph freezes the tag argument -- starts from zero too.
        if (last) ws.done[dsc.ig] = 0ull;
        *s_last = last;
      }
      if (!consumers_barrier()) return;
      if (*s_last) {  // every run of (i, g) is in: merge them
        __threadfence();
        merge_runs<D, G, C::NW>(ws, out, i_seq, g_kv, M, Hkv, dsc.S, dsc.L, R, P, chunk, kCost,
                                smem + C::OFF_MACC);
      }
    }
    tile_reset<G>(acc, m_run, l_lane);  // the next run starts from nothing
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

struct StepLaunchInfo {
  int blocks_per_sm = 0;
  bool configured = false;
};

// Blocks per SM of one step-kernel instantiation on device `dev`
// (configures the kernel's shared-memory attributes on first use).
template <int D, int G>
int step_blocks_per_sm(int dev) {
  using C = Geo<D, G>;
  static StepLaunchInfo info[kMaxDevices];
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (!info[dev].configured) {
    // both wait variants have the same shared memory and launch bounds
    for (auto kern : {fd_step_kernel<D, G, false>, fd_step_kernel<D, G, true>}) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return -1;
      }
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    }
    int bps = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, fd_step_kernel<D, G, false>,
                                                      C::THREADS, C::SMEM_BYTES) != cudaSuccess ||
        bps < 1)
      return -1;
    info[dev].blocks_per_sm = bps;
    info[dev].configured = true;
  }
  return info[dev].blocks_per_sm;
}

// Rows (kv head x cache row) below which one block has too little to
// stream for the launch and pipeline fill to pay off.
constexpr long long kMinRowsPerBlock = 32;


template <int D, int G>
int launch_step_impl(const float *q, float *k_cache, float *v_cache, const SeqArgs &seqs,
                     const float *k_rows, const float *v_rows, float *out, int M, int Hkv,
                     int chunk, void *workspace, int *d_status, cudaStream_t stream) {
  const int max_len = seqs.max_len;
  using C = Geo<D, G>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVS_ERR_LAUNCH;
  const int bps = step_blocks_per_sm<D, G>(dev);
  const int sms = device_sm_count();
  if (bps <= 0 || sms <= 0) return KVS_ERR_LAUNCH;
  const long long rows_max = (long long)M * Hkv * max_len;
  const long long by_rows = std::max(1ll, (rows_max + kMinRowsPerBlock - 1) / kMinRowsPerBlock);
  const int grid =
      (int)std::min<long long>({(long long)sms * bps, (long long)kMaxChunkBlocks, by_rows});
  const WsView ws = workspace_view(workspace, M, Hkv, G, D);
  const float qscale = (float)(1.4426950408889634074 / std::sqrt((double)D));
  const cudaError_t e = launch_pdl(poll_waits() ? fd_step_kernel<D, G, true>
                                                : fd_step_kernel<D, G, false>,
                                   dim3(grid), dim3(C::THREADS), C::SMEM_BYTES, stream, q,
                                   k_cache, v_cache,
                                   SeqMap{seqs.positions, seqs.slots, seqs.done, max_len,
                                          seqs.num_slots, Hkv},
                                   k_rows, v_rows, out, ws, M, Hkv, chunk, qscale, fresh_tag(),
                                   d_status);
  return e == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

template <int D>
int dispatch_group(int G, const float *q, float *k_cache, float *v_cache,
                   const SeqArgs &seqs, const float *k_rows, const float *v_rows,
                   float *out, int M, int Hkv, int chunk, void *workspace,
                   int *d_status, cudaStream_t stream) {
  switch (G) {
#define KVS_CASE(g)                                                                           \
  case g:                                                                                     \
    return launch_step_impl<D, g>(q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, Hkv, chunk, \
                                  workspace, d_status, stream);
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

// Distinct for consecutive calls of this process (a 32-bit counter started
// at a time-derived value, never 0), so a counter left by an earlier call, or
// whatever a fresh workspace holds, is recognised as stale.
unsigned fresh_tag() {
  static std::atomic<unsigned> counter{
      (unsigned)(std::chrono::steady_clock::now().time_since_epoch().count() * 2654435761ull)};
  unsigned t;
  do {
    t = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
  } while (t == 0u);
  return t;
}

int set_wait_limit_step(uint64_t ns) {
  if (set_unit_wait_limit(ns) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  return KVS_OK;
}

int device_sm_count() {
  static int cache[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  if (cache[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev] = n;
  }
  return cache[dev];
}

int prepare_step_kernel(int H, int Hkv, int D) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVS_ERR_LAUNCH;
  if (Hkv < 1 || H % Hkv != 0) return KVS_ERR_DIMS;
  const int G = H / Hkv;
  int bps = -1;
  switch (D * 16 + G) {
#define KVS_PREP(d, g)                          \
  case d * 16 + g:                              \
    bps = step_blocks_per_sm<d, g>(dev);        \
    break;
    KVS_PREP(64, 1) KVS_PREP(64, 2) KVS_PREP(64, 3) KVS_PREP(64, 4)
    KVS_PREP(64, 5) KVS_PREP(64, 6) KVS_PREP(64, 7) KVS_PREP(64, 8)
    KVS_PREP(128, 1) KVS_PREP(128, 2) KVS_PREP(128, 3) KVS_PREP(128, 4)
    KVS_PREP(128, 5) KVS_PREP(128, 6) KVS_PREP(128, 7) KVS_PREP(128, 8)
#undef KVS_PREP
    default:
      return KVS_ERR_UNSUPPORTED;
  }
  return (bps > 0 && device_sm_count() > 0) ? KVS_OK : KVS_ERR_LAUNCH;
}

int launch_fd_step(const float *q, float *k_cache, float *v_cache, const SeqArgs &seqs,
                   const float *k_rows, const float *v_rows, float *out, int M, int H, int Hkv,
                   int D, int chunk, void *workspace, int *d_status, cudaStream_t stream) {
  const int G = H / Hkv;
  if (D == 128)
    return dispatch_group<128>(G, q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, Hkv, chunk,
                               workspace, d_status, stream);
  if (D == 64)
    return dispatch_group<64>(G, q, k_cache, v_cache, seqs, k_rows, v_rows, out, M, Hkv, chunk,
                              workspace, d_status, stream);
  return KVS_ERR_UNSUPPORTED;
}

}  // namespace kvs
