// flash_decode.cu -- split-K decode attention for sm_103a: the chunk kernel
// (softmax partials over runs of cache chunks) and the reduce kernel (the
// rescaled merge of the partials).
//
// Source: realizar 0.8.5, src/cuda/executor/head_dim.rs,
// flash_decoding_attention_into (PAR-118): doc comment (split the KV cache
// into chunks processed in parallel, then merge the partial results with
// softmax rescaling), "Step 3: Compute max chunks needed" (a sequence of
// length L has ceil(L / chunk) chunks), "Step 4" (chunk kernel, launched
// there with one 32-thread block per (query head, sequence, chunk)), "Step
// 5" (reduce kernel, one block per (query head, sequence)).
//
// GB300 design (what differs from the pages):
//  * Scheduling atom = chunk (sequence i, kv head g, chunk c) of `chunk`
//    cache rows, ordered (i, g, c).  One chunk serves all G = H/Hkv query
//    heads of its group, so every K/V byte leaves HBM once per call (the
//    pages' per-query-head blocks read each row G times).
//  * Persistent grid: #SMs x (CTAs per SM) blocks.  Block b takes the chunks
//    whose first cache row falls in its 1/P share of all live rows
//    (balanced by rows, so partial last chunks do not unbalance the SMs).
//    Lengths, chunk counts and ranges are derived on the device from the
//    device-resident positions.
//  * A block merges consecutive chunks of the same (i, g) on the fly: its
//    online-softmax state simply continues, so it writes ONE partial per run
//    of chunks, not one per chunk.  A run that starts at chunk 0 owns partial
//    slot i*Hkv + g; a run that starts inside (i, g) is the first run of its
//    block b and owns slot M*Hkv + b.  Each block records its first chunk in a
//    small table so the reduce can find the runs of any (i, g).
//  * Warp-specialised block: one producer warp streams each run's K and V
//    rows (contiguous ranges in the [Lmax][D] layout) and the group's q rows
//    into a ring of shared-memory stages with 1-D bulk asynchronous copies
//    (TMA, cp.async.bulk + mbarrier transaction counts); NW consumer warps
//    compute.  Every wait is bounded in time.
//  * Consumer warp tile: RW rows x G heads.  Lanes split head_dim (one
//    float4 per lane per row); q for the G heads lives in registers,
//    pre-multiplied by log2(e)/sqrt(D) so the softmax runs in base 2.  The
//    RW*G partial dot products are reduced with a transposing butterfly
//    (each shuffle level halves the values a lane holds), leaving one score
//    per lane.  Per tile and head: tile max -> running max, rescale factor,
//    exp2 of the lane's own score, then P.V with float4 reads of V.
//  * End of a run: the NW warps' (max, sum, acc) states merge in shared
//    memory into the run's partial: acc (unnormalised), m, l.
//  * Kernels are launched with programmatic stream serialisation: each one
//    waits (griddepcontrol.wait) before touching global memory, so the
//    launch of the next kernel overlaps the tail of the previous one.
//
// Partial semantics (per query head, run R of rows):
//   m = max_{j in R} s_j,  l = sum exp2(s_j - m),  acc = sum exp2(s_j - m) v_j,
//   s_j = log2(e) q.k_j / sqrt(D).
// Reduce: M* = max m,  out = sum 2^(m - M*) acc / sum 2^(m - M*) l.

#include <cmath>
#include <mutex>

#include "kvs_device.cuh"
#include "kvs_launch.h"

namespace kvs {

namespace {

__host__ __device__ constexpr int pow2ceil(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}
__host__ __device__ constexpr int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}
__host__ __device__ constexpr int round_up(int x, int a) { return (x + a - 1) / a * a; }

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// Compile-time geometry of one (head_dim, group) instantiation.
template <int D_, int G_>
struct Geo {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr int NW = 4;                    // consumer warps
  static constexpr int THREADS = (NW + 1) * 32;   // + one producer warp
  static constexpr int S = 3;                     // pipeline stages
  static constexpr int LPR = D / 4;               // lanes per row (float4 each)
  static constexpr int RPI = 32 / LPR;            // rows per warp instruction
  static constexpr int RP = (LPR / G) < 8 ? (LPR / G) : 8;  // rows per lane group
  static constexpr int NSLOT = pow2ceil(RP * G);  // butterfly slots (<= LPR)
  static constexpr int LOG2NS = ilog2(NSLOT);
  static constexpr int SPAN = LPR / NSLOT;        // lanes sharing one slot
  static constexpr int RW = RPI * RP;             // rows per warp tile
  static constexpr int T = NW * RW;               // rows per stage
  static constexpr int RWP = round_up(RW, 4);     // padded score row length
  static constexpr int GP = round_up(G, 4);       // padded p row length
  static constexpr int KV_BYTES = T * D * 4;      // one of K or V per stage
  static constexpr int Q_BYTES = G * D * 4;
  static constexpr int STAGE_BYTES = round_up(2 * KV_BYTES + Q_BYTES, 128);
  static constexpr int OFF_SCORE = S * STAGE_BYTES;
  static constexpr int SCORE_BYTES = NW * G * RWP * 4;
  static constexpr int OFF_P = OFF_SCORE + SCORE_BYTES;
  static constexpr int P_BYTES = NW * RW * GP * 4;
  static constexpr int OFF_MACC = round_up(OFF_P + P_BYTES, 128);
  static constexpr int MACC_BYTES = NW * G * D * 4;
  static constexpr int OFF_MM = OFF_MACC + MACC_BYTES;
  static constexpr int OFF_ML = OFF_MM + round_up(NW * G * 4, 16);
  static constexpr int OFF_MLL = OFF_ML + round_up(NW * G * 4, 16);
  static constexpr int OFF_BAR = round_up(OFF_MLL + NW * 32 * 4, 16);
  static constexpr int OFF_INFO = OFF_BAR + (2 * S + 1) * 8;  // 4 x int64
  static constexpr int OFF_FLAG = OFF_INFO + 32;              // abort, no_abort
  static constexpr int SMEM_BYTES = round_up(OFF_FLAG + 16, 128);
  static_assert(G >= 1 && G <= LPR, "group larger than lanes per row");
  static_assert(RP * G <= LPR, "slots exceed lanes");
  static_assert(RW * G <= 32 * RPI, "tile too large");
};

// Length attended by sequence i (0 for an out-of-range position).
__device__ __forceinline__ int seq_len_at(const int32_t *positions, int i, int max_len) {
  const int p = __ldg(positions + i);
  return (p >= 0 && p < max_len) ? p + 1 : 0;
}

// ---------------------------------------------------------------------------
// Split plan on the device (warp-cooperative; every lane returns the result)
// ---------------------------------------------------------------------------
struct SplitTotals {
  long long rows;   // sum_i Hkv * L_i   (live (kv head, row) pairs)
  long long units;  // sum_i Hkv * ceil(L_i / chunk)
};

__device__ SplitTotals warp_split_totals(const int32_t *positions, int M, int Hkv, int max_len,
                                         int chunk, int lane) {
  long long rows = 0, units = 0;
  for (int i = lane; i < M; i += 32) {
    const int L = seq_len_at(positions, i, max_len);
    rows += (long long)Hkv * L;
    units += (long long)Hkv * ((L + chunk - 1) / chunk);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    rows += __shfl_xor_sync(0xffffffffu, rows, o);
    units += __shfl_xor_sync(0xffffffffu, units, o);
  }
  return {rows, units};
}

// Global index of the first chunk whose first row is at or after row t of
// the (i, g, row)-ordered row space; `total_units` if t is past the end.
__device__ long long warp_first_unit_at_row(long long t, const int32_t *positions, int M,
                                            int Hkv, int max_len, int chunk,
                                            long long total_units, int lane) {
  long long row_base = 0, unit_base = 0;
  for (int i0 = 0; i0 < M; i0 += 32) {
    const int i = i0 + lane;
    const int L = (i < M) ? seq_len_at(positions, i, max_len) : 0;
    const int n = (L + chunk - 1) / chunk;
    const long long rows = (long long)Hkv * L, units = (long long)Hkv * n;
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
    const long long rexcl = row_base + rinc - rows;
    const long long uexcl = unit_base + uinc - units;
    const bool hit = rows > 0 && t >= rexcl && t < rexcl + rows;
    long long u = 0;
    if (hit) {
      const long long off = t - rexcl;
      const long long g = off / L;
      const long long r = off - g * L;
      u = uexcl + g * n + (r + chunk - 1) / chunk;  // == next (i, g)'s first chunk when c == n
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, hit);
    if (ballot) return __shfl_sync(0xffffffffu, u, __ffs(ballot) - 1);
    row_base += __shfl_sync(0xffffffffu, rinc, 31);
    unit_base += __shfl_sync(0xffffffffu, uinc, 31);
  }
  return total_units;
}

// (i, g, c) of global chunk index u (< total units).
__device__ int3 warp_unit_to_igc(long long u, const int32_t *positions, int M, int Hkv,
                                 int max_len, int chunk, int lane) {
  long long unit_base = 0;
  for (int i0 = 0; i0 < M; i0 += 32) {
    const int i = i0 + lane;
    const int L = (i < M) ? seq_len_at(positions, i, max_len) : 0;
    const int n = (L + chunk - 1) / chunk;
    const long long units = (long long)Hkv * n;
    long long uinc = units;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long b = __shfl_up_sync(0xffffffffu, uinc, o);
      if (lane >= o) uinc += b;
    }
    const long long uexcl = unit_base + uinc - units;
    const bool hit = units > 0 && u >= uexcl && u < uexcl + units;
    int3 r = make_int3(0, 0, 0);
    if (hit) {
      const long long rem = u - uexcl;
      r = make_int3(i, (int)(rem / n), (int)(rem % n));
    }
    const unsigned ballot = __ballot_sync(0xffffffffu, hit);
    if (ballot) {
      const int src = __ffs(ballot) - 1;
      return make_int3(__shfl_sync(0xffffffffu, r.x, src), __shfl_sync(0xffffffffu, r.y, src),
                       __shfl_sync(0xffffffffu, r.z, src));
    }
    unit_base += __shfl_sync(0xffffffffu, uinc, 31);
  }
  return make_int3(M, 0, 0);
}

// A run: consecutive chunks of one (i, g) inside a block's range.
struct Run {
  int i, g, c;  // first chunk of the run
  int L, n;     // sequence length, chunks of the sequence
  int units;    // chunks in the run
};

__device__ __forceinline__ Run make_run(int i, int g, int c, long long remaining,
                                        const int32_t *positions, int max_len, int chunk) {
  Run r;
  r.i = i;
  r.g = g;
  r.c = c;
  r.L = seq_len_at(positions, i, max_len);
  r.n = (r.L + chunk - 1) / chunk;
  r.units = (int)min((long long)(r.n - c), remaining);
  return r;
}

// The run after `r` (called only while chunks remain): next kv head of the
// sequence, else the next sequence that has rows.  Never reads past M-1; if
// the list ended (it cannot when the range came from the same positions) the
// run is empty (units = 0), which ends the loops.
__device__ __forceinline__ Run next_run(const Run &r, long long remaining,
                                        const int32_t *positions, int M, int Hkv,
                                        int max_len, int chunk) {
  if (r.g + 1 < Hkv) return make_run(r.i, r.g + 1, 0, remaining, positions, max_len, chunk);
  for (int i = r.i + 1; i < M; ++i) {
    if (seq_len_at(positions, i, max_len) > 0)
      return make_run(i, 0, 0, remaining, positions, max_len, chunk);
  }
  Run e = r;
  e.units = 0;
  e.L = 0;
  return e;
}

// Transposing butterfly: lane li (within a group of LPR lanes) holds v[NS]
// partial sums; afterwards it returns the full sum (over the LPR lanes) of
// slot li / (LPR / NS).
template <int NS, int LOG2NS, int LPR>
__device__ __forceinline__ float butterfly_sum(float (&v)[NS], int li) {
#pragma unroll
  for (int k = 0; k < LOG2NS; ++k) {
    const int half = NS >> (k + 1);
    const int dist = LPR >> (k + 1);
    const bool upper = (li & dist) != 0;
#pragma unroll
    for (int j = 0; j < half; ++j) {
      const float send = upper ? v[j] : v[j + half];
      const float keep = upper ? v[j + half] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, dist);
    }
  }
  float r = v[0];
#pragma unroll
  for (int dist = LPR / NS / 2; dist >= 1; dist >>= 1)
    r += __shfl_xor_sync(0xffffffffu, r, dist);
  return r;
}

// ---------------------------------------------------------------------------
// Chunk kernel
// ---------------------------------------------------------------------------
template <int D, int G>
__global__ void __launch_bounds__(Geo<D, G>::THREADS, 2)
    fd_chunk_kernel(const float *__restrict__ q, const float *__restrict__ k_cache,
                    const float *__restrict__ v_cache,
                    const int32_t *__restrict__ positions, WsView ws, int M, int Hkv,
                    int max_len, int chunk, float qscale, int *d_status) {
  using C = Geo<D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::S;
  uint64_t *mbar = empty + C::S;
  long long *info = reinterpret_cast<long long *>(smem + C::OFF_INFO);  // u0, u1, i, g|c
  volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
  volatile int *no_abort = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = Hkv * G;

  // Everything below reads inputs a previous kernel may have written, and
  // writes the workspace a previous reduce may still read.
  grid_dependency_wait();

  // ---- split plan: this block's chunk range (warp 0), barrier init --------
  if (warp == 0) {
    const SplitTotals tot = warp_split_totals(positions, M, Hkv, max_len, chunk, lane);
    const long long P = gridDim.x;
    const long long b = blockIdx.x;
    const long long t0 = tot.rows * b / P;
    const long long t1 = tot.rows * (b + 1) / P;
    const long long u0 = warp_first_unit_at_row(t0, positions, M, Hkv, max_len, chunk,
                                                tot.units, lane);
    const long long u1 = (b + 1 == P) ? tot.units
                                      : warp_first_unit_at_row(t1, positions, M, Hkv, max_len,
                                                               chunk, tot.units, lane);
    const int3 igc = (u0 < tot.units)
                         ? warp_unit_to_igc(u0, positions, M, Hkv, max_len, chunk, lane)
                         : make_int3(M, 0, 0);
    if (lane == 0) {
      info[0] = u0;
      info[1] = u1;
      info[2] = igc.x;
      info[3] = ((long long)igc.y << 32) | (unsigned)igc.z;
      // run table entry: this block's first chunk; w = 1 if it has work
      ws.table[b] = make_int4(igc.x, igc.y, igc.z, u0 < u1 ? 1 : 0);
      if (b == 0) *ws.num_blocks = (int)P;
      for (int s = 0; s < C::S; ++s) {
        mbar_init(&full[s], 1);
        mbar_init(&empty[s], C::NW);
      }
      mbar_init(mbar, C::NW);
      *abort = 0;
      *no_abort = 0;
      fence_mbar_init();
    }
  }
  __syncthreads();
  allow_dependent_launch();
  const long long u0 = info[0], u1 = info[1];
  if (u0 >= u1) return;
  const int start_i = (int)info[2];
  const int start_g = (int)(info[3] >> 32);
  const int start_c = (int)(info[3] & 0xffffffff);

  if (warp == C::NW) {
    // ===================== producer warp: one lane issues copies ==========
    if (lane != 0) return;
    const uint64_t pol_stream = policy_evict_first();
    uint32_t k = 0;
    bool ok = true;
    long long remaining = u1 - u0;
    Run run = make_run(start_i, start_g, start_c, remaining, positions, max_len, chunk);
    while (ok && remaining > 0 && run.units > 0) {
      const int r0 = run.c * chunk;
      const int r1 = (int)min((long long)(run.c + run.units) * chunk, (long long)run.L);
      const size_t head_base = ((size_t)run.i * Hkv + run.g) * (size_t)max_len;
      for (int rs = r0, st = 0; rs < r1; rs += C::T, ++st, ++k) {
        const uint32_t s = k % C::S;
        const uint32_t use = k / C::S;
        if (!mbar_wait(&empty[s], (use & 1u) ^ 1u, abort)) {
          ok = false;
          break;
        }
        const int nrows = min(C::T, r1 - rs);
        const uint32_t kv_bytes = (uint32_t)nrows * D * 4;
        const uint32_t bytes = 2 * kv_bytes + (st == 0 ? (uint32_t)C::Q_BYTES : 0u);
        unsigned char *stage = smem + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], bytes);
        const size_t row0 = (head_base + rs) * D;
        bulk_g2s_hint(stage, k_cache + row0, kv_bytes, &full[s], pol_stream);
        bulk_g2s_hint(stage + C::KV_BYTES, v_cache + row0, kv_bytes, &full[s], pol_stream);
        if (st == 0)
          bulk_g2s(stage + 2 * C::KV_BYTES,
                   q + ((size_t)run.i * H + (size_t)run.g * G) * D, C::Q_BYTES, &full[s]);
      }
      remaining -= run.units;
      if (ok && remaining > 0)
        run = next_run(run, remaining, positions, M, Hkv, max_len, chunk);
    }
    if (!ok) {
      *abort = 1;
      record_status(d_status, KVS_ERR_TIMEOUT);
      // let every copy already issued land before the block can exit
      for (uint32_t j = (k > (uint32_t)C::S ? k - C::S : 0u); j < k; ++j)
        mbar_wait(&full[j % C::S], (j / C::S) & 1u, no_abort);
    }
    return;
  }

  // ========================= consumer warps ================================
  const int w = warp;
  const int gi = lane / C::LPR;  // row group within the warp instruction
  const int li = lane % C::LPR;  // float4 column
  float *sS = reinterpret_cast<float *>(smem + C::OFF_SCORE) + w * G * C::RWP;  // [G][RWP]
  float *sP = reinterpret_cast<float *>(smem + C::OFF_P) + w * C::RW * C::GP;   // [RW][GP]
  float4 *sAcc = reinterpret_cast<float4 *>(smem + C::OFF_MACC);               // [NW][G][D/4]
  float *sM = reinterpret_cast<float *>(smem + C::OFF_MM);                     // [NW][G]
  float *sL = reinterpret_cast<float *>(smem + C::OFF_ML);                     // [NW][G]
  float *sLl = reinterpret_cast<float *>(smem + C::OFF_MLL);                   // [NW][32]

  for (int e = lane; e < G * C::RWP; e += 32) sS[e] = neg_inf();
  for (int e = lane; e < C::RW * C::GP; e += 32) sP[e] = 0.f;
  __syncwarp();

  // this lane's score slot
  const int slot = li / C::SPAN;
  const bool slot_used = slot < C::RP * G;
  const bool owner = slot_used && (li % C::SPAN) == 0;
  const int slot_r = slot / G;
  const int slot_h = slot - slot_r * G;
  const int slot_row = slot_r * C::RPI + gi;  // row within the warp tile

  float4 qv[G];
  float4 acc[G];
  float m_run[G];
  float l_lane = 0.f;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    m_run[h] = neg_inf();
  }

  uint32_t k = 0;
  uint32_t mphase = 0;
  long long remaining = u1 - u0;
  Run run = make_run(start_i, start_g, start_c, remaining, positions, max_len, chunk);
  while (remaining > 0 && run.units > 0) {
    const int r0 = run.c * chunk;
    const int r1 = (int)min((long long)(run.c + run.units) * chunk, (long long)run.L);
    for (int rs = r0, st = 0; rs < r1; rs += C::T, ++st, ++k) {
      const uint32_t s = k % C::S;
      const uint32_t use = k / C::S;
      if (!mbar_wait(&full[s], use & 1u, abort)) {
        *abort = 1;
        record_status(d_status, KVS_ERR_TIMEOUT);
        return;
      }
      const unsigned char *stage = smem + s * C::STAGE_BYTES;
      const float4 *sK = reinterpret_cast<const float4 *>(stage);
      const float4 *sV = reinterpret_cast<const float4 *>(stage + C::KV_BYTES);
      if (st == 0) {
        const float4 *sQ = reinterpret_cast<const float4 *>(stage + 2 * C::KV_BYTES);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 t = sQ[h * C::LPR + li];
          qv[h] = make_float4(t.x * qscale, t.y * qscale, t.z * qscale, t.w * qscale);
        }
      }
      const int nrows = min(C::T, r1 - rs);
      const int my_valid = min(max(nrows - w * C::RW, 0), C::RW);
      if (my_valid > 0) {
        const int tile0 = w * C::RW;
        // ---- scores: partial dot products, then the butterfly ----
        float part[C::NSLOT];
#pragma unroll
        for (int j = 0; j < C::NSLOT; ++j) part[j] = 0.f;
#pragma unroll
        for (int r = 0; r < C::RP; ++r) {
          const int row = tile0 + r * C::RPI + gi;
          const float4 kv = sK[row * C::LPR + li];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float d = qv[h].x * kv.x;
            d = fmaf(qv[h].y, kv.y, d);
            d = fmaf(qv[h].z, kv.z, d);
            d = fmaf(qv[h].w, kv.w, d);
            part[r * G + h] = d;
          }
        }
        const float sc = butterfly_sum<C::NSLOT, C::LOG2NS, C::LPR>(part, li);
        const bool valid = slot_used && slot_row < my_valid;
        const float s_val = valid ? sc : neg_inf();
        if (owner) sS[slot_h * C::RWP + slot_row] = s_val;
        __syncwarp();
        // ---- running max and rescale factors (all lanes, all heads) ----
        float alpha[G];
        float m_new[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float4 *row4 = reinterpret_cast<const float4 *>(sS + h * C::RWP);
          float tmax = neg_inf();
#pragma unroll
          for (int j = 0; j < C::RWP / 4; ++j) {
            const float4 t = row4[j];
            tmax = fmaxf(tmax, fmaxf(fmaxf(t.x, t.y), fmaxf(t.z, t.w)));
          }
          m_new[h] = fmaxf(m_run[h], tmax);
          alpha[h] = (m_new[h] == m_run[h]) ? 1.f : exp2f(m_run[h] - m_new[h]);
        }
        // ---- own-slot probability ----
        float mh = m_new[0];
#pragma unroll
        for (int h = 1; h < G; ++h) mh = (slot_h == h) ? m_new[h] : mh;
        float ah = alpha[0];
#pragma unroll
        for (int h = 1; h < G; ++h) ah = (slot_h == h) ? alpha[h] : ah;
        const float p = valid ? exp2f(s_val - mh) : 0.f;
        if (owner) {
          sP[slot_row * C::GP + slot_h] = p;
          l_lane = l_lane * ah + p;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          m_run[h] = m_new[h];
          acc[h].x *= alpha[h];
          acc[h].y *= alpha[h];
          acc[h].z *= alpha[h];
          acc[h].w *= alpha[h];
        }
        __syncwarp();
        // ---- P.V ----
#pragma unroll
        for (int r = 0; r < C::RP; ++r) {
          const int trow = r * C::RPI + gi;
          if (trow < my_valid) {
            const float4 vv = sV[(tile0 + trow) * C::LPR + li];
            float pr[C::GP];
#pragma unroll
            for (int j = 0; j < C::GP / 4; ++j) {
              const float4 t = reinterpret_cast<const float4 *>(sP + trow * C::GP)[j];
              pr[4 * j + 0] = t.x;
              pr[4 * j + 1] = t.y;
              pr[4 * j + 2] = t.z;
              pr[4 * j + 3] = t.w;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
              acc[h].x = fmaf(pr[h], vv.x, acc[h].x);
              acc[h].y = fmaf(pr[h], vv.y, acc[h].y);
              acc[h].z = fmaf(pr[h], vv.z, acc[h].z);
              acc[h].w = fmaf(pr[h], vv.w, acc[h].w);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    // ---- end of run: merge the NW warp states into the run's partial ----
    if (C::RPI > 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int o = C::LPR; o < 32; o <<= 1) {
          acc[h].x += __shfl_xor_sync(0xffffffffu, acc[h].x, o);
          acc[h].y += __shfl_xor_sync(0xffffffffu, acc[h].y, o);
          acc[h].z += __shfl_xor_sync(0xffffffffu, acc[h].z, o);
          acc[h].w += __shfl_xor_sync(0xffffffffu, acc[h].w, o);
        }
      }
    }
    if (gi == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) sAcc[(w * G + h) * C::LPR + li] = acc[h];
    }
    sLl[w * 32 + lane] = owner ? l_lane : 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h)
      if (lane == h) sM[w * G + h] = m_run[h];
    __syncwarp();
    if (lane < G) {
      float lsum = 0.f;
      for (int l2 = 0; l2 < 32; ++l2) {
        const int s2 = (l2 % C::LPR) / C::SPAN;
        if (s2 < C::RP * G && (s2 % G) == lane) lsum += sLl[w * 32 + l2];
      }
      sL[w * G + lane] = lsum;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(mbar);
    if (!mbar_wait(mbar, mphase, abort)) {
      *abort = 1;
      record_status(d_status, KVS_ERR_TIMEOUT);
      return;
    }
    mphase ^= 1u;
    {
      // slot of this run: (i, g) if it starts at chunk 0, else this block's
      const long long slot_id = (run.c == 0) ? (long long)run.i * Hkv + run.g
                                             : (long long)M * Hkv + blockIdx.x;
      const int t = threadIdx.x;  // 0 .. NW*32-1
      for (int e = t; run.L > 0 && e < G * C::LPR; e += C::NW * 32) {
        const int h = e / C::LPR;
        const int d4 = e - h * C::LPR;
        float mx = neg_inf();
#pragma unroll
        for (int w2 = 0; w2 < C::NW; ++w2) mx = fmaxf(mx, sM[w2 * G + h]);
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        float lsum = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < C::NW; ++w2) {
          const float mw = sM[w2 * G + h];
          const float sc = (mw == neg_inf()) ? 0.f : exp2f(mw - mx);
          const float4 b = sAcc[(w2 * G + h) * C::LPR + d4];
          a.x = fmaf(sc, b.x, a.x);
          a.y = fmaf(sc, b.y, a.y);
          a.z = fmaf(sc, b.z, a.z);
          a.w = fmaf(sc, b.w, a.w);
          lsum = fmaf(sc, sL[w2 * G + h], lsum);
        }
        const size_t sl = (size_t)slot_id * G + h;
        reinterpret_cast<float4 *>(ws.acc)[sl * C::LPR + d4] = a;
        if (d4 == 0) ws.ml[sl] = make_float2(mx, lsum);
      }
    }
    if (lane == 0) mbar_arrive(mbar);
    if (!mbar_wait(mbar, mphase, abort)) {
      *abort = 1;
      record_status(d_status, KVS_ERR_TIMEOUT);
      return;
    }
    mphase ^= 1u;
    // reset the running state for the next run
    l_lane = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
      m_run[h] = neg_inf();
    }
    remaining -= run.units;
    if (remaining > 0) run = next_run(run, remaining, positions, M, Hkv, max_len, chunk);
  }
}

// ---------------------------------------------------------------------------
// Reduce kernel: one 128-thread block per (sequence, query head).
// ---------------------------------------------------------------------------
// (i, g, c) < (e.x, e.y, e.z) lexicographically
__device__ __forceinline__ bool igc_before(int i, int g, int c, int4 e) {
  return i < e.x || (i == e.x && (g < e.y || (g == e.y && c < e.z)));
}

template <int D>
__global__ void __launch_bounds__(128)
    fd_reduce_kernel(const int32_t *__restrict__ positions, WsView ws, float *__restrict__ out,
                     int M, int Hkv, int G, int max_len, int P, int *d_status) {
  constexpr int LPR = D / 4;
  constexpr int NP = 128 / LPR;  // run phases
  grid_dependency_wait();
  allow_dependent_launch();
  const int H = Hkv * G;
  const int ih = blockIdx.x;
  const int i = ih / H;
  const int h = ih - i * H;
  const int g = h / G;
  const int hh = h - g * G;
  const int t = threadIdx.x;
  const int cp = t / LPR;
  const int d4 = t % LPR;
  const float4 *acc4 = reinterpret_cast<const float4 *>(ws.acc);
  __shared__ int4 s_tab[kMaxChunkBlocks];
  __shared__ int s_first, s_count;
  __shared__ float s_m[NP], s_l[NP];
  __shared__ float4 s_acc[NP][LPR];

  // Everything that does not depend on the block table is loaded at once:
  // the position, the chunk-0 run's partial and the table itself.
  const size_t slot0 = ((size_t)i * Hkv + g) * G + hh;
  const int L = seq_len_at(positions, i, max_len);
  float2 ml0 = make_float2(0.f, 0.f);
  float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (cp == 0) {
    ml0 = ws.ml[slot0];
    acc0 = acc4[slot0 * LPR + d4];
  }
  for (int b = t; b < P; b += 128) s_tab[b] = ws.table[b];

  float4 *o4 = reinterpret_cast<float4 *>(out) + (size_t)ih * LPR;
  if (L == 0) {
    const float nan = __int_as_float(0x7fc00000);
    if (t < LPR) o4[t] = make_float4(nan, nan, nan, nan);
    if (t == 0 && h == 0) record_status(d_status, KVS_ERR_POSITION);
    return;
  }
  __syncthreads();
  // Runs of (i, g): the run at chunk 0 (slot i*Hkv + g) and the first run of
  // every block whose range starts inside (i, g) (slot M*Hkv + b).  The table
  // is sorted by chunk: find the first entry after (i, g, 0).
  if (t == 0) {
    int lo = 0, hi = P;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (igc_before(i, g, 0, s_tab[mid])) hi = mid;
      else lo = mid + 1;
    }
    int cnt = 0;
    while (lo + cnt < P && s_tab[lo + cnt].x == i && s_tab[lo + cnt].y == g) ++cnt;
    s_first = lo;
    s_count = cnt;
  }
  __syncthreads();
  const int first = s_first;
  const int nruns = 1 + s_count;  // run 0 is the chunk-0 run

  // Each phase cp merges runs cp, cp + NP, ... online (running max and
  // rescaling), then the NP phase states are merged.
  float m = neg_inf(), l = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  if (cp == 0) {
    m = ml0.x;
    l = ml0.y;
    a = acc0;
  }
  for (int r = (cp == 0 ? NP : cp); r < nruns; r += NP) {
    if (s_tab[first + r - 1].w == 0) continue;  // a block without work
    const size_t sl = ((size_t)M * Hkv + first + r - 1) * G + hh;
    const float2 ml = ws.ml[sl];
    const float4 b = acc4[sl * LPR + d4];
    const float mn = fmaxf(m, ml.x);
    const float wa = (m == neg_inf()) ? 0.f : exp2f(m - mn);
    const float wb = exp2f(ml.x - mn);
    a.x = fmaf(wb, b.x, wa * a.x);
    a.y = fmaf(wb, b.y, wa * a.y);
    a.z = fmaf(wb, b.z, wa * a.z);
    a.w = fmaf(wb, b.w, wa * a.w);
    l = fmaf(wb, ml.y, wa * l);
    m = mn;
  }
  if (nruns <= NP) {
    // at most one run per phase: phases >= nruns hold nothing
    if (nruns == 1) {
      if (cp == 0) {
        const float inv = 1.f / l;
        o4[d4] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
      }
      return;
    }
  }
  if (d4 == 0) {
    s_m[cp] = m;
    s_l[cp] = l;
  }
  s_acc[cp][d4] = a;
  __syncthreads();
  if (cp == 0) {
    float mx = s_m[0];
#pragma unroll
    for (int j = 1; j < NP; ++j) mx = fmaxf(mx, s_m[j]);
    float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
    float lt = 0.f;
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      const float w = (s_m[j] == neg_inf()) ? 0.f : exp2f(s_m[j] - mx);
      const float4 b = s_acc[j][d4];
      r.x = fmaf(w, b.x, r.x);
      r.y = fmaf(w, b.y, r.y);
      r.z = fmaf(w, b.z, r.z);
      r.w = fmaf(w, b.w, r.w);
      lt = fmaf(w, s_l[j], lt);
    }
    const float inv = 1.f / lt;
    o4[d4] = make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv);
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

struct ChunkLaunchInfo {
  int blocks_per_sm = 0;
  bool configured = false;
};

// Blocks per SM of one chunk-kernel instantiation on the current device
// (configures the kernel's shared-memory attributes on first use).
template <int D, int G>
int chunk_blocks_per_sm(int dev) {
  using C = Geo<D, G>;
  static ChunkLaunchInfo info[kMaxDevices];
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (!info[dev].configured) {
    auto kern = fd_chunk_kernel<D, G>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return -1;
    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    int bps = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, C::THREADS, C::SMEM_BYTES) !=
            cudaSuccess ||
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
int chunk_grid(int M, int Hkv, int max_len) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  const int bps = chunk_blocks_per_sm<D, G>(dev);
  const int sms = device_sm_count();
  if (bps <= 0 || sms <= 0) return -1;
  const long long rows_max = (long long)M * Hkv * max_len;
  const long long by_rows = std::max(1ll, (rows_max + kMinRowsPerBlock - 1) / kMinRowsPerBlock);
  return (int)std::min<long long>({(long long)sms * bps, (long long)kMaxChunkBlocks, by_rows});
}

template <int D, int G>
int launch_chunks_impl(const float *q, const float *k_cache, const float *v_cache,
                       const int32_t *positions, int M, int Hkv, int max_len, int chunk,
                       void *workspace, int *d_status, cudaStream_t stream) {
  using C = Geo<D, G>;
  const int grid = chunk_grid<D, G>(M, Hkv, max_len);
  if (grid <= 0) return KVS_ERR_LAUNCH;
  const WsView ws = workspace_view(workspace, M, Hkv, G, D);
  const float qscale = (float)(1.4426950408889634074 / std::sqrt((double)D));
  const cudaError_t e = launch_pdl(fd_chunk_kernel<D, G>, dim3(grid), dim3(C::THREADS),
                                   C::SMEM_BYTES, stream, q, k_cache, v_cache, positions, ws, M,
                                   Hkv, max_len, chunk, qscale, d_status);
  return e == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

template <int D>
int grid_for_group(int G, int M, int Hkv, int max_len) {
  switch (G) {
    case 1: return chunk_grid<D, 1>(M, Hkv, max_len);
    case 2: return chunk_grid<D, 2>(M, Hkv, max_len);
    case 3: return chunk_grid<D, 3>(M, Hkv, max_len);
    case 4: return chunk_grid<D, 4>(M, Hkv, max_len);
    case 5: return chunk_grid<D, 5>(M, Hkv, max_len);
    case 6: return chunk_grid<D, 6>(M, Hkv, max_len);
    case 7: return chunk_grid<D, 7>(M, Hkv, max_len);
    case 8: return chunk_grid<D, 8>(M, Hkv, max_len);
    default: return -1;
  }
}

template <int D>
int dispatch_group(int G, const float *q, const float *k_cache, const float *v_cache,
                   const int32_t *positions, int M, int Hkv, int max_len, int chunk,
                   void *workspace, int *d_status, cudaStream_t stream) {
  switch (G) {
#define KVS_CASE(g)                                                                      \
  case g:                                                                                \
    return launch_chunks_impl<D, g>(q, k_cache, v_cache, positions, M, Hkv, max_len,    \
                                    chunk, workspace, d_status, stream);
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

int launch_fd_chunks(const float *q, const float *k_cache, const float *v_cache,
                     const int32_t *positions, int M, int H, int Hkv, int D, int max_len,
                     int chunk, void *workspace, int *d_status, cudaStream_t stream) {
  const int G = H / Hkv;
  if (D == 128)
    return dispatch_group<128>(G, q, k_cache, v_cache, positions, M, Hkv, max_len, chunk,
                               workspace, d_status, stream);
  if (D == 64)
    return dispatch_group<64>(G, q, k_cache, v_cache, positions, M, Hkv, max_len, chunk,
                              workspace, d_status, stream);
  return KVS_ERR_UNSUPPORTED;
}

int launch_fd_reduce(const int32_t *positions, float *out, int M, int H, int Hkv, int D,
                     int max_len, const void *workspace, int *d_status, cudaStream_t stream) {
  const int G = H / Hkv;
  const WsView ws = workspace_view(const_cast<void *>(workspace), M, Hkv, G, D);
  const unsigned blocks = (unsigned)((int64_t)M * H);
  // the chunk kernel's grid size: the number of valid block-table entries
  const int P = (D == 128) ? grid_for_group<128>(G, M, Hkv, max_len)
                           : grid_for_group<64>(G, M, Hkv, max_len);
  if (P <= 0) return KVS_ERR_LAUNCH;
  static bool carveout_set[kMaxDevices] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices && !carveout_set[dev]) {
    // the same L1/shared split as the chunk kernel, so SMs need no
    // reconfiguration between the two launches
    cudaFuncSetAttribute(fd_reduce_kernel<128>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    cudaFuncSetAttribute(fd_reduce_kernel<64>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    carveout_set[dev] = true;
  }
  cudaError_t e;
  if (D == 128)
    e = launch_pdl(fd_reduce_kernel<128>, dim3(blocks), dim3(128), 0, stream, positions, ws, out,
                   M, Hkv, G, max_len, P, d_status);
  else if (D == 64)
    e = launch_pdl(fd_reduce_kernel<64>, dim3(blocks), dim3(128), 0, stream, positions, ws, out,
                   M, Hkv, G, max_len, P, d_status);
  else
    return KVS_ERR_UNSUPPORTED;
  return e == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

}  // namespace kvs
