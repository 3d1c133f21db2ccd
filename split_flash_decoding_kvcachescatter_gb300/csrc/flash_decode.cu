// flash_decode.cu -- split-K decode attention for sm_103a: the chunk kernel
// (partials per chunk of cache rows) and the reduce kernel (rescaled merge).
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
//  * Work unit = (sequence i, kv head g, chunk c).  One unit serves all
//    G = H/Hkv query heads of the group, so every K/V byte is read from HBM
//    once per call (the pages' per-query-head blocks read each row G times).
//  * Persistent grid: #SMs x (CTAs per SM) blocks; block b takes a
//    contiguous range of the unit list, ordered (i, g, c).  The unit list is
//    built on the device from the device-resident positions, so the host
//    never needs the lengths.
//  * Warp-specialised CTA: one producer warp streams each unit's K and V
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
//  * End of a unit: the NW warps' (max, sum, acc) states merge in shared
//    memory into the unit's partial: acc (unnormalised), m, l.
//
// Partial semantics (per query head, chunk c over rows R_c):
//   m_c = max_{j in R_c} s_j,  l_c = sum exp2(s_j - m_c),
//   acc_c = sum exp2(s_j - m_c) v_j,   s_j = log2(e) q.k_j / sqrt(D).
// Reduce: M* = max_c m_c,  out = sum_c 2^(m_c - M*) acc_c / sum_c 2^(m_c - M*) l_c.

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
  static constexpr int OFF_RANGE = OFF_BAR + (2 * S + 1) * 8;  // 2 x int64
  static constexpr int OFF_FLAG = OFF_RANGE + 16;                // abort, drain, i, g, c
  static constexpr int SMEM_BYTES = round_up(OFF_FLAG + 32, 128);
  static_assert(G >= 1 && G <= LPR, "group larger than lanes per row");
  static_assert(RP * G <= LPR, "slots exceed lanes");
  static_assert(RW * G <= 32 * RPI, "tile too large");
};

// Length attended by sequence i (0 for an out-of-range position).
__device__ __forceinline__ int seq_len_at(const int32_t *positions, int i, int max_len) {
  const int p = __ldg(positions + i);
  return (p >= 0 && p < max_len) ? p + 1 : 0;
}

// Position in the (i, g, c) unit list.
struct Cursor {
  int i, g, c, n, L;
};

// Advances to the next unit.  Never reads past sequence M-1: if the list
// ended early (it cannot when the range was computed from the same
// positions) the cursor is left empty (n = L = 0), which makes every loop
// over its rows a no-op.
__device__ __forceinline__ void cursor_next(Cursor &cu, const int32_t *positions, int M,
                                            int Hkv, int max_len, int chunk) {
  if (++cu.c < cu.n) return;
  cu.c = 0;
  if (++cu.g < Hkv) return;
  cu.g = 0;
  do {
    if (++cu.i >= M) {
      cu.i = M - 1;
      cu.n = cu.L = 0;
      return;
    }
    cu.L = seq_len_at(positions, cu.i, max_len);
    cu.n = (cu.L + chunk - 1) / chunk;
  } while (cu.n == 0);
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
                    const int32_t *__restrict__ positions, float *__restrict__ part_acc,
                    float2 *__restrict__ part_ml, int M, int Hkv, int max_len,
                    int chunk, int64_t n_max, float qscale, int *d_status) {
  using C = Geo<D, G>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::S;
  uint64_t *mbar = empty + C::S;
  long long *s_range = reinterpret_cast<long long *>(smem + C::OFF_RANGE);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG);
  volatile int *no_abort = reinterpret_cast<volatile int *>(smem + C::OFF_FLAG + 4);
  int *cta_info = reinterpret_cast<int *>(smem + C::OFF_FLAG + 8);  // [i, g, c]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = Hkv * G;

  // ---- unit range of this CTA (warp 0), barrier init (thread 0) ----------
  if (warp == 0) {
    long long total = 0;
    for (int i = lane; i < M; i += 32) {
      const int L = seq_len_at(positions, i, max_len);
      total += (long long)Hkv * ((L + chunk - 1) / chunk);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    const long long P = gridDim.x;
    const long long u0 = total * (long long)blockIdx.x / P;
    const long long u1 = total * (long long)(blockIdx.x + 1) / P;
    // locate u0: scan sequences in blocks of 32
    long long base = 0;
    int found_i = -1;
    long long found_base = 0;
    if (u0 < u1) {
      for (int i0 = 0; i0 < M && found_i < 0; i0 += 32) {
        const int i = i0 + lane;
        long long units = 0;
        if (i < M) {
          const int L = seq_len_at(positions, i, max_len);
          units = (long long)Hkv * ((L + chunk - 1) / chunk);
        }
        long long incl = units;  // inclusive scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const long long excl = base + incl - units;
        const bool hit = units > 0 && u0 >= excl && u0 < excl + units;
        const unsigned ballot = __ballot_sync(0xffffffffu, hit);
        if (ballot) {
          const int src = __ffs(ballot) - 1;
          found_i = i0 + src;
          found_base = __shfl_sync(0xffffffffu, excl, src);
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) {
      s_range[0] = u0;
      s_range[1] = u1;
      if (u0 < u1) {
        const int L = seq_len_at(positions, found_i, max_len);
        const int n = (L + chunk - 1) / chunk;
        const long long rem = u0 - found_base;
        cta_info[0] = found_i;
        cta_info[1] = (int)(rem / n);
        cta_info[2] = (int)(rem % n);
      }
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
  const long long u0 = s_range[0], u1 = s_range[1];
  if (u0 >= u1) return;

  Cursor cu;
  cu.i = cta_info[0];
  cu.g = cta_info[1];
  cu.c = cta_info[2];
  cu.L = seq_len_at(positions, cu.i, max_len);
  cu.n = (cu.L + chunk - 1) / chunk;

  if (warp == C::NW) {
    // ===================== producer warp: one lane issues copies ==========
    if (lane != 0) return;
    const uint64_t pol_stream = policy_evict_first();
    uint32_t k = 0;
    bool ok = true;
    for (long long u = u0; u < u1 && ok; ++u) {
      const int r0 = cu.c * chunk;
      const int r1 = min(r0 + chunk, cu.L);
      const size_t head_base = ((size_t)cu.i * Hkv + cu.g) * (size_t)max_len;
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
                   q + ((size_t)cu.i * H + (size_t)cu.g * G) * D, C::Q_BYTES, &full[s]);
      }
      if (ok && u + 1 < u1) cursor_next(cu, positions, M, Hkv, max_len, chunk);
    }
    if (!ok) {
      *abort = 1;
      record_status(d_status, KVS_ERR_TIMEOUT);
      // let every copy already issued land before the CTA can exit
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
  for (long long u = u0; u < u1; ++u) {
    const int r0 = cu.c * chunk;
    const int r1 = min(r0 + chunk, cu.L);
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

    // ---- end of unit: merge the NW warp states into the chunk partial ----
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
      const int t = threadIdx.x;  // 0 .. NW*32-1
      const size_t slot0 = ((size_t)cu.i * H + (size_t)cu.g * G) * (size_t)n_max + cu.c;
      for (int e = t; cu.L > 0 && e < G * C::LPR; e += C::NW * 32) {
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
        const size_t sl = slot0 + (size_t)h * (size_t)n_max;
        reinterpret_cast<float4 *>(part_acc)[sl * C::LPR + d4] = a;
        if (d4 == 0) part_ml[sl] = make_float2(mx, lsum);
      }
    }
    if (lane == 0) mbar_arrive(mbar);
    if (!mbar_wait(mbar, mphase, abort)) {
      *abort = 1;
      record_status(d_status, KVS_ERR_TIMEOUT);
      return;
    }
    mphase ^= 1u;
    // reset the running state for the next unit
    l_lane = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
      m_run[h] = neg_inf();
    }
    if (u + 1 < u1) cursor_next(cu, positions, M, Hkv, max_len, chunk);
  }
}

// ---------------------------------------------------------------------------
// Reduce kernel: one 128-thread block per (sequence, query head).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128)
    fd_reduce_kernel(const int32_t *__restrict__ positions,
                     const float *__restrict__ part_acc,
                     const float2 *__restrict__ part_ml, float *__restrict__ out,
                     int H, int max_len, int chunk, int64_t n_max, int *d_status) {
  constexpr int LPR = D / 4;
  constexpr int NP = 128 / LPR;  // chunk phases
  const int ih = blockIdx.x;
  const int i = ih / H;
  const int t = threadIdx.x;
  const int L = seq_len_at(positions, i, max_len);
  float4 *o4 = reinterpret_cast<float4 *>(out) + (size_t)ih * LPR;
  if (L == 0) {
    const float nan = __int_as_float(0x7fc00000);
    if (t < LPR) o4[t] = make_float4(nan, nan, nan, nan);
    if (t == 0 && ih % H == 0) record_status(d_status, KVS_ERR_POSITION);
    return;
  }
  const int n = (L + chunk - 1) / chunk;
  const size_t base = (size_t)ih * (size_t)n_max;
  __shared__ float s_red[4];
  __shared__ float4 s_acc[NP][LPR];
  __shared__ float s_l[NP][LPR];

  // pass 1: global max of the chunk maxima
  float mx = neg_inf();
  for (int c = t; c < n; c += 128) mx = fmaxf(mx, part_ml[base + c].x);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((t & 31) == 0) s_red[t >> 5] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));

  // pass 2: rescaled sums
  const int cp = t / LPR;
  const int d4 = t % LPR;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  const float4 *acc4 = reinterpret_cast<const float4 *>(part_acc);
  for (int c = cp; c < n; c += NP) {
    const float2 ml = part_ml[base + c];
    const float w = exp2f(ml.x - mx);
    const float4 b = acc4[(base + c) * LPR + d4];
    a.x = fmaf(w, b.x, a.x);
    a.y = fmaf(w, b.y, a.y);
    a.z = fmaf(w, b.z, a.z);
    a.w = fmaf(w, b.w, a.w);
    l = fmaf(w, ml.y, l);
  }
  s_acc[cp][d4] = a;
  s_l[cp][d4] = l;
  __syncthreads();
  if (cp == 0) {
    float4 r = s_acc[0][d4];
    float lt = s_l[0][d4];
#pragma unroll
    for (int j = 1; j < NP; ++j) {
      const float4 b = s_acc[j][d4];
      r.x += b.x;
      r.y += b.y;
      r.z += b.z;
      r.w += b.w;
      lt += s_l[j][d4];
    }
    const float inv = 1.f / lt;
    o4[d4] = make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv);
  }
}

// ---------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------
struct ChunkLaunchInfo {
  int blocks_per_sm = 0;
  bool configured = false;
};

constexpr int kMaxDevices = 64;

template <int D, int G>
int launch_chunks_impl(const float *q, const float *k_cache, const float *v_cache,
                       const int32_t *positions, int M, int Hkv, int max_len,
                       int chunk, void *workspace, int *d_status,
                       cudaStream_t stream) {
  using C = Geo<D, G>;
  static ChunkLaunchInfo info[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVS_ERR_LAUNCH;
  auto kern = fd_chunk_kernel<D, G>;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!info[dev].configured) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES) != cudaSuccess)
        return KVS_ERR_LAUNCH;
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      int bps = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kern, C::THREADS,
                                                        C::SMEM_BYTES) != cudaSuccess ||
          bps < 1)
        return KVS_ERR_LAUNCH;
      info[dev].blocks_per_sm = bps;
      info[dev].configured = true;
    }
  }
  const int sms = device_sm_count();
  if (sms <= 0) return KVS_ERR_LAUNCH;
  const int grid = sms * info[dev].blocks_per_sm;
  const PartialLayout lay = partial_layout(M, Hkv * G, D, max_len, chunk);
  float *acc = reinterpret_cast<float *>(workspace);
  float2 *ml = reinterpret_cast<float2 *>(reinterpret_cast<unsigned char *>(workspace) +
                                          lay.acc_bytes);
  const float qscale = (float)(1.4426950408889634074 / std::sqrt((double)D));
  kern<<<grid, C::THREADS, C::SMEM_BYTES, stream>>>(q, k_cache, v_cache, positions, acc, ml,
                                                    M, Hkv, max_len, chunk, lay.n_max,
                                                    qscale, d_status);
  return cudaGetLastError() == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
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

int launch_fd_reduce(const int32_t *positions, float *out, int M, int H, int D, int max_len,
                     int chunk, const void *workspace, int *d_status, cudaStream_t stream) {
  const PartialLayout lay = partial_layout(M, H, D, max_len, chunk);
  const float *acc = reinterpret_cast<const float *>(workspace);
  const float2 *ml = reinterpret_cast<const float2 *>(
      reinterpret_cast<const unsigned char *>(workspace) + lay.acc_bytes);
  const unsigned blocks = (unsigned)((int64_t)M * H);
  if (D == 128)
    fd_reduce_kernel<128><<<blocks, 128, 0, stream>>>(positions, acc, ml, out, H, max_len,
                                                      chunk, lay.n_max, d_status);
  else if (D == 64)
    fd_reduce_kernel<64><<<blocks, 128, 0, stream>>>(positions, acc, ml, out, H, max_len,
                                                     chunk, lay.n_max, d_status);
  else
    return KVS_ERR_UNSUPPORTED;
  return cudaGetLastError() == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

}  // namespace kvs
