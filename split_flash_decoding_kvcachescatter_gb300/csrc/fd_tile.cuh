// fd_tile.cuh -- pieces shared by the decode-attention kernels: the stage
// geometry of one (head_dim, group) instantiation and the consumer warps'
// per-stage math (scores, base-2 online softmax, P.V) and end-of-run merge
// of their states.
//
// Source: realizar 0.8.5, src/cuda/executor/head_dim.rs,
// flash_decoding_attention_into (PAR-118), doc comment: each chunk of the KV
// cache yields a running max, a running sum and a weighted-V accumulator,
// and the chunk results are merged with softmax rescaling.  Here the
// "chunk" a consumer warp sees is one stage of T cache rows shared by the G
// query heads of a kv group.
#pragma once

#include <cstdint>

#include "kvs_device.cuh"
#include "kvsdecode.h"

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
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// Stage descriptor written by the producer, read by the consumers.
constexpr int kRunStart = 1;  // first stage of a run: the stage also holds q
constexpr int kRunEnd = 2;    // last stage of a run: merge, write the partial
constexpr int kNoMore = 4;    // no stage: the block is done
struct StageDesc {
  int flags;
  int nrows;     // rows in this stage
  int ig;        // i * Hkv + g
  int run_rows;  // rows of the whole run
  int L;         // length of sequence i
  int pad;
  long long slot;  // partial slot of the run
  long long S;     // first row of (i, g) in the (i, g, row) order
};

// Scratch of the (i, g) merge (aliases the warp-state merge area).
constexpr int kMergeWindow = 32;  // candidate blocks examined per pass
// Partial loads a merging thread keeps in flight: 8, or 4 for groups of more
// than 5 heads, whose chunk loop leaves fewer registers free.
__host__ __device__ constexpr int merge_batch(int G) { return G <= 5 ? 8 : 4; }
constexpr int kMergeScratchBytes = kMergeWindow * 4 + 16;

// Shared memory budget of the stage ring (two blocks per SM).
constexpr int kRingBytes = 96 * 1024;

// Compile-time geometry of one (head_dim, group) instantiation.
//
// A consumer warp folds NSUB sub-tiles of RW1 rows per stage.  Sub-tile u of
// warp w holds stage rows [(u * NW + w) * RW1, +RW1), so a partial stage is
// spread over the warps.  The sub-tiles' butterflies are independent, so a
// warp overlaps their shuffle chains: more rows per stage for little more
// latency, which is what a latency-bound step (few rows per block) needs.
//
// SHFL_MAX takes each head's running max over the warp's scores with
// shuffles, straight from the lanes that hold them after the butterfly,
// instead of through a shared-memory score tile (fewer instructions and no
// store-load round trip: faster for a latency-bound block; measured on
// GB300, the score tile is slightly faster where blocks are many and the
// stream bandwidth-bound).
template <int D_, int G_, int NW_ = 4, int MINB_ = 2, int NSUB_ = 1, bool SHFL_MAX_ = false>
struct Geo {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr int NW = NW_;                  // consumer warps
  static constexpr int MINB = MINB_;              // blocks per SM the budget is for
  static constexpr int NSUB = NSUB_;              // sub-tiles per warp and stage
  static constexpr bool SHFL_MAX = SHFL_MAX_;
  static constexpr int THREADS = (NW + 1) * 32;   // + one producer warp
  static constexpr int LPR = D / 4;               // lanes per row (float4 each)
  static constexpr int RPI = 32 / LPR;            // rows per warp instruction
  static constexpr int RP = (LPR / G) < 8 ? (LPR / G) : 8;  // rows per lane group
  static constexpr int NSLOT = pow2ceil(RP * G);  // butterfly slots (<= LPR)
  static constexpr int LOG2NS = ilog2(NSLOT);
  static constexpr int SPAN = LPR / NSLOT;        // lanes sharing one slot
  static constexpr int RW1 = RPI * RP;            // rows per sub-tile
  static constexpr int RW = RW1 * NSUB;           // rows per warp and stage
  static constexpr int T = NW * RW;               // rows per stage
  static constexpr int RWP = round_up(RW, 4);     // padded score row length
  static constexpr int GP = round_up(G, 4);       // padded p row length
  static constexpr int KV_BYTES = T * D * 4;      // one of K or V per stage
  static constexpr int Q_BYTES = G * D * 4;
  static constexpr int STAGE_BYTES = round_up(2 * KV_BYTES + Q_BYTES, 128);
  // pipeline stages: as many as fit in kRingBytes, at least 3 and at most 8
  // (small stages -- head_dim 64 with a large group -- get a deeper ring, so
  // that one block alone still keeps tens of KB of K/V in flight)
  static constexpr int S = cmin(8, cmax(3, kRingBytes / STAGE_BYTES));
  static constexpr int OFF_SCORE = S * STAGE_BYTES;
  static constexpr int SCORE_BYTES = SHFL_MAX ? 0 : NW * G * RWP * 4;
  static constexpr int OFF_P = OFF_SCORE + SCORE_BYTES;
  static constexpr int P_BYTES = NW * RW * GP * 4;
  static constexpr int OFF_MACC = round_up(OFF_P + P_BYTES, 128);
  static constexpr int MACC_BYTES = cmax(NW * G * D * 4, kMergeScratchBytes);
  static constexpr int OFF_MM = OFF_MACC + round_up(MACC_BYTES, 16);
  static constexpr int OFF_ML = OFF_MM + round_up(NW * G * 4, 16);
  static constexpr int OFF_MLL = OFF_ML + round_up(NW * G * 4, 16);
  static constexpr int OFF_DESC = round_up(OFF_MLL + NW * 32 * 4, 16);
  static constexpr int OFF_BAR = OFF_DESC + S * (int)sizeof(StageDesc);
  static constexpr int OFF_INFO = OFF_BAR + (2 * S + 1) * 8;  // R, U, tag (int64)
  static constexpr int OFF_FLAG = OFF_INFO + 32;              // abort, -, last
  static constexpr int SMEM_BYTES = round_up(OFF_FLAG + 16, 128);
  static_assert(G >= 1 && G <= LPR, "group larger than lanes per row");
  static_assert(RP * G <= LPR, "slots exceed lanes");
  static_assert(RW1 * G <= 32 * RPI, "tile too large");
  static_assert(NSUB >= 1, "at least one sub-tile");
  // MINB blocks per SM: 228 KB of shared memory less 1 KB reserved per block
  // (checked by each kernel; a geometry that does not fit may still be named
  // here, so that a kernel can pick the largest NSUB that does)
  static constexpr bool FITS = SMEM_BYTES <= (228 * 1024) / MINB - 1024;
};

// ---------------------------------------------------------------------------
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

__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// Where each sequence's cache lives and how many rows it attends.
//   pos[i]   position of sequence i: it attends rows 0..pos[i]
//   slot[i]  its slot in the cache pool [num_slots][Hkv][max_len][D]
//            (null: slot i)
//   done[i]  nonzero: finished -- scattered, but not attended (null: none)
// ---------------------------------------------------------------------------
//
// Loads here are coherent (ld.global.ca, not the read-only ld.global.nc):
// these arrays may come from the preceding kernel in the stream, which with
// programmatic dependent launch can still be writing them while this kernel
// is already resident; the read-only path is only valid for data that does
// not change during the kernel's life, and was measured to return stale
// positions in that case.
struct SeqMap {
  const int32_t *pos;
  const int32_t *slot;
  const uint8_t *done;
  int max_len;
  int num_slots;
  int Hkv;

  __device__ __forceinline__ int slot_of(int i) const { return slot ? __ldca(slot + i) : i; }
  __device__ __forceinline__ bool finished(int i) const { return done && __ldca(done + i) != 0; }
  // KVS_OK, or why sequence i can be neither scattered nor attended
  __device__ __forceinline__ int error(int i) const {
    const int p = __ldca(pos + i);
    if (p < 0 || p >= max_len) return KVS_ERR_POSITION;
    if (slot) {
      const int s = __ldca(slot + i);
      if (s < 0 || s >= num_slots) return KVS_ERR_SLOT;
    }
    return KVS_OK;
  }
  // rows attended by sequence i (0: finished, or a bad position or slot)
  __device__ __forceinline__ int len(int i) const {
    if (finished(i)) return 0;
    const int p = __ldca(pos + i);
    if (p < 0 || p >= max_len) return 0;
    if (slot) {
      const int s = __ldca(slot + i);
      if (s < 0 || s >= num_slots) return 0;
    }
    return p + 1;
  }
  // index of row r of kv head g of sequence i's cache, in rows of D floats
  __device__ __forceinline__ size_t row_index(int i, int g, int r) const {
    return ((size_t)slot_of(i) * Hkv + g) * (size_t)max_len + r;
  }
};

// ---------------------------------------------------------------------------
// One consumer warp's view of the stage ring (TileLane) and its running
// state for the current run of rows, which the caller keeps in registers:
// for each of the G heads the running max m (log2 units), the lane's share
// of the running sum and the lane's float4 column of the unnormalised
// accumulator.
//
// Warp tile: NSUB sub-tiles of RW1 rows x G heads per stage.  Lane (gi, li):
// gi = row group within a warp instruction, li = float4 column of head_dim.
// In each sub-tile a lane forms RP*G partial dot products; the transposing
// butterfly leaves lane li with the full score of slot li / SPAN (row
// slot_row of the sub-tile, head slot_h).  Scores and probabilities are kept
// per warp row u * RW1 + (row in sub-tile u).
// ---------------------------------------------------------------------------
template <class C>
struct TileLane {
  int w, lane, gi, li;
  int slot_h, slot_row;
  bool slot_used, owner;
  float *sS;     // [G][RWP] this warp's tile scores (not with SHFL_MAX)
  float *sP;     // [RW][GP] this warp's tile probabilities
  float4 *sAcc;  // [NW][G][D/4] warp accumulators at a run end
  float *sM;     // [NW][G] warp maxima at a run end
  float *sL;     // [NW][G] warp sums at a run end
  float *sLl;    // [NW][32] lane sums at a run end
};

// The lane's view; also clears this warp's score and probability tiles.
template <class C>
__device__ __forceinline__ TileLane<C> tile_lane(unsigned char *smem, int warp, int lane) {
  constexpr int G = C::G;
  TileLane<C> t;
  t.w = warp;
  t.lane = lane;
  t.gi = lane / C::LPR;
  t.li = lane % C::LPR;
  t.sS = reinterpret_cast<float *>(smem + C::OFF_SCORE) + warp * G * C::RWP;
  t.sP = reinterpret_cast<float *>(smem + C::OFF_P) + warp * C::RW * C::GP;
  t.sAcc = reinterpret_cast<float4 *>(smem + C::OFF_MACC);
  t.sM = reinterpret_cast<float *>(smem + C::OFF_MM);
  t.sL = reinterpret_cast<float *>(smem + C::OFF_ML);
  t.sLl = reinterpret_cast<float *>(smem + C::OFF_MLL);
  if (!C::SHFL_MAX)
    for (int e = lane; e < G * C::RWP; e += 32) t.sS[e] = neg_inf();
  for (int e = lane; e < C::RW * C::GP; e += 32) t.sP[e] = 0.f;
  __syncwarp();
  const int slot = t.li / C::SPAN;
  t.slot_used = slot < C::RP * G;
  t.owner = t.slot_used && (t.li % C::SPAN) == 0;
  const int slot_r = slot / G;
  t.slot_h = slot - slot_r * G;
  t.slot_row = slot_r * C::RPI + t.gi;
  return t;
}

// Running state back to "no rows yet".
template <int G>
__device__ __forceinline__ void tile_reset(float4 (&acc)[G], float (&m_run)[G], float &l_lane) {
  l_lane = 0.f;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
    m_run[h] = neg_inf();
  }
}

// q rows of the group (a run's first stage), pre-scaled by log2(e)/sqrt(D).
template <class C>
__device__ __forceinline__ void tile_load_q(const TileLane<C> &t, const unsigned char *stage,
                                            float qscale, float4 (&qv)[C::G]) {
  constexpr int G = C::G;
  const float4 *sQ = reinterpret_cast<const float4 *>(stage + 2 * C::KV_BYTES);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float4 v = sQ[h * C::LPR + t.li];
    qv[h] = make_float4(v.x * qscale, v.y * qscale, v.z * qscale, v.w * qscale);
  }
}

// Folds the stage's nrows K/V rows (this warp's tile of them) into the
// running state.
template <class C>
__device__ __forceinline__ void tile_consume(const TileLane<C> &t, const unsigned char *stage,
                                             int nrows, const float4 (&qv)[C::G],
                                             float4 (&acc)[C::G], float (&m_run)[C::G],
                                             float &l_lane) {
  constexpr int G = C::G;
  const float4 *sK = reinterpret_cast<const float4 *>(stage);
  const float4 *sV = reinterpret_cast<const float4 *>(stage + C::KV_BYTES);
  constexpr int NSUB = C::NSUB;
  // rows of sub-tile u in this stage; sub-tile 0 has the warp's lowest rows
  int valid_u[NSUB];
#pragma unroll
  for (int u = 0; u < NSUB; ++u)
    valid_u[u] = min(max(nrows - (u * C::NW + t.w) * C::RW1, 0), C::RW1);
  if (valid_u[0] <= 0) return;
  // ---- scores: partial dot products, then the butterflies (the rows past
  //      nrows hold stale data, which the valid masks below discard) ----
  float s_val[NSUB];
  bool valid[NSUB];
#pragma unroll
  for (int u = 0; u < NSUB; ++u) {
    const int base = (u * C::NW + t.w) * C::RW1;
    float part[C::NSLOT];
#pragma unroll
    for (int j = 0; j < C::NSLOT; ++j) part[j] = 0.f;
#pragma unroll
    for (int r = 0; r < C::RP; ++r) {
      const int row = base + r * C::RPI + t.gi;
      const float4 kv = sK[row * C::LPR + t.li];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float d = qv[h].x * kv.x;
        d = fmaf(qv[h].y, kv.y, d);
        d = fmaf(qv[h].z, kv.z, d);
        d = fmaf(qv[h].w, kv.w, d);
        part[r * G + h] = d;
      }
    }
    const float sc = butterfly_sum<C::NSLOT, C::LOG2NS, C::LPR>(part, t.li);
    valid[u] = t.slot_used && t.slot_row < valid_u[u];
    s_val[u] = valid[u] ? sc : neg_inf();
  }
  // ---- running max and rescale factors (all lanes, all heads) ----
  float hmax = 0.f;  // SHFL_MAX: in lane h * SPAN, the max of head h
  if (C::SHFL_MAX) {
    hmax = s_val[0];
#pragma unroll
    for (int u = 1; u < NSUB; ++u) hmax = fmaxf(hmax, s_val[u]);
    // Lane (gi, li) holds the score of slot li / SPAN = (r, h), so head h
    // sits at lanes (r * G + h) * SPAN + s of every row group gi.  First
    // over the row groups (lanes LPR apart), then over the RP rows of a
    // group (G * SPAN apart; a shift past the group's LPR lanes keeps the
    // lane's own value).  Invalid slots hold -inf.
#pragma unroll
    for (int o = C::LPR; o < 32; o <<= 1)
      hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, o));
#pragma unroll
    for (int d = G * C::SPAN; d < C::RP * G * C::SPAN; d <<= 1)
      hmax = fmaxf(hmax, __shfl_down_sync(0xffffffffu, hmax, d, C::LPR));
  } else {
    if (t.owner) {
#pragma unroll
      for (int u = 0; u < NSUB; ++u)
        t.sS[t.slot_h * C::RWP + u * C::RW1 + t.slot_row] = s_val[u];
    }
    __syncwarp();
  }
  float alpha[G];
  float m_new[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float tmax = neg_inf();
    if (C::SHFL_MAX) {
      tmax = __shfl_sync(0xffffffffu, hmax, h * C::SPAN);
    } else {
      const float4 *row4 = reinterpret_cast<const float4 *>(t.sS + h * C::RWP);
#pragma unroll
      for (int j = 0; j < C::RWP / 4; ++j) {
        const float4 v = row4[j];
        tmax = fmaxf(tmax, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
      }
    }
    m_new[h] = fmaxf(m_run[h], tmax);
    alpha[h] = (m_new[h] == m_run[h]) ? 1.f : exp2f(m_run[h] - m_new[h]);
  }
  // ---- own-slot probability ----
  float mh = m_new[0];
#pragma unroll
  for (int h = 1; h < G; ++h) mh = (t.slot_h == h) ? m_new[h] : mh;
  float ah = alpha[0];
#pragma unroll
  for (int h = 1; h < G; ++h) ah = (t.slot_h == h) ? alpha[h] : ah;
  float psum = 0.f;
#pragma unroll
  for (int u = 0; u < NSUB; ++u) {
    const float p = valid[u] ? exp2f(s_val[u] - mh) : 0.f;
    if (t.owner) t.sP[(u * C::RW1 + t.slot_row) * C::GP + t.slot_h] = p;
    psum += p;
  }
  if (t.owner) l_lane = l_lane * ah + psum;
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
  for (int u = 0; u < NSUB; ++u) {
    const int base = (u * C::NW + t.w) * C::RW1;
#pragma unroll
    for (int r = 0; r < C::RP; ++r) {
      const int trow = r * C::RPI + t.gi;
      if (trow < valid_u[u]) {
        const float4 vv = sV[(base + trow) * C::LPR + t.li];
        float pr[C::GP];
#pragma unroll
        for (int j = 0; j < C::GP / 4; ++j) {
          const float4 v =
              reinterpret_cast<const float4 *>(t.sP + (u * C::RW1 + trow) * C::GP)[j];
          pr[4 * j + 0] = v.x;
          pr[4 * j + 1] = v.y;
          pr[4 * j + 2] = v.z;
          pr[4 * j + 3] = v.w;
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
}

// End of a run: this warp's (m, l, acc) into shared memory.  The block's
// consumer warps must then synchronise before merged_warp_states() reads them.
template <class C>
__device__ __forceinline__ void tile_publish(const TileLane<C> &t, float4 (&acc)[C::G],
                                             const float (&m_run)[C::G], float l_lane) {
  constexpr int G = C::G;
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
  if (t.gi == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) t.sAcc[(t.w * G + h) * C::LPR + t.li] = acc[h];
  }
  t.sLl[t.w * 32 + t.lane] = t.owner ? l_lane : 0.f;
#pragma unroll
  for (int h = 0; h < G; ++h)
    if (t.lane == h) t.sM[t.w * G + h] = m_run[h];
  __syncwarp();
  if (t.lane < G) {
    float lsum = 0.f;
    for (int l2 = 0; l2 < 32; ++l2) {
      const int s2 = (l2 % C::LPR) / C::SPAN;
      if (s2 < C::RP * G && (s2 % G) == t.lane) lsum += t.sLl[t.w * 32 + l2];
    }
    t.sL[t.w * G + t.lane] = lsum;
  }
}

// The run's (m, l, acc) of head h = e / (D/4), float4 column d4 = e % (D/4),
// merged over the NW published warp states (m = -inf when the run has no row).
template <class C>
__device__ __forceinline__ void merged_warp_states(const unsigned char *smem, int e, float4 &a,
                                                   float &mx, float &lsum) {
  constexpr int G = C::G;
  const float4 *sAcc = reinterpret_cast<const float4 *>(smem + C::OFF_MACC);
  const float *sM = reinterpret_cast<const float *>(smem + C::OFF_MM);
  const float *sL = reinterpret_cast<const float *>(smem + C::OFF_ML);
  const int h = e / C::LPR;
  const int d4 = e - h * C::LPR;
  mx = neg_inf();
#pragma unroll
  for (int w2 = 0; w2 < C::NW; ++w2) mx = fmaxf(mx, sM[w2 * G + h]);
  a = make_float4(0.f, 0.f, 0.f, 0.f);
  lsum = 0.f;
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
}

}  // namespace
}  // namespace kvs
