// prefill.cu -- attention over whole sequences (prefill) on the 5th-generation
// tensor cores: tcgen05.mma with FP16 operands in shared memory and FP32
// accumulators in tensor memory (TMEM).
//
// Source: realizar 0.8.5, src/cuda/executor/head_dim.rs,
// tensor_core_attention (PARITY-001.3): q, k, v [n_heads][seq_len][head_dim]
// given as FP32 and converted to FP16 on the GPU; S = Q K^T and P V on the
// tensor cores; FP32 output; optional causal mask.  The pages' kernel uses
// WMMA 16x16 tiles, one block of 8 warps per 16 query rows.
//
// GB300 design (flash-attention forward, one pass over the keys):
//  * A pack kernel rounds q, k and v to FP16 once into the caller's
//    workspace, already cut into 128-row tiles in the canonical no-swizzle
//    K-major layout of the tensor cores (8-row x 16-byte core matrices,
//    K-adjacent ones 128 B apart); V is stored transposed (head_dim rows of
//    128 keys), so that P V is again a K-major product.  Every tile is one
//    contiguous block.
//  * Attention block = (head, 128 query rows), 4 warps; thread t owns query
//    row t, which is TMEM lane t of both accumulators.  One thread moves each
//    tile with a single 1-D bulk asynchronous copy (TMA) into a two-stage
//    ring (K and V^T of the next key tile land while this one is computed)
//    and issues the tensor-core work:
//      S = Q K^T as head_dim/16 tcgen05.mma (M=128, N=128, K=16) into TMEM
//      columns [0, 128), and P V as 8 tcgen05.mma (M=128, N=head_dim) into
//      columns [128, 128 + head_dim), each committed to an mbarrier.
//  * Each thread reads its score row from TMEM (tcgen05.ld 32x32b), takes
//    the tile maximum, forms p = exp2(s - m) in FP32, rounds it to FP16 into
//    the P tile (shared memory) and sums the rounded values; after P V it
//    folds that row into its FP32 output with the online-softmax rescale.
//  * Causal: key tiles after the query tile are skipped; keys j > i and keys
//    past seq_len get p = 0.
// Every mbarrier wait is bounded; on expiry the block records
// KVS_ERR_TIMEOUT, lets its copies land, frees its TMEM and returns.

#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "kvs_device.cuh"
#include "kvs_launch.h"
#include "kvsdecode.h"

namespace kvs {

namespace {

constexpr int kPM = 128;         // query rows per block (MMA M)
constexpr int kPN = 128;         // keys per tile
constexpr int kPThreads = 128;   // thread t <-> query row t <-> TMEM lane t
constexpr uint32_t kTmemCols = 256;  // S tile [0, 128) + P.V tile [128, 128 + D)

// ---- tensor memory and tcgen05 (inline PTX) ---------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, FP16 inputs, FP32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The mbarrier gets one arrival when every tcgen05.mma this thread issued is done.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
  uint32_t u[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
        "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
        "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]),
        "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
        "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]),
        "=r"(u[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __uint_as_float(u[i]);
}

// 32 consecutive FP32 columns of this thread's TMEM lane, written.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(__float_as_uint(r[0])), "r"(__float_as_uint(r[1])), "r"(__float_as_uint(r[2])),
      "r"(__float_as_uint(r[3])), "r"(__float_as_uint(r[4])), "r"(__float_as_uint(r[5])),
      "r"(__float_as_uint(r[6])), "r"(__float_as_uint(r[7])), "r"(__float_as_uint(r[8])),
      "r"(__float_as_uint(r[9])), "r"(__float_as_uint(r[10])), "r"(__float_as_uint(r[11])),
      "r"(__float_as_uint(r[12])), "r"(__float_as_uint(r[13])), "r"(__float_as_uint(r[14])),
      "r"(__float_as_uint(r[15])), "r"(__float_as_uint(r[16])), "r"(__float_as_uint(r[17])),
      "r"(__float_as_uint(r[18])), "r"(__float_as_uint(r[19])), "r"(__float_as_uint(r[20])),
      "r"(__float_as_uint(r[21])), "r"(__float_as_uint(r[22])), "r"(__float_as_uint(r[23])),
      "r"(__float_as_uint(r[24])), "r"(__float_as_uint(r[25])), "r"(__float_as_uint(r[26])),
      "r"(__float_as_uint(r[27])), "r"(__float_as_uint(r[28])), "r"(__float_as_uint(r[29])),
      "r"(__float_as_uint(r[30])), "r"(__float_as_uint(r[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: no swizzle, K-major canonical layout.
//   start address, leading byte offset (K-adjacent core matrices) and stride
//   byte offset (8-row groups), each >> 4; bits 46-48 = 0b001; base offset,
//   offset mode and swizzle mode 0.
__device__ __forceinline__ uint64_t smem_desc(const void *p, uint32_t lbo, uint32_t sbo) {
  const uint32_t a = smem_addr(p);
  uint64_t d = (uint64_t)((a & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor of kind::f16: D FP32, A and B FP16, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Byte offset of element (r, c) of a tile whose rows hold C FP16 values
// (K-major): core matrix (r/8, c/8) of 8 rows x 16 bytes, K-adjacent core
// matrices 128 bytes apart (leading byte offset), 8-row groups C/8*128
// bytes apart (stride byte offset).
__device__ __forceinline__ uint32_t cm_off(int r, int c, int C) {
  return (uint32_t)((((r >> 3) * (C >> 3) + (c >> 3)) << 7) + ((r & 7) << 4) + ((c & 7) << 1));
}

__device__ __forceinline__ uint4 pack8(const float *x) {
  uint4 u;
  __half2 h;
  h = __floats2half2_rn(x[0], x[1]);
  u.x = *reinterpret_cast<uint32_t *>(&h);
  h = __floats2half2_rn(x[2], x[3]);
  u.y = *reinterpret_cast<uint32_t *>(&h);
  h = __floats2half2_rn(x[4], x[5]);
  u.z = *reinterpret_cast<uint32_t *>(&h);
  h = __floats2half2_rn(x[6], x[7]);
  u.w = *reinterpret_cast<uint32_t *>(&h);
  return u;
}

// ---- pack: FP32 [H][S][D] -> FP16 tiles in the tensor-core layout ----------
// Workspace: Q tiles, K tiles, V^T tiles, each [H][T][tile] with T =
// ceil(S / 128) and a tile of 128 * D FP16 values (rows past S are zero).
__host__ __device__ constexpr size_t prefill_tile_bytes(int D) { return (size_t)kPM * D * 2; }

template <int D>
__global__ void __launch_bounds__(256)
    prefill_pack_kernel(const float *__restrict__ q, const float *__restrict__ k,
                        const float *__restrict__ v, unsigned char *__restrict__ ws, int H, int S) {
  grid_dependency_wait();
  const int T = (S + kPM - 1) / kPM;
  const size_t tile = prefill_tile_bytes(D);
  const long long per_tensor = (long long)H * T * (kPM * D / 8);  // 16-byte chunks
  unsigned char *wq = ws;
  unsigned char *wk = ws + (size_t)H * T * tile;
  unsigned char *wv = wk + (size_t)H * T * tile;
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < 3 * per_tensor;
       e += (long long)gridDim.x * blockDim.x) {
    const int which = (int)(e / per_tensor);
    const long long f = e - (long long)which * per_tensor;
    const long long ht = f / (kPM * D / 8);  // h * T + t
    const int w = (int)(f - ht * (kPM * D / 8));
    const int h = (int)(ht / T);
    const int t = (int)(ht - (long long)h * T);
    float x[8];
    uint32_t off;
    if (which < 2) {  // Q or K: chunk w = (row r, 8 columns from c)
      const int r = w / (D / 8);
      const int c = (w - r * (D / 8)) * 8;
      const int row = t * kPM + r;
      const float *src = (which == 0 ? q : k) + ((size_t)h * S + row) * D + c;
      if (row < S) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(src) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = 0.f;
      }
      off = cm_off(r, c, D);
    } else {  // V^T: chunk w = (column d, 8 keys from j); consecutive w, consecutive d
      const int d = w % D;
      const int j = (w / D) * 8;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int key = t * kPM + j + u;
        x[u] = key < S ? __ldg(v + ((size_t)h * S + key) * D + d) : 0.f;
      }
      off = cm_off(d, j, kPN);
    }
    unsigned char *dst = (which == 0 ? wq : which == 1 ? wk : wv) + ht * tile + off;
    *reinterpret_cast<uint4 *>(dst) = pack8(x);
  }
  allow_dependent_launch();
}

template <int D>
struct PGeo {
  static constexpr int TILE = kPM * D * 2;  // one FP16 tile of Q, K or V^T
  static constexpr int P_BYTES = kPM * kPN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_STAGE = OFF_Q + TILE;             // 2 x (K tile, V^T tile)
  static constexpr int OFF_P = OFF_STAGE + 2 * 2 * TILE;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;            // q, full[2], mma
  static constexpr int OFF_TMEM = OFF_BAR + 4 * 8;           // TMEM base address
  static constexpr int OFF_FLAG = OFF_TMEM + 8;              // abort flag
  static constexpr int SMEM_BYTES = OFF_FLAG + 16;
  static_assert(SMEM_BYTES <= 227 * 1024, "one block per SM must fit");
};

template <int D>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_tc_kernel(const unsigned char *__restrict__ ws, float *__restrict__ out, int S,
                      int causal, float sl2, int *d_status) {
  using PG = PGeo<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *sQ = smem + PG::OFF_Q;
  unsigned char *sP = smem + PG::OFF_P;
  uint64_t *bar_q = reinterpret_cast<uint64_t *>(smem + PG::OFF_BAR);
  uint64_t *full = bar_q + 1;  // [2]: K and V^T tiles of a stage landed
  uint64_t *bar_mma = bar_q + 3;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + PG::OFF_TMEM);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + PG::OFF_FLAG);
  volatile int *no_abort = reinterpret_cast<volatile int *>(smem + PG::OFF_FLAG + 4);

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int h = blockIdx.y;
  const int qt = blockIdx.x;
  const int i = qt * kPM + t;  // this thread's query row
  const int T = (S + kPN - 1) / kPN;
  const int n_kt = causal ? min(qt + 1, T) : T;
  const size_t tile = (size_t)PG::TILE;
  const size_t per_tensor = (size_t)gridDim.y * T * tile;
  const unsigned char *gQ = ws + ((size_t)h * T + qt) * tile;
  const unsigned char *gKh = ws + per_tensor + (size_t)h * T * tile;
  const unsigned char *gVh = ws + 2 * per_tensor + (size_t)h * T * tile;
  auto stage_k = [&](int s) { return smem + PG::OFF_STAGE + s * 2 * PG::TILE; };
  auto stage_v = [&](int s) { return smem + PG::OFF_STAGE + s * 2 * PG::TILE + PG::TILE; };

  constexpr uint32_t kIdescS = idesc_f16_f32(kPM, kPN);
  constexpr uint32_t kIdescO = idesc_f16_f32(kPM, D);
  constexpr uint32_t kSboD = (D / 8) * 128;    // 8-row group stride, rows of D values
  constexpr uint32_t kSboN = (kPN / 8) * 128;  // 8-row group stride, rows of 128 values

  grid_dependency_wait();
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // Thread 0 moves the tiles and issues the tensor-core work.  Order of its
  // MMAs: S(0), then per key tile kt: P V(kt), S(kt+1).  One commit after
  // S(kt+1) (or after the last P V) covers both, since a commit tracks every
  // MMA the thread issued before it.
  uint32_t issued = 0;  // key tiles whose copies were issued
  int t0_ok = 1;        // thread 0: every wait so far succeeded
  auto issue_tile = [&](int st) {
    mbar_arrive_expect_tx(&full[st], 2 * PG::TILE);
    bulk_g2s(stage_k(st), gKh + issued * tile, PG::TILE, &full[st]);
    bulk_g2s(stage_v(st), gVh + issued * tile, PG::TILE, &full[st]);
    ++issued;
  };
  if (t == 0) {
    mbar_init(bar_q, 1);
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(bar_mma, 1);
    *abort = 0;
    *no_abort = 0;
    fence_mbar_init();
    mbar_arrive_expect_tx(bar_q, PG::TILE);
    bulk_g2s(sQ, gQ, PG::TILE, bar_q);
    while ((int)issued < n_kt && issued < 2) issue_tile(issued & 1);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t tm_s = tmem + lane_base;
  const uint32_t tm_o = tmem + lane_base + kPN;

  auto issue_s = [&](int kt) {  // thread 0: S(kt) = Q K(kt)^T, once K(kt) has landed
    if (!mbar_wait(&full[kt & 1], (kt >> 1) & 1, abort)) {
      t0_ok = 0;
      return;
    }
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
      mma_f16(tmem, smem_desc(sQ + ks * 256, 128, kSboD),
              smem_desc(stage_k(kt & 1) + ks * 256, 128, kSboD), kIdescS, ks > 0 ? 1u : 0u);
  };
  if (t == 0) {
    if (!mbar_wait(bar_q, 0, abort)) t0_ok = 0;
    if (t0_ok) issue_s(0);
    mma_commit(bar_mma);
  }

  float m = neg_inf_f();
  float l = 0.f;
  uint32_t mma_phase = 0;
  bool failed = false;
  for (int kt = 0; kt < n_kt; ++kt) {
    const int key0 = kt * kPN;
    const int st = kt & 1;
    // S(kt) and P V(kt-1) are done
    const bool ok = mbar_wait(bar_mma, mma_phase, abort);
    mma_phase ^= 1u;
    if (__syncthreads_or(!ok || (t == 0 && !t0_ok))) {
      failed = true;
      break;
    }
    tc_fence_after();
    // the stage of key tile kt-1 is free: bring key tile kt+1 into it
    if (t == 0 && kt >= 1 && (int)issued < n_kt) issue_tile(issued & 1);
    // ---- row maximum of the tile (masked) ----
    float mt = neg_inf_f();
#pragma unroll
    for (int ch = 0; ch < kPN / 32; ++ch) {
      float r[32];
      tmem_ld32(tm_s + ch * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const int j = key0 + ch * 32 + u;
        const bool live = j < S && (!causal || j <= i);
        if (live) mt = fmaxf(mt, r[u] * sl2);
      }
    }
    const float m_new = fmaxf(m, mt);
    const float alpha = (m_new == neg_inf_f()) ? 1.f : exp2f(m - m_new);
    // ---- rescale the output accumulator (TMEM) where the maximum moved ----
    if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        float r[32];
        tmem_ld32(tm_o + ch * 32, r);
        tmem_wait_ld();
#pragma unroll
        for (int u = 0; u < 32; ++u) r[u] *= alpha;
        tmem_st32(tm_o + ch * 32, r);
      }
      tmem_wait_st();
    }
    // ---- P (FP16) into shared memory, and its row sum ----
    float lt = 0.f;
#pragma unroll
    for (int ch = 0; ch < kPN / 32; ++ch) {
      float r[32];
      tmem_ld32(tm_s + ch * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        float p8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int j = key0 + ch * 32 + g8 * 8 + u;
          const bool live = j < S && (!causal || j <= i) && m_new != neg_inf_f();
          const float p = live ? exp2f(r[g8 * 8 + u] * sl2 - m_new) : 0.f;
          p8[u] = __half2float(__float2half_rn(p));
          lt += p8[u];
        }
        *reinterpret_cast<uint4 *>(sP + cm_off(t, ch * 32 + g8 * 8, kPN)) = pack8(p8);
      }
    }
    l = l * alpha + lt;
    m = m_new;
    fence_proxy_async_shared();
    tc_fence_before();
    __syncthreads();
    // ---- thread 0: O (+)= P V(kt), then S(kt+1) ----
    if (t == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kPN / 16; ++ks)
        mma_f16(tmem + kPN, smem_desc(sP + ks * 256, 128, kSboN),
                smem_desc(stage_v(st) + ks * 256, 128, kSboN), kIdescO,
                (kt > 0 || ks > 0) ? 1u : 0u);
      if (kt + 1 < n_kt && t0_ok) issue_s(kt + 1);
      mma_commit(bar_mma);
    }
  }
  if (!failed) {  // the last P V
    const bool ok = mbar_wait(bar_mma, mma_phase, abort);
    failed = __syncthreads_or(!ok);
  }

  if (failed) {
    if (t == 0) {
      *abort = 1;
      record_status(d_status, KVS_ERR_TIMEOUT);
      // let the copies already issued land before the block exits
      mbar_wait(bar_q, 0, no_abort);
      for (uint32_t j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
        mbar_wait(&full[j & 1], (j >> 1) & 1, no_abort);
    }
  } else {
    tc_fence_after();
    const float inv = 1.f / l;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      float r[32];
      tmem_ld32(tm_o + ch * 32, r);
      tmem_wait_ld();
      if (i < S) {
        float4 *o4 = reinterpret_cast<float4 *>(out + ((size_t)h * S + i) * D + ch * 32);
#pragma unroll
        for (int u = 0; u < 8; ++u)
          o4[u] = make_float4(r[4 * u] * inv, r[4 * u + 1] * inv, r[4 * u + 2] * inv,
                              r[4 * u + 3] * inv);
      }
    }
  }
  allow_dependent_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
int launch_prefill_impl(const float *q, const float *k, const float *v, float *out, int H, int S,
                        int causal, void *workspace, int *d_status, cudaStream_t stream) {
  using PG = PGeo<D>;
  static bool configured[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVS_ERR_LAUNCH;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PG::SMEM_BYTES) != cudaSuccess) {
      cudaGetLastError();
      return KVS_ERR_LAUNCH;
    }
    configured[dev] = true;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return KVS_ERR_LAUNCH;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  cudaError_t e = launch_pdl(prefill_pack_kernel<D>, dim3(sms * 4), dim3(256), 0, stream, q, k, v,
                             ws, H, S);
  if (e != cudaSuccess) return KVS_ERR_LAUNCH;
  const float sl2 = (float)(1.4426950408889634074 / std::sqrt((double)D));
  const dim3 grid((S + kPM - 1) / kPM, H, 1);
  e = launch_pdl(prefill_tc_kernel<D>, grid, dim3(kPThreads), PG::SMEM_BYTES, stream,
                 static_cast<const unsigned char *>(ws), out, S, causal, sl2, d_status);
  return e == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

}  // namespace

size_t prefill_workspace_bytes(int H, int S, int D) {
  const size_t T = ((size_t)S + kPM - 1) / kPM;
  return 3 * (size_t)H * T * prefill_tile_bytes(D);
}

int launch_prefill(const float *q, const float *k, const float *v, float *out, int H, int S, int D,
                   int causal, void *workspace, int *d_status, cudaStream_t stream) {
  if (D == 64)
    return launch_prefill_impl<64>(q, k, v, out, H, S, causal, workspace, d_status, stream);
  if (D == 128)
    return launch_prefill_impl<128>(q, k, v, out, H, S, causal, workspace, d_status, stream);
  return KVS_ERR_UNSUPPORTED;
}

}  // namespace kvs
