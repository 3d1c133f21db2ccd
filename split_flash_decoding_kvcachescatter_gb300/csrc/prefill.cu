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
//  * Block = (head, 128 query rows), 4 warps; thread t owns query row t,
//    which is TMEM lane t of both accumulators.
//  * The Q tile is converted to FP16 once into shared memory; per tile of
//    128 keys the block converts K (rows) and V (transposed: head_dim rows
//    of 128 keys) into shared memory, in the canonical no-swizzle K-major
//    layout (8-row x 16-byte core matrices, K-adjacent ones 128 B apart).
//  * One thread issues S = Q K^T as head_dim/16 tcgen05.mma (M=128, N=128,
//    K=16) into TMEM columns [0, 128) and commits them to an mbarrier.
//  * Each thread reads its score row from TMEM (tcgen05.ld 32x32b), takes
//    the tile maximum, forms p = exp2(s - m) in FP32, rounds it to FP16 into
//    the P tile (shared memory) and sums the rounded values.
//  * One thread issues P V as 8 tcgen05.mma (M=128, N=head_dim, K=16) into
//    TMEM columns [128, 128 + head_dim); each thread folds that row into its
//    FP32 output accumulator with the online-softmax rescale.
//  * Causal: key tiles after the query tile are skipped; keys j > i and keys
//    past seq_len get p = 0.
// Every mbarrier wait is bounded; on expiry the block records
// KVS_ERR_TIMEOUT, frees its TMEM and returns.

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

// rows [row0, row0 + 128) of a [S][D] FP32 matrix -> FP16 tile [128][D]
// (rows past S are zero).
template <int D>
__device__ __forceinline__ void load_rows_f16(unsigned char *tile, const float *src, int row0,
                                              int S) {
  constexpr int CH = D / 8;  // 8-value chunks per row
  for (int e = threadIdx.x; e < kPM * CH; e += kPThreads) {
    const int r = e / CH;
    const int c = (e - r * CH) * 8;
    float x[8];
    if (row0 + r < S) {
      const float4 *p = reinterpret_cast<const float4 *>(src + (size_t)(row0 + r) * D + c);
      const float4 a = __ldg(p), b = __ldg(p + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = 0.f;
    }
    *reinterpret_cast<uint4 *>(tile + cm_off(r, c, D)) = pack8(x);
  }
}

// keys [key0, key0 + 128) of V [S][D] -> FP16 tile V^T [D][128] (keys past
// S are zero).  A warp covers 32 consecutive d of one 8-key chunk, so each
// of its 8 loads is one coalesced row segment.
template <int D>
__device__ __forceinline__ void load_vt_f16(unsigned char *tile, const float *v, int key0, int S) {
  for (int e = threadIdx.x; e < D * (kPN / 8); e += kPThreads) {
    const int d = e % D;
    const int j = (e / D) * 8;
    float x[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      x[u] = (key0 + j + u < S) ? __ldg(v + (size_t)(key0 + j + u) * D + d) : 0.f;
    *reinterpret_cast<uint4 *>(tile + cm_off(d, j, kPN)) = pack8(x);
  }
}

template <int D>
struct PGeo {
  static constexpr int Q_BYTES = kPM * D * 2;
  static constexpr int K_BYTES = kPN * D * 2;
  static constexpr int VT_BYTES = D * kPN * 2;
  static constexpr int P_BYTES = kPM * kPN * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_VT = OFF_K + K_BYTES;
  static constexpr int OFF_P = OFF_VT + VT_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;      // one mbarrier
  static constexpr int OFF_TMEM = OFF_BAR + 8;         // TMEM base address
  static constexpr int OFF_FLAG = OFF_TMEM + 8;        // abort flag (never set here)
  static constexpr int SMEM_BYTES = OFF_FLAG + 16;
};

template <int D>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_tc_kernel(const float *__restrict__ q, const float *__restrict__ k,
                      const float *__restrict__ v, float *__restrict__ out, int S, int causal,
                      float sl2, int *d_status) {
  using PG = PGeo<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  unsigned char *sQ = smem + PG::OFF_Q;
  unsigned char *sK = smem + PG::OFF_K;
  unsigned char *sVt = smem + PG::OFF_VT;
  unsigned char *sP = smem + PG::OFF_P;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + PG::OFF_BAR);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + PG::OFF_TMEM);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + PG::OFF_FLAG);

  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int h = blockIdx.y;
  const int qt = blockIdx.x;
  const int i = qt * kPM + t;  // this thread's query row
  const size_t head = (size_t)h * S * D;

  grid_dependency_wait();
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (t == 0) {
    mbar_init(bar, 1);
    *abort = 0;
    fence_mbar_init();
  }
  load_rows_f16<D>(sQ, q + head, qt * kPM, S);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t tm_s = tmem + lane_base;
  const uint32_t tm_o = tmem + lane_base + kPN;

  constexpr uint32_t kIdescS = idesc_f16_f32(kPM, kPN);
  constexpr uint32_t kIdescO = idesc_f16_f32(kPM, D);
  constexpr uint32_t kSboD = (D / 8) * 128;    // 8-row group stride, rows of D values
  constexpr uint32_t kSboN = (kPN / 8) * 128;  // 8-row group stride, rows of 128 values

  float o[D];
#pragma unroll
  for (int d = 0; d < D; ++d) o[d] = 0.f;
  float m = neg_inf_f();
  float l = 0.f;
  uint32_t phase = 0;
  bool failed = false;

  const int n_kt_all = (S + kPN - 1) / kPN;
  const int n_kt = causal ? min(qt + 1, n_kt_all) : n_kt_all;
  for (int kt = 0; kt < n_kt && !failed; ++kt) {
    const int key0 = kt * kPN;
    load_rows_f16<D>(sK, k + head, key0, S);
    load_vt_f16<D>(sVt, v + head, key0, S);
    fence_proxy_async_shared();  // the tensor cores read what the threads wrote
    __syncthreads();
    // ---- S = Q K^T into TMEM columns [0, 128) ----
    if (t == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_f16(tmem, smem_desc(sQ + ks * 256, 128, kSboD), smem_desc(sK + ks * 256, 128, kSboD),
                kIdescS, ks > 0 ? 1u : 0u);
      mma_commit(bar);
    }
    bool ok = mbar_wait(bar, phase, abort);
    phase ^= 1u;
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();
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
          const int c = ch * 32 + g8 * 8 + u;
          const int j = key0 + c;
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
    // ---- P V into TMEM columns [128, 128 + D) ----
    if (t == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kPN / 16; ++ks)
        mma_f16(tmem + kPN, smem_desc(sP + ks * 256, 128, kSboN),
                smem_desc(sVt + ks * 256, 128, kSboN), kIdescO, ks > 0 ? 1u : 0u);
      mma_commit(bar);
    }
    ok = mbar_wait(bar, phase, abort);
    phase ^= 1u;
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    tc_fence_after();
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      float r[32];
      tmem_ld32(tm_o + ch * 32, r);
      tmem_wait_ld();
#pragma unroll
      for (int u = 0; u < 32; ++u) o[ch * 32 + u] = fmaf(o[ch * 32 + u], alpha, r[u]);
    }
    tc_fence_before();
    __syncthreads();  // TMEM and the tiles are free for the next key tile
  }

  if (failed) {
    if (t == 0) record_status(d_status, KVS_ERR_TIMEOUT);
  } else if (i < S) {
    const float inv = 1.f / l;
    float4 *o4 = reinterpret_cast<float4 *>(out + head + (size_t)i * D);
#pragma unroll
    for (int d4 = 0; d4 < D / 4; ++d4)
      o4[d4] = make_float4(o[4 * d4] * inv, o[4 * d4 + 1] * inv, o[4 * d4 + 2] * inv,
                           o[4 * d4 + 3] * inv);
  }
  allow_dependent_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
int launch_prefill_impl(const float *q, const float *k, const float *v, float *out, int H, int S,
                        int causal, int *d_status, cudaStream_t stream) {
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
  const float sl2 = (float)(1.4426950408889634074 / std::sqrt((double)D));
  const dim3 grid((S + kPM - 1) / kPM, H, 1);
  const cudaError_t e = launch_pdl(prefill_tc_kernel<D>, grid, dim3(kPThreads), PG::SMEM_BYTES,
                                   stream, q, k, v, out, S, causal, sl2, d_status);
  return e == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

}  // namespace

int launch_prefill(const float *q, const float *k, const float *v, float *out, int H, int S, int D,
                   int causal, int *d_status, cudaStream_t stream) {
  if (D == 64) return launch_prefill_impl<64>(q, k, v, out, H, S, causal, d_status, stream);
  if (D == 128) return launch_prefill_impl<128>(q, k, v, out, H, S, causal, d_status, stream);
  return KVS_ERR_UNSUPPORTED;
}

}  // namespace kvs
