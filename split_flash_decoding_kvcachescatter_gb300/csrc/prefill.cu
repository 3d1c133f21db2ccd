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
//  * q, k and v are rounded to FP16 once into the caller's workspace,
//    already cut into 128-row tiles in the canonical no-swizzle K-major
//    layout of the tensor cores (8-row x 16-byte core matrices, K-adjacent
//    ones 128 B apart); V is stored transposed (head_dim rows of 128 keys),
//    so that P V is again a K-major product.  Every tile is one contiguous
//    block, moved later by a single 1-D bulk copy (TMA).  The tiles needed
//    first (the first round's Q tiles, the first 60 % of the key tiles) are
//    packed by a separate launch at full bandwidth; two warps of the
//    attention kernel pack the rest while it runs, in the order the items
//    need them, and publish each tile with a flag that the copy warp waits
//    for.
//  * Attention work item = (head, two 128-row query tiles A and B); a
//    persistent grid of one 12-warp block per SM walks the items, longest
//    first, in a snake order across the blocks.  Warpgroup 0 runs the
//    softmax of tile A, warpgroup 1 that of tile B (thread t owns query row
//    t, which is TMEM lane t), warp 8 issues the tensor-core work
//    (tcgen05.mma, M = 128, K = 16, FP32 accumulators in TMEM, completion by
//    tcgen05.commit on mbarriers) in the order P V_A(kt), S_A(kt+1),
//    P V_B(kt), S_B(kt+1), warp 9 moves the tiles (K and V^T through two
//    stages each), and warps 10-11 pack, so one tile's softmax runs while
//    the other tile's products are on the tensor cores.  The barriers count
//    on across items: the next item's tiles load and its first products run
//    while the softmax warps write the current item's output.
//  * Softmax: each thread reads its score row from TMEM (tcgen05.ld 32x32b,
//    64 columns at a time) once: p = 2^(s - m) on the special-function unit
//    against a reference maximum, rounded to FP16 and written back over
//    scores already read (tcgen05.st), where P V takes it as its A operand;
//    the FP32 values are summed into the row sum.  The reference maximum
//    moves only when the row maximum grows by more than 2^8 (log2 units), so
//    P written earlier and the output accumulator in TMEM are rarely
//    rescaled.
//  * Causal: key tiles after the query tile are skipped; keys j > i and keys
//    past seq_len get p = 0 (selects, on the diagonal and last tiles only).
// Every wait (mbarriers, tile flags) is bounded; on expiry the block records
// KVS_ERR_TIMEOUT, lets its copies and tensor-core products finish, frees its
// TMEM and returns.

#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "kvs_device.cuh"
#include "kvs_launch.h"
#include "kvsdecode.h"

namespace kvs {

namespace {

constexpr int kPM = 128;         // query rows per block (MMA M)
constexpr int kPN = 128;         // keys per tile

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
// D[tmem] (+)= A[tmem] * B[smem]^T: A (M rows in TMEM lanes, K FP16 values
// packed two per 32-bit column, the lower half first), FP16 inputs, FP32
// accumulate.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
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
// 64 consecutive FP32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&r)[64]) {
  uint32_t u[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31]), "=r"(u[32]), "=r"(u[33]), "=r"(u[34]), "=r"(u[35]), "=r"(u[36]), "=r"(u[37]), "=r"(u[38]), "=r"(u[39]), "=r"(u[40]), "=r"(u[41]), "=r"(u[42]), "=r"(u[43]), "=r"(u[44]), "=r"(u[45]), "=r"(u[46]), "=r"(u[47]), "=r"(u[48]), "=r"(u[49]), "=r"(u[50]), "=r"(u[51]), "=r"(u[52]), "=r"(u[53]), "=r"(u[54]), "=r"(u[55]), "=r"(u[56]), "=r"(u[57]), "=r"(u[58]), "=r"(u[59]), "=r"(u[60]), "=r"(u[61]), "=r"(u[62]), "=r"(u[63])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 64; ++i) r[i] = __uint_as_float(u[i]);
}
// 32 consecutive 32-bit columns of this thread's TMEM lane, as raw words.
__device__ __forceinline__ void tmem_ld32u(uint32_t taddr, uint32_t (&w)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]), "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]), "=r"(w[15]), "=r"(w[16]), "=r"(w[17]), "=r"(w[18]), "=r"(w[19]), "=r"(w[20]), "=r"(w[21]), "=r"(w[22]), "=r"(w[23]), "=r"(w[24]), "=r"(w[25]), "=r"(w[26]), "=r"(w[27]), "=r"(w[28]), "=r"(w[29]), "=r"(w[30]), "=r"(w[31])
      : "r"(taddr));
}
// 32 consecutive 32-bit columns of this thread's TMEM lane, written.
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&w)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15]), "r"(w[16]), "r"(w[17]), "r"(w[18]), "r"(w[19]), "r"(w[20]), "r"(w[21]), "r"(w[22]), "r"(w[23]), "r"(w[24]), "r"(w[25]), "r"(w[26]), "r"(w[27]), "r"(w[28]), "r"(w[29]), "r"(w[30]), "r"(w[31])
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

// 2^x on the special-function unit (inputs far below the FP32 range give 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Keys of a tile that a row does not attend become -inf (no branches).
__device__ __forceinline__ void mask_keys(float (&r)[32], int key0, int S, bool causal, int i) {
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    const int j = key0 + u;
    r[u] = (j < S && (!causal || j <= i)) ? r[u] : -__int_as_float(0x7f800000);
  }
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

// ---- packing: FP32 [H][S][D] -> FP16 tiles in the tensor-core layout ------
// Workspace: a flag per tile and a task counter (zeroed before every launch),
// padded to 256 bytes, then the Q tiles, K tiles and V^T tiles, each
// [H][T][tile] with T = ceil(S / 128) and a tile of 128 * D FP16 values
// (rows past S are zero).
__host__ __device__ constexpr size_t prefill_tile_bytes(int D) { return (size_t)kPM * D * 2; }
__host__ __device__ constexpr size_t prefill_flag_bytes(int H, int T) {
  return ((4 * (3 * (size_t)H * T + 1)) + 255) / 256 * 256;
}

// One tile of the packing work: tensor 0 (Q), 1 (K) or 2 (V^T), head h,
// tile t.
struct PTile {
  int tensor, h, t;
};

// Query tiles of the pair with rank pr in the item list (see prefill_item).
__device__ __forceinline__ int prefill_pair_tiles(int pr, int T, int causal, int *qa) {
  const int np = (T + 1) / 2;
  *qa = 2 * (causal ? np - 1 - pr : pr);
  return *qa + 1 < T ? 2 : 1;
}

// Task `task` of the in-kernel packing list, in the order the attention
// items need the tiles: K and V^T key tile by key tile from tile s0 (tile s
// of every head), the Q tiles of one further pair rank (from rq) after every
// second key tile, and the Q tiles left at the end.  The Q tiles of pair
// ranks below rq and the K and V^T tiles below s0 are packed before the
// attention kernel starts.
__device__ PTile prefill_task(int task, int H, int T, int causal, int rq, int s0) {
  const int np = (T + 1) / 2;
  int qa = 0;
  int next = rq;
  for (int s = s0; s < T; ++s) {
    if (task < 2 * H) return PTile{1 + (task & 1), task >> 1, s};
    task -= 2 * H;
    if (((s - s0) & 1) && next < np) {
      const int nq = prefill_pair_tiles(next, T, causal, &qa);
      if (task < H * nq) return PTile{0, task / nq, qa + task % nq};
      task -= H * nq;
      ++next;
    }
  }
  for (; next < np; ++next) {
    const int nq = prefill_pair_tiles(next, T, causal, &qa);
    if (task < H * nq) return PTile{0, task / nq, qa + task % nq};
    task -= H * nq;
  }
  return PTile{0, 0, 0};  // not reached for task < the list's length
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(unsigned *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Orders this thread's generic-proxy view of global memory with its later
// bulk (async-proxy) copies.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Warp-collective: waits until the flag of tile n (of f[0, last)) is set.
// Lane j reads the flag of tile n + j (acquire), so one round trip learns
// about 32 tiles; `mask` keeps which of [base, base + 32) were seen set, and
// a tile already seen costs nothing.  Bound and abort as in mbar_wait; the
// outcome is the same in every lane.
template <bool kPoll>
__device__ __forceinline__ bool tile_wait(const unsigned *f, int n, int last, uint32_t &mask,
                                          int &base, volatile int *abort, int lane) {
  if (n >= base && n - base < 32 && ((mask >> (n - base)) & 1u)) return true;
  base = n;
  auto look = [&]() {
    const int t = n + lane;
    return __ballot_sync(0xffffffffu, t < last && ld_acquire_u32(f + t) != 0u);
  };
  mask = look();
  if (mask & 1u) return true;
  const uint64_t limit = kPoll ? (uint64_t)g_wait_limit_ns : kWaitLimitNs;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (!kPoll) __nanosleep(128);
    mask = look();
    if (mask & 1u) return true;
    int stop = 0;
    if (lane == 0) stop = (*abort != 0) || (global_timer_ns() - t0 >= limit);
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
}

// The tiles needed first, packed at full bandwidth before the attention
// starts: grid (pieces * D/16, H); piece z of a head is a Q tile of a pair
// rank below rq (two per rank), then K and V^T of key tiles 0, 1, ...;
// block j of a Q or K tile converts 256 16-byte pieces, of a V^T tile 16 of
// its D rows (staged through shared memory).  Each tile's flag is set for
// the attention kernel, which reads it only after this kernel completed.
template <int D>
__global__ void __launch_bounds__(256)
    prefill_pack_kernel(const float *__restrict__ q, const float *__restrict__ k,
                        const float *__restrict__ v, unsigned char *__restrict__ ws, int H, int S,
                        int causal, int rq) {
  constexpr int kVPad = kPN + 4;
  __shared__ __align__(16) float sv[16 * kVPad];
  grid_dependency_wait();
  const int T = (S + kPM - 1) / kPM;
  PTile p;
  p.h = blockIdx.y;
  const int z = (int)blockIdx.x / (D / 16);
  const int bx = (int)blockIdx.x % (D / 16);
  if (z < 2 * rq) {
    int qa = 0;
    const int nq = prefill_pair_tiles(z >> 1, T, causal, &qa);
    if ((z & 1) >= nq) return;  // the pair has no tile B
    p.tensor = 0;
    p.t = qa + (z & 1);
  } else {
    p.tensor = 1 + ((z - 2 * rq) & 1);
    p.t = (z - 2 * rq) >> 1;
  }
  const size_t tile = prefill_tile_bytes(D);
  unsigned *flags = reinterpret_cast<unsigned *>(ws);
  unsigned char *dst = ws + prefill_flag_bytes(H, T) + (((size_t)p.tensor * H + p.h) * T + p.t) * tile;
  if (p.tensor < 2) {
    const int w = bx * 256 + threadIdx.x;
    const int r = (w / (8 * (D / 8))) * 8 + (w & 7);
    const int c = ((w >> 3) % (D / 8)) * 8;
    const int row = p.t * kPM + r;
    float x[8];
    if (row < S) {
      const float4 *src = reinterpret_cast<const float4 *>((p.tensor == 0 ? q : k) +
                                                           ((size_t)p.h * S + row) * D + c);
      const float4 a = __ldcg(src), b = __ldcg(src + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
      x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = 0.f;
    }
    *reinterpret_cast<uint4 *>(dst + cm_off(r, c, D)) = pack8(x);
  } else {
    const int d0 = bx * 16;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int e = threadIdx.x + 256 * u;
      const int key = e >> 2, f4 = e & 3;
      const int gkey = p.t * kPN + key;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (gkey < S)
        a = __ldcg(reinterpret_cast<const float4 *>(v + ((size_t)p.h * S + gkey) * D + d0) + f4);
      sv[(4 * f4 + 0) * kVPad + key] = a.x;
      sv[(4 * f4 + 1) * kVPad + key] = a.y;
      sv[(4 * f4 + 2) * kVPad + key] = a.z;
      sv[(4 * f4 + 3) * kVPad + key] = a.w;
    }
    __syncthreads();
    const int w = threadIdx.x;
    const int dr = 8 * (w >> 7) + (w & 7);
    const int g = (w >> 3) & 15;
    const float4 *row4 = reinterpret_cast<const float4 *>(sv + dr * kVPad + 8 * g);
    const float4 a = row4[0], b = row4[1];
    const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    *reinterpret_cast<uint4 *>(dst + cm_off(d0 + dr, 8 * g, kPN)) = pack8(x);
  }
  // read only after this kernel has completed (the attention's dependency wait)
  if (bx == 0 && threadIdx.x == 0) flags[((size_t)p.tensor * H + p.h) * T + p.t] = 1u;
  allow_dependent_launch();
}

// Block layout: two 128-row query tiles (A = qa, B = qa + 1) share every K
// and V^T tile.  Warpgroup 0 does the softmax of tile A, warpgroup 1 that of
// tile B (thread t of a warpgroup owns row t, TMEM lane t), warp 8 issues
// the tensor-core work, warp 9 moves the tiles and warps 10-11 pack tiles,
// so one tile's softmax runs while the other tile's products are on the
// tensor cores.  TMEM columns: S_A [0, 128), S_B [128, 256),
// O_A [256, 256 + D), O_B [256 + D, 256 + 2D).  The softmax writes P_x in
// FP16 over the first 64 columns of S_x (two values per column) and P V
// reads it from there, so no shared memory holds P; K and V^T have two
// stages each (a third V^T stage measured no faster), and the pack warps'
// staging takes the room a third stage would.
//
// The grid is persistent: one block per SM walks a list of items (head,
// pair of query tiles).  Its barriers keep counting from one item to the
// next, so the copy warp loads the next item's Q and first K and V^T tiles,
// and the tensor-core warp starts its S products, while the softmax warps
// still write the current item's output rows.
constexpr int kPWarpgroups = 2;
constexpr float kRescaleLog2 = 8.f;
constexpr int kPMmaWarp = 4 * kPWarpgroups;            // warp 8
constexpr int kPCopyWarp = kPMmaWarp + 1;              // warp 9
constexpr int kPPackWarp0 = kPCopyWarp + 1;            // warps 10 and 11
constexpr int kPPackWarps = 2;
constexpr int kPBlockThreads = (kPPackWarp0 + kPPackWarps) * 32;  // 384
constexpr int kPStgRows = 16;                          // rows of one staged chunk
constexpr uint32_t kPTmemCols = 512;

template <int D>
struct PGeo {
  static constexpr int TILE = kPM * D * 2;  // one FP16 tile of Q, K or V^T
  static constexpr int OFF_Q = 0;                        // Q_A, Q_B
  static constexpr int KS = 2;                           // K stages
  static constexpr int VS = 2;                           // V^T stages
  static constexpr int OFF_K = OFF_Q + 2 * TILE;
  static constexpr int OFF_V = OFF_K + KS * TILE;
  // staging of the pack warps: two buffers each of kPStgRows FP32 rows,
  // padded by 16 bytes (conflict-free reads along a row and down a column)
  static constexpr int STG_STRIDE = D + 4;                 // floats per staged row
  static constexpr int STG_BUF = kPStgRows * STG_STRIDE * 4;
  static constexpr int OFF_STG = OFF_V + VS * TILE;
  static constexpr int OFF_BAR = OFF_STG + kPPackWarps * 2 * STG_BUF;
  // barriers: q, qfree, kfull[KS], kfree[KS], vfull[VS], vfree[VS], sfull[2],
  // pfull[2], pvdone, odone[2], staging[2 * kPPackWarps]
  static constexpr int NBAR = 2 + 2 * KS + 2 * VS + 7 + 2 * kPPackWarps;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;    // TMEM base address
  static constexpr int OFF_FLAG = OFF_TMEM + 8;          // abort
  // A block holds all 512 TMEM columns, so a second block on the SM would
  // only wait for them: ask for more than half of the SM's 228 KB of shared
  // memory (less the 1 KB each block reserves) so that one block fits.
  static constexpr int ONE_PER_SM = 116 * 1024;
  static constexpr int SMEM_BYTES = OFF_FLAG + 16 > ONE_PER_SM ? OFF_FLAG + 16 : ONE_PER_SM;
  static_assert(SMEM_BYTES <= 227 * 1024, "one block per SM must fit");
};

// One work item: head h and the query tiles qa (A) and qa + 1 (B, absent
// when qa + 1 == T), with the key tiles each attends.
struct PItem {
  int h, qa, n_a, n_b, n_all;
  bool has_b;
};

// Item idx of the list: head fastest; with the causal mask, the pairs with
// the most key tiles first (longest first across the blocks).
__device__ __forceinline__ PItem prefill_item(int idx, int H, int T, int causal) {
  PItem it;
  const int pr = idx / H;
  it.h = idx - pr * H;
  it.qa = 2 * (causal ? (T + 1) / 2 - 1 - pr : pr);
  it.has_b = it.qa + 1 < T;
  it.n_a = causal ? it.qa + 1 : T;
  it.n_b = it.has_b ? (causal ? it.qa + 2 : T) : 0;
  it.n_all = it.n_a > it.n_b ? it.n_a : it.n_b;
  return it;
}

// Item of round r for block b of P: rounds of P consecutive items, the
// block order reversed every other round (a snake), so that the heavy and
// the light end of the longest-first list even out across the blocks
// (within 2 % of a greedy dynamic schedule for the causal case).  Indexes
// only grow with r, so the first one past the list ends the walk.
__device__ __forceinline__ int prefill_item_index(int b, int r, int P) {
  return r * P + ((r & 1) ? P - 1 - b : b);
}

template <int D, bool kPoll>
__global__ void __launch_bounds__(kPBlockThreads, 1)
    prefill_tc_kernel(const float *__restrict__ q, const float *__restrict__ k,
                      const float *__restrict__ v, unsigned char *__restrict__ ws,
                      float *__restrict__ out, int H, int S, int causal, float sl2,
                      int *d_status, int rq, int s0, int nt_in) {
  using PG = PGeo<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + PG::OFF_BAR);
  constexpr int KS = PG::KS, VS = PG::VS;
  uint64_t *bar_q = bars + 0;      // Q_A, Q_B of the item landed
  uint64_t *qfree = bar_q + 1;     // the item's S products done (commit): Q may be replaced
  uint64_t *kfull = qfree + 1;     // [KS] K stage landed
  uint64_t *kfree = kfull + KS;    // [KS] the S products reading a K stage done (commit)
  uint64_t *vfull = kfree + KS;    // [VS] V^T stage landed
  uint64_t *vfree = vfull + VS;    // [VS] the P V products reading a V^T stage done (commit)
  uint64_t *sfull = vfree + VS;    // [2] S_x ready (commit)
  uint64_t *pfull = sfull + 2;     // [2] P_x written, O_x rescaled (128 arrivals)
  uint64_t *pvdone = pfull + 2;    // every product issued so far is done (commit)
  uint64_t *odone = pvdone + 1;    // [2] the item's last P V_x done: O_x final (commit)
  uint64_t *stgfull = odone + 2;   // [2 * kPPackWarps] a staged chunk landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + PG::OFF_TMEM);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + PG::OFF_FLAG);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int T = (S + kPN - 1) / kPN;   // query tiles = key tiles
  const int NI = H * ((T + 1) / 2);    // items
  const int P = (int)gridDim.x;
  const int b = (int)blockIdx.x;
  const size_t tile = (size_t)PG::TILE;
  const size_t per_tensor = (size_t)H * T * tile;
  unsigned *flags = reinterpret_cast<unsigned *>(ws);  // [3][H][T] tile packed, then the counter
  unsigned char *tiles = ws + prefill_flag_bytes(H, T);

  constexpr uint32_t kIdescS = idesc_f16_f32(kPM, kPN);
  constexpr uint32_t kIdescO = idesc_f16_f32(kPM, D);
  constexpr uint32_t kSboD = (D / 8) * 128;    // 8-row group stride, rows of D values
  constexpr uint32_t kSboN = (kPN / 8) * 128;  // 8-row group stride, rows of 128 values

  grid_dependency_wait();
  if (warp == 0) {
    tmem_alloc(tmem_slot, kPTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(qfree, 1);
    for (int j = 0; j < KS; ++j) {
      mbar_init(&kfull[j], 1);
      mbar_init(&kfree[j], 1);
    }
    for (int j = 0; j < VS; ++j) {
      mbar_init(&vfull[j], 1);
      mbar_init(&vfree[j], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sfull[x], 1);
      mbar_init(&pfull[x], kPM);
    }
    mbar_init(pvdone, 1);
    mbar_init(&odone[0], 1);
    mbar_init(&odone[1], 1);
    for (int j = 0; j < 2 * kPPackWarps; ++j) mbar_init(&stgfull[j], 1);
    *abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp == kPCopyWarp) {
    // ======================= copies ==========================================
    // Tiles are counted over all items: K tile number nk goes to stage
    // nk % KS once the S products of tile nk - KS are done, V^T tile nv to
    // stage nv % VS once the P V products of tile nv - VS are.  Item j's Q
    // replaces item j - 1's once the S products of item j - 1 are done.
    // The whole warp runs the loop (it reads the tile flags 32 at a time);
    // lane 0 issues the copies.
    {
      unsigned char *sQ = smem + PG::OFF_Q;
      unsigned char *sK = smem + PG::OFF_K;
      unsigned char *sV = smem + PG::OFF_V;
      int nk = 0, nv = 0;  // K and V^T tiles issued
      int jq = -1;         // the last item whose Q was issued
      bool ok = true;
      for (int rd = 0; ok; ++rd) {
        const int idx = prefill_item_index(b, rd, P);
        if (idx >= NI) break;
        const PItem it = prefill_item(idx, H, T, causal);
        const unsigned char *gQh = tiles + (size_t)it.h * T * tile;
        const unsigned char *gKh = gQh + per_tensor;
        const unsigned char *gVh = gQh + 2 * per_tensor;
        if (rd > 0 &&
            !(ok = __all_sync(0xffffffffu, mbar_wait<kPoll>(qfree, (uint32_t)(rd - 1) & 1u, abort))))
          break;
        // a tile is bulk-copied only once a pack warp has published it
        const unsigned *fq = flags + (size_t)it.h * T;
        const unsigned *fk = fq + (size_t)H * T;
        const unsigned *fv = fk + (size_t)H * T;
        uint32_t mq = 0, mk = 0, mv = 0;
        int bq = 0, bk = 0, bv = 0;
        // (tiles packed before this kernel started need no look)
        if (idx / H >= rq) {
          if (!(ok = tile_wait<kPoll>(fq, it.qa, T, mq, bq, abort, lane))) break;
          if (it.has_b && !(ok = tile_wait<kPoll>(fq, it.qa + 1, T, mq, bq, abort, lane))) break;
        }
        if (lane == 0) {
          fence_proxy_async_global();
          mbar_arrive_expect_tx(bar_q, (it.has_b ? 2 : 1) * PG::TILE);
          bulk_g2s(sQ, gQh + (size_t)it.qa * tile, PG::TILE, bar_q);
          if (it.has_b) bulk_g2s(sQ + PG::TILE, gQh + (size_t)(it.qa + 1) * tile, PG::TILE, bar_q);
        }
        jq = rd;
        for (int n = 0; n < it.n_all; ++n) {
          const int ks = nk % KS, vs = nv % VS;
          if (nk >= KS &&
              !(ok = __all_sync(0xffffffffu, mbar_wait<kPoll>(&kfree[ks],
                                                               (uint32_t)((nk - KS) / KS) & 1u, abort))))
            break;
          if (n >= s0 && !(ok = tile_wait<kPoll>(fk, n, it.n_all, mk, bk, abort, lane))) break;
          if (lane == 0) {
            fence_proxy_async_global();
            mbar_arrive_expect_tx(&kfull[ks], PG::TILE);
            bulk_g2s(sK + ks * PG::TILE, gKh + (size_t)n * tile, PG::TILE, &kfull[ks]);
          }
          ++nk;
          if (nv >= VS &&
              !(ok = __all_sync(0xffffffffu, mbar_wait<kPoll>(&vfree[vs],
                                                               (uint32_t)((nv - VS) / VS) & 1u, abort))))
            break;
          if (n >= s0 && !(ok = tile_wait<kPoll>(fv, n, it.n_all, mv, bv, abort, lane))) break;
          if (lane == 0) {
            fence_proxy_async_global();
            mbar_arrive_expect_tx(&vfull[vs], PG::TILE);
            bulk_g2s(sV + vs * PG::TILE, gVh + (size_t)n * tile, PG::TILE, &vfull[vs]);
          }
          ++nv;
        }
      }
      if (lane == 0) {
        if (!ok) {
          *abort = 1;
          record_status(d_status, KVS_ERR_TIMEOUT);
        }
        // Every copy issued lands before the block can exit, also when
        // another role gave up and no longer waits for it.  Only the latest
        // Q load and the last KS K tiles and VS V^T tiles can still be in
        // flight (an earlier one landed before its slot was refilled), so
        // each wait is for its own phase.
        if (jq >= 0) mbar_wait_drain(bar_q, (uint32_t)jq & 1u);
        for (int j = (nk > KS ? nk - KS : 0); j < nk; ++j)
          mbar_wait_drain(&kfull[j % KS], (uint32_t)(j / KS) & 1u);
        for (int j = (nv > VS ? nv - VS : 0); j < nv; ++j)
          mbar_wait_drain(&vfull[j % VS], (uint32_t)(j / VS) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == kPMmaWarp) {
    // ======================= tensor-core work ================================
    if (lane == 0) {
      // shared-memory descriptors of the tiles; step ks of a product adds
      // ks * 256 bytes (16 in the descriptor's address field)
      const uint64_t dq0 = smem_desc(smem + PG::OFF_Q, 128, kSboD);
      const uint64_t dk0 = smem_desc(smem + PG::OFF_K, 128, kSboD);
      const uint64_t dv0 = smem_desc(smem + PG::OFF_V, 128, kSboN);
      constexpr uint64_t kTileStep = PG::TILE >> 4;  // one tile further on
      int gk = 0, gv = 0;      // K and V^T tile numbers of the item's tile 0
      int sb[2] = {0, 0};      // S_x products of the earlier items
      uint32_t pv_phase = 0;
      bool ok = true;
      bool issued = false;   // products issued since the last completed pvdone wait
      bool pending = false;  // a commit on pvdone whose wait did not complete
      for (int rd = 0; ok; ++rd) {
        const int idx = prefill_item_index(b, rd, P);
        if (idx >= NI) break;
        const PItem it = prefill_item(idx, H, T, causal);
        auto issue_s = [&](int x, int n) {  // S_x(n) = Q_x K(n)^T
          const uint64_t a = dq0 + (x ? kTileStep : 0);
          const uint64_t bk = dk0 + (uint64_t)((gk + n) % KS) * kTileStep;
          const uint32_t d = tmem + x * kPN;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            mma_f16(d, a + 16 * ks, bk + 16 * ks, kIdescS, ks > 0 ? 1u : 0u);
          mma_commit(&sfull[x]);
        };
        auto issue_pv = [&](int x, int n) {  // O_x (+)= P_x(n) V^T(n), P_x from TMEM
          const uint64_t bv = dv0 + (uint64_t)((gv + n) % VS) * kTileStep;
          const uint32_t d = tmem + 2 * kPN + x * D;
          const uint32_t a = tmem + x * kPN;
#pragma unroll
          for (int ks = 0; ks < kPN / 16; ++ks)
            mma_f16_ts(d, a + ks * 8, bv + 16 * ks, kIdescO, (n > 0 || ks > 0) ? 1u : 0u);
        };
        ok = mbar_wait<kPoll>(bar_q, (uint32_t)rd & 1u, abort) &&
             mbar_wait<kPoll>(&kfull[gk % KS], (uint32_t)(gk / KS) & 1u, abort);
        if (!ok) break;
        tc_fence_after();
        issue_s(0, 0);
        if (it.n_b > 0) issue_s(1, 0);
        mma_commit(&kfree[gk % KS]);
        if (it.n_all == 1) mma_commit(qfree);
        issued = true;
        for (int kt = 0; kt < it.n_all && ok; ++kt) {
          const int gvk = gv + kt;
          ok = mbar_wait<kPoll>(&vfull[gvk % VS], (uint32_t)(gvk / VS) & 1u, abort);  // V^T(kt)
          bool k_next = false;  // K(kt+1) has landed
          for (int x = 0; x < 2 && ok; ++x) {
            const int n_x = x == 0 ? it.n_a : it.n_b;
            if (kt < n_x) {  // P V_x(kt), once softmax x(kt) has written P_x
              ok = mbar_wait<kPoll>(&pfull[x], (uint32_t)(sb[x] + kt) & 1u, abort);
              if (!ok) break;
              tc_fence_after();
              issue_pv(x, kt);
              issued = true;
              // O_x is final once its last product is done.  (A tile without
              // products gets no commit, and its softmax warps no wait, so
              // they never fall a phase behind.)
              if (kt + 1 == n_x) mma_commit(&odone[x]);
            }
            if (kt + 1 < n_x) {  // S_x(kt+1) overwrites P_x(kt): after P V_x(kt)
              mma_commit(pvdone);
              ok = mbar_wait<kPoll>(pvdone, pv_phase, abort);
              if (!ok) {
                pending = true;
                break;
              }
              pv_phase ^= 1u;
              issued = false;
              if (!k_next) {
                const int gkn = gk + kt + 1;
                ok = mbar_wait<kPoll>(&kfull[gkn % KS], (uint32_t)(gkn / KS) & 1u, abort);
                if (!ok) break;
                tc_fence_after();
                k_next = true;
              }
              issue_s(x, kt + 1);
              issued = true;
            }
          }
          if (!ok) break;
          mma_commit(&vfree[gvk % VS]);                                   // P V(kt)
          if (kt + 1 < it.n_all) mma_commit(&kfree[(gk + kt + 1) % KS]);  // S(kt+1)
          if (kt + 2 == it.n_all) mma_commit(qfree);  // the item's last S products
        }
        if (!ok) break;
        // the item's last P V products done: the next item's S_x may
        // overwrite P_x
        mma_commit(pvdone);
        ok = mbar_wait<kPoll>(pvdone, pv_phase, abort);
        if (!ok) {
          pending = true;
          break;
        }
        pv_phase ^= 1u;
        issued = false;
        gk += it.n_all;
        gv += it.n_all;
        sb[0] += it.n_a;
        sb[1] += it.n_b;
      }
      if (!ok) {
        *abort = 1;
        record_status(d_status, KVS_ERR_TIMEOUT);
        // Every product issued finishes before the block frees the tensor
        // memory and exits.  A pending commit covers them all (nothing was
        // issued after it); otherwise commit once more.  At most one commit
        // is outstanding, so the parity wait is for that commit's phase.
        if (!pending && issued) {
          mma_commit(pvdone);
          pending = true;
        }
        if (pending) mbar_wait_drain(pvdone, pv_phase);
      }
    }
    __syncwarp();
  } else if (warp >= kPPackWarp0) {
    // ======================= packing =========================================
    // Each pack warp takes tiles from the task list (one atomicAdd per tile,
    // fetched a tile ahead) and moves a tile as 8 chunks of 16 rows: lane 0
    // bulk-copies the FP32 rows into a staging buffer (rows padded by 16
    // bytes), the warp rounds them to FP16 and stores 16-byte pieces in the
    // tensor-core layout, then publishes the tile's flag.  Two buffers: the
    // next chunk is in flight while this one converts.
    const int pw = warp - kPPackWarp0;
    float *stg = reinterpret_cast<float *>(smem + PG::OFF_STG + pw * 2 * PG::STG_BUF);
    uint64_t *sbar = stgfull + 2 * pw;
    unsigned *counter = flags + 3 * (size_t)H * T;
    const unsigned NT = (unsigned)nt_in;
    constexpr int kChunks = kPM / kPStgRows;
    constexpr int kBufFloats = PG::STG_BUF / 4;
    // Task numbers count up from zero (the counter is zeroed before every
    // launch that has tasks; with none, the counter is not touched), and
    // compare unsigned, so every warp's walk ends.
    unsigned tl = 0;  // lane 0: the next task number, fetched ahead
    auto fetch = [&]() {
      if (lane == 0) tl = atomicAdd(counter, 1u);
    };
    auto take = [&]() { return __shfl_sync(0xffffffffu, tl, 0); };
    // chunk c of tile p into buffer bb (rows past S are not copied)
    auto issue = [&](const PTile &p, int c, uint32_t bb) {
      if (lane == 0) {
        const int row0 = p.t * kPM + c * kPStgRows;
        const int nvalid = max(0, min(kPStgRows, S - row0));
        const float *src = (p.tensor == 0 ? q : p.tensor == 1 ? k : v) +
                           ((size_t)p.h * S + row0) * D;
        mbar_arrive_expect_tx(&sbar[bb], (uint32_t)nvalid * D * 4);
        for (int r = 0; r < nvalid; ++r)
          bulk_g2s(stg + bb * kBufFloats + r * PG::STG_STRIDE, src + (size_t)r * D, D * 4,
                   &sbar[bb]);
      }
    };
    bool ok = true;
    uint32_t issued = 0, done = 0;  // chunks issued and converted by this warp
    unsigned task = NT;
    if (NT > 0) {
      fetch();
      task = take();
    }
    PTile cur{0, 0, 0}, nxt{0, 0, 0};
    if (task < NT) {
      cur = prefill_task((int)task, H, T, causal, rq, s0);
      issue(cur, 0, 0);
      issued = 1;
      fetch();
    }
    int c = 0;
    while (task < NT) {
      // the next chunk goes into the other buffer, converted a chunk ago
      unsigned ntask = NT;
      if (c + 1 < kChunks) {
        issue(cur, c + 1, issued & 1u);
        ++issued;
      } else {
        ntask = take();
        if (ntask < NT) {
          nxt = prefill_task((int)ntask, H, T, causal, rq, s0);
          issue(nxt, 0, issued & 1u);
          ++issued;
        }
      }
      const uint32_t bb = done & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait<kPoll>(&sbar[bb], (done >> 1) & 1u, abort))) {
        ok = false;
        break;
      }
      const float *sb = stg + bb * kBufFloats;
      const int nvalid = max(0, min(kPStgRows, S - (cur.t * kPM + c * kPStgRows)));
      unsigned char *dst = tiles + (((size_t)cur.tensor * H + cur.h) * T + cur.t) * PG::TILE;
      if (cur.tensor < 2) {
        // Q, K: lane (rr, cg) converts row 8 * half + rr, 8 columns from
        // 8 * (cg + 4 * cc); eight lanes fill one 128-byte core matrix
        const int rr = lane & 7, cg = lane >> 3;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int lr = 8 * half + rr;
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            const int col = 8 * (cg + 4 * cc);
            float x[8];
            if (lr < nvalid) {
              const float4 a = *reinterpret_cast<const float4 *>(sb + lr * PG::STG_STRIDE + col);
              const float4 e = *reinterpret_cast<const float4 *>(sb + lr * PG::STG_STRIDE + col + 4);
              x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
              x[4] = e.x; x[5] = e.y; x[6] = e.z; x[7] = e.w;
            } else {
#pragma unroll
              for (int u = 0; u < 8; ++u) x[u] = 0.f;
            }
            *reinterpret_cast<uint4 *>(dst + cm_off(c * kPStgRows + lr, col, D)) = pack8(x);
          }
        }
      } else {
        // V^T: lane converts column d = lane + 32 j of v over keys 8g..8g+7
        // of the chunk into one 16-byte piece of V^T row d
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {
          const int d = lane + 32 * j;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              x[u] = (8 * g + u < nvalid) ? sb[(8 * g + u) * PG::STG_STRIDE + d] : 0.f;
            *reinterpret_cast<uint4 *>(dst + cm_off(d, c * kPStgRows + 8 * g, kPN)) = pack8(x);
          }
        }
      }
      ++done;
      __syncwarp();
      if (lane == 0) fence_proxy_async_shared();  // a bulk copy refills the buffer next
      if (c + 1 == kChunks) {
        // the tile is complete: every lane's stores are visible at GPU
        // scope before the flag says so
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async_global();
          st_release_u32(flags + ((size_t)cur.tensor * H + cur.h) * T + cur.t, 1u);
        }
        task = ntask;
        cur = nxt;
        c = 0;
        if (task < NT) fetch();
      } else {
        ++c;
      }
    }
    if (!ok) {
      *abort = 1;
      record_status(d_status, KVS_ERR_TIMEOUT);
    }
    // staged copies still in flight land before the block exits
    if (lane == 0)
      for (uint32_t j = done; j < issued; ++j) mbar_wait_drain(&sbar[j & 1u], (j >> 1) & 1u);
    __syncwarp();
  } else {
    // ======================= softmax of tile x ===============================
    const int x = warp >> 2;             // warpgroup
    const int t = threadIdx.x & 127;     // row within the tile
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tm_s = tmem + lane_base + x * kPN;
    const uint32_t tm_o = tmem + lane_base + 2 * kPN + x * D;
    int sb = 0;  // S_x products of the earlier items
    int ob = 0;  // earlier items with a tile x (odone[x] phases)
    for (int rd = 0; !failed; ++rd) {
      const int idx = prefill_item_index(b, rd, P);
      if (idx >= NI) break;
      const PItem it = prefill_item(idx, H, T, causal);
      const int q_tile = it.qa + x;
      const int i = q_tile * kPM + t;      // query row
      const int n_x = x == 0 ? it.n_a : it.n_b;
      float m = neg_inf_f();
      float l = 0.f;  // the row's sum of 2^(s - m)
      for (int kt = 0; kt < n_x; ++kt) {
        const int key0 = kt * kPN;
        const uint32_t ph = (uint32_t)(sb + kt) & 1u;
        // S_x(kt) is ready; it was issued after P V_x(kt-1) completed, so O_x
        // is quiescent too
        // all lanes of the warp leave together: the TMEM loads and stores
        // below are .sync.aligned (the whole warp executes them)
        if (!__all_sync(0xffffffffu, mbar_wait<kPoll>(&sfull[x], ph, abort))) {
          failed = true;
          break;
        }
        tc_fence_after();
        // keys needing a mask: past S, or past the row on the diagonal tile
        const bool masked = (key0 + kPN > S) || (causal && kt == q_tile);
        // ---- one pass over the scores, in two chunks of 64 keys ----
        // The reference maximum m_ref only moves when a chunk's maximum exceeds
        // it by more than kRescaleLog2 (log2 units): below that, p = 2^(s - m_ref)
        // stays under 2^kRescaleLog2 (FP16 holds it), the result is the same,
        // and nothing needs rescaling.  P of chunk c (FP16, two keys per
        // column) goes to columns [32c, 32c + 32), whose scores were read with
        // chunk 0.  When chunk 1 moves m_ref, chunk 0's P (already in TMEM) is
        // scaled by the power of two 2^(old - new): exact in FP16 down to the
        // subnormals, where it rounds like a direct evaluation would.
        // (Every row attends a key in chunk 0: key0 <= row on the diagonal
        // tile, and key0 < S.)
        float m_ref = m;
        float lt = 0.f;
#pragma unroll 1
        for (int ch = 0; ch < kPN / 64; ++ch) {
          float r[64];
          tmem_ld64(tm_s + ch * 64, r);
          tmem_wait_ld();
          if (masked) {
            mask_keys(*reinterpret_cast<float(*)[32]>(&r[0]), key0 + ch * 64, S, causal, i);
            mask_keys(*reinterpret_cast<float(*)[32]>(&r[32]), key0 + ch * 64 + 32, S, causal, i);
          }
          // chunk maximum as a tree (max is exact in any order; a chain of 64
          // dependent fmaxf would sit on the tile's critical path)
          float mx[32];
#pragma unroll
          for (int u = 0; u < 32; ++u) mx[u] = fmaxf(r[u], r[u + 32]);
#pragma unroll
          for (int w2 = 16; w2 >= 1; w2 >>= 1) {
#pragma unroll
            for (int u = 0; u < w2; ++u) mx[u] = fmaxf(mx[u], mx[u + w2]);
          }
          float cm = mx[0] * sl2;
          const float m_prev = m_ref;
          if (cm > m_ref + kRescaleLog2) m_ref = cm;
          if (ch > 0 && __any_sync(0xffffffffu, m_ref != m_prev)) {  // rare
            const float f = (m_ref != m_prev) ? ex2(m_prev - m_ref) : 1.f;
            lt *= f;
            const __half2 f2 = __float2half2_rn(f);
            uint32_t w0[32];
            tmem_wait_st();  // chunk 0's P has landed
            tmem_ld32u(tm_s, w0);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) {
              const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&w0[u]), f2);
              w0[u] = *reinterpret_cast<const uint32_t *>(&v);
            }
            tmem_st32u(tm_s, w0);
          }
          const float mb = (m_ref == neg_inf_f()) ? 0.f : m_ref;
          uint32_t w[32];
          // Two keys per paired FP32 instruction for the scaling and the sum
          // (each key rounds as it would alone): the softmax is bound by
          // instruction issue, not by the exponentials.  The sum runs in two
          // independent pairs (one dependent chain would sit on the critical
          // path).
          float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
          const float2 sl2x2 = make_float2(sl2, sl2), nmb2 = make_float2(-mb, -mb);
#pragma unroll
          for (int u = 0; u < 32; ++u) {
            const float2 x2 = __ffma2_rn(make_float2(r[2 * u], r[2 * u + 1]), sl2x2, nmb2);
            const float p0 = ex2(x2.x), p1 = ex2(x2.y);
            const __half2 hp = __floats2half2_rn(p0, p1);
            ls[u & 1] = __fadd2_rn(ls[u & 1], make_float2(p0, p1));
            w[u] = *reinterpret_cast<const uint32_t *>(&hp);
          }
          lt += (ls[0].x + ls[1].x) + (ls[0].y + ls[1].y);
          tmem_st32u(tm_s + ch * 32, w);
        }
        const float m_new = m_ref;
        const float alpha = (m == neg_inf_f()) ? 1.f : ex2(m - m_new);
        // ---- rescale the output accumulator (TMEM) where the maximum moved ----
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float r[32];
            tmem_ld32(tm_o + c * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int u = 0; u < 32; ++u) r[u] *= alpha;
            tmem_st32(tm_o + c * 32, r);
          }
        }
        l = l * alpha + lt;
        m = m_new;
        tmem_wait_st();  // P and the rescaled O are in TMEM before P V reads them
        tc_fence_before();
        mbar_arrive(&pfull[x]);
      }
      if (failed) break;
      sb += n_x;
      if (n_x == 0) continue;
      // the tile's last P V product is done: O_x is final.  Its rows go out
      // while the tensor cores already work on the next item's S products.
      if (!__all_sync(0xffffffffu, mbar_wait<kPoll>(&odone[x], (uint32_t)ob & 1u, abort))) {
        failed = true;
        break;
      }
      ++ob;
      tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll 1
      for (int ch = 0; ch < D / 32; ++ch) {
        float o[32];
        tmem_ld32(tm_o + ch * 32, o);
        tmem_wait_ld();
        if (i < S) {
          float4 *o4 = reinterpret_cast<float4 *>(out + ((size_t)it.h * S + i) * D + ch * 32);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            o4[u] = make_float4(o[4 * u] * inv, o[4 * u + 1] * inv, o[4 * u + 2] * inv,
                                o[4 * u + 3] * inv);
        }
      }
    }
    if (failed) {
      *abort = 1;
      record_status(d_status, KVS_ERR_TIMEOUT);
    }
  }
  allow_dependent_launch();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kPTmemCols);
}

template <int D>
int launch_prefill_impl(const float *q, const float *k, const float *v, float *out, int H, int S,
                        int causal, void *workspace, int *d_status, cudaStream_t stream) {
  using PG = PGeo<D>;
  static bool configured[64] = {false};
  static int num_sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KVS_ERR_LAUNCH;
  if (!configured[dev]) {
    if (cudaDeviceGetAttribute(&num_sms[dev], cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        num_sms[dev] < 1) {
      cudaGetLastError();
      return KVS_ERR_LAUNCH;
    }
    for (auto kern : {prefill_tc_kernel<D, false>, prefill_tc_kernel<D, true>}) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PG::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return KVS_ERR_LAUNCH;
      }
    }
    configured[dev] = true;
  }
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  const float sl2 = (float)(1.4426950408889634074 / std::sqrt((double)D));
  const int T = (S + kPM - 1) / kPM;
  // tile and task numbers are 32-bit (far beyond any workspace a GPU holds)
  if (3LL * H * T > (1LL << 30)) return KVS_ERR_UNSUPPORTED;
  // one block per SM (the shared memory and the 512 TMEM columns allow no
  // second), each walking its share of the items; more blocks than SMs
  // would only run one after another
  const long long items = (long long)H * ((T + 1) / 2);
  const int grid = (int)std::min<long long>(items, num_sms[dev]);
  // packed before the attention starts: the Q tiles of the first round's
  // pairs and the first s0 key tiles of K and V^T
  const int np = (T + 1) / 2;
  // key tiles left to the pack warps: 40 % of them, fewer when one key
  // tile of every head (K and V^T) is more than 4 MiB of FP32, so that the
  // pack warps (about 1.5 TB/s beside the attention) stay ahead of the
  // items; none below 16 key tiles, where the in-kernel packing only adds
  // latency.  Measured on GB300 (H=32, S=4096, D=128, causal), key tiles
  // packed upfront: 55 % 172.9 us, 60 % 167.6, 65 % 168.2, 70 % 169.8,
  // 100 % 179.7, 0 % 211.8; with no in-kernel share, 64 and 128 heads at
  // S=1024 ran 20 % faster than with 40 %.
  const double step_bytes = 2.0 * H * kPM * D * 4;
  const int n_in =
      T < 16 ? 0 : (int)(0.4 * T * std::min(1.0, (double)(4 << 20) / step_bytes));
  const int s0 = T - n_in;
  // the Q tiles of the first round's pairs; all of them when the pack warps
  // get no key tiles (then the later rounds' Q tiles would come too late)
  const int rq = n_in > 0 ? std::min(np, (grid + H - 1) / H) : np;
  int nq_up = 0;
  for (int pr = 0; pr < rq; ++pr) {
    const int qa = 2 * (causal ? np - 1 - pr : pr);
    nq_up += qa + 1 < T ? 2 : 1;
  }
  const int nt_in = 3 * H * T - H * nq_up - 2 * H * s0;
  // the tile flags and the task counter start at zero in every call that
  // packs in the attention kernel (otherwise no flag is read)
  if (nt_in > 0 && cudaMemsetAsync(ws, 0, prefill_flag_bytes(H, T), stream) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  if (rq + s0 > 0) {
    if (launch_pdl(prefill_pack_kernel<D>, dim3((2 * rq + 2 * s0) * (D / 16), H), dim3(256), 0, stream,
                   q, k, v, ws, H, S, causal, rq) != cudaSuccess)
      return KVS_ERR_LAUNCH;
  }
  const cudaError_t e =
      launch_pdl(poll_waits() ? prefill_tc_kernel<D, true> : prefill_tc_kernel<D, false>,
                 dim3(grid), dim3(kPBlockThreads), PG::SMEM_BYTES, stream, q, k, v, ws, out, H,
                 S, causal, sl2, d_status, rq, s0, nt_in);
  return e == cudaSuccess ? KVS_OK : KVS_ERR_LAUNCH;
}

}  // namespace

int set_wait_limit_prefill(uint64_t ns) {
  if (set_unit_wait_limit(ns) != cudaSuccess) {
    cudaGetLastError();
    return KVS_ERR_LAUNCH;
  }
  return KVS_OK;
}

size_t prefill_workspace_bytes(int H, int S, int D) {
  const size_t T = ((size_t)S + kPM - 1) / kPM;
  return prefill_flag_bytes((int)H, (int)T) + 3 * (size_t)H * T * prefill_tile_bytes(D);
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
