// Prefill kernels of libmoe (sm_103a): T tokens through one layer at once.
//
// "Optimizing a 14.3 GB model for an 8 GB machine", section "Splitting the work
// improved attention and prefill": batched prefill dequantises a small 16-bit
// tile of the affine int4 weights, runs the hardware matrix primitive on it and
// throws the tile away, so the stored weights never change.  Here that
// primitive is tcgen05 (fifth-generation tensor cores, operands and
// accumulators in tensor memory), and the batch is grouped by expert first:
//
//   k_pf_prep          RMS norm (or copy) of every token: x in bf16 (router)
//                      and fp16 (matrix operand), |x|^2 and max|x_i| per token.
//   k_pf_row_stats     |w|^2 and max|w_i| of the router rows (once per layer).
//   k_pf_logits_approx every (token, expert) logit in fp32 with a rigorous
//                      error bound.
//   k_pf_route         per token: the experts the bound cannot rule out, their
//                      exact fixed-point logits (the same 2^-40 grid as the
//                      decode kernels), top-k (ties to the lower index) and
//                      softmax gates.
//   k_pf_count /       stable counting sort of the T*k (token, position) pairs
//   k_pf_scatter       by expert, and the list of work items per expert.
//   k_pf_gather        the pairs' x rows, in that order, as one fp16 matrix.
//   k_pf_gemm          grouped int4 x fp16 GEMM on tcgen05.  A CTA owns 128
//                      weight rows and 128 (or 32) token rows of one expert.
//                      Warp 0's lane 0 streams the int4 blocks (bulk copies)
//                      and the token rows (TMA tensor loads, 128-byte swizzle,
//                      into shared memory).  Eight dequantising warps turn
//                      each 64-wide k step of the int4 blocks into fp16 and
//                      store it straight into tensor memory (the A operand).
//                      Warp 1 allocates tensor memory and one of its threads
//                      issues the MMAs (A from tensor memory, B from shared
//                      memory) into a fp32 accumulator in tensor memory; the
//                      eight warps then read it back for the epilogue:
//                      GELU(gate) * up (gate/up pass), the expert output per
//                      pair (routed down pass), or the shared expert's output
//                      per token (shared down pass).
//   k_pf_combine       per token: the shared output plus the gate-weighted
//                      routed outputs in top-k order, and the residual.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "kernels.h"

namespace moe {

namespace {

constexpr int kM = 128;                 // weight rows per CTA tile
// Token rows per CTA tile: 256 when the groups are large (each dequantised
// weight tile then serves twice the tokens of a 128-row tile; one CTA per SM),
// 128 for mid-sized groups, 32 when every expert has only a few rows.
template <int N>
struct Tile {
  static constexpr int kSlots = 4;                     // k-step slots (A in tensor memory, B in shared)
  static constexpr int kBBytes = N * 128;              // one N-row x 64-col fp16 tile
  static constexpr int kRawStages = N == 32 ? 4 : 2;   // int4 stages (more when the tokens are few)
  static constexpr int kTmemCols = N == 256 ? 512 : 256;   // accumulator (N) + four 32-column A slots
};
constexpr int kRawG = 4;                // int4 groups per raw stage
constexpr int kRawStride = kRawG * kGroupBytes;   // bytes of one 16-row tile in a raw stage
constexpr int kRawBytes = 8 * kRawStride;         // 8 tiles of 16 rows = 128 rows
constexpr int kDqWarps = 8;             // dequant + epilogue warps, one 16-row tile each per k step
constexpr int kThreads = 32 * (2 + kDqWarps);  // warp 0 producer, warp 1 MMA + TMEM, warps 2..9 dequant + epilogue

template <int N>
struct GemmSmem {
  static constexpr int kSlots = Tile<N>::kSlots;
  static constexpr int kRawStages = Tile<N>::kRawStages;
  uint8_t b[kSlots][Tile<N>::kBBytes];  // fp16 token tiles, K-major, 128-byte swizzle (1024-aligned, TMA)
  uint8_t raw[kRawStages][kRawBytes];   // int4 blocks as stored
  uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  uint64_t b_full[kSlots], a_full[kSlots], slot_empty[kSlots];
  uint64_t acc_full;
  uint32_t tmem_base;
  int abort;
  int row_info[N];                      // epilogue: pair index (routed down) of each token row
};
static_assert(offsetof(GemmSmem<128>, b) % 1024 == 0 && offsetof(GemmSmem<32>, b) % 1024 == 0 &&
                  offsetof(GemmSmem<256>, b) % 1024 == 0 && Tile<32>::kBBytes % 1024 == 0,
              "swizzled tiles need 1 KB alignment");
static_assert(offsetof(GemmSmem<128>, raw) % 128 == 0 && offsetof(GemmSmem<32>, raw) % 128 == 0 &&
                  offsetof(GemmSmem<256>, raw) % 128 == 0 &&
                  kRawStride % 16 == 0,
              "bulk copy targets need 16 B");
static_assert(offsetof(GemmSmem<128>, raw_full) % 8 == 0 && offsetof(GemmSmem<32>, raw_full) % 8 == 0 &&
                  offsetof(GemmSmem<256>, raw_full) % 8 == 0,
              "mbarriers need 8 B");
static_assert(sizeof(GemmSmem<256>) + 1024 <= 227 * 1024, "256-row token tiles fit one CTA per SM");

// ------------------------------------------------------------------ tcgen05 / TMA primitives

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major tile whose rows are 128 bytes, with
// the 128-byte swizzle; 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu)   // start address
         | (static_cast<uint64_t>(1) << 16)              // leading byte offset (unused with this swizzle)
         | (static_cast<uint64_t>(1024 >> 4) << 32)      // stride byte offset: 8 rows x 128 B
         | (static_cast<uint64_t>(1) << 46)              // descriptor version
         | (static_cast<uint64_t>(2) << 61);             // 128-byte swizzle
}

// Instruction descriptor: fp16 A and B (both K-major), fp32 accumulator, M x N.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// D (tensor memory) += A (tensor memory) x B (shared-memory descriptor).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, int acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// 32 consecutive fp32 accumulator columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float gelu_f(float v, int variant) {
  if (variant == 1) return 0.5f * v * (1.f + tanhf(0.7978845608028654f * (v + 0.044715f * v * v * v)));
  return 0.5f * v * (1.f + erff(v * 0.7071067811865476f));
}

// Event time k of CTA (0, 0) when a timeline is attached (diagnostics).
__device__ __forceinline__ void pf_stamp(const PfGemm& p, int k) {
  if (p.tl && blockIdx.x == 0 && blockIdx.y == 0) {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    p.tl[k] = t;
  }
}

template <class Sm>
__device__ __forceinline__ bool wait_or_abort(Sm& S, uint64_t* bar, uint32_t parity, uint32_t* err) {
  if (mbar_wait_bounded(bar, parity, err)) return true;
  S.abort = 1;
  return false;
}

// ------------------------------------------------------------------ dequantisation

// Column order of the 16-bit operands inside every 16-wide k block.  The
// tensor-memory store shape .16x256b gives lane (g, t4) of a warp the 32-bit
// columns 2 t4 and 2 t4 + 1 of rows g and g + 8; the stored int4 fragments give
// the same lane the k pairs {2 t4, 2 t4 + 1} and {2 t4 + 8, 2 t4 + 9}.  So the A
// operand in tensor memory holds k in the order pi(k) below, and every B operand
// (activations, GELU products) is written in the same order; the products pair
// up unchanged.
__host__ __device__ __forceinline__ int k16_pos(int i) {
  const int k = i & 15;
  return (i & ~15) | (4 * ((k & 7) >> 1) + (k & 1) + 2 * (k >> 3));
}

// One 16-row tile x 64-column group of int4 weights (a block as stored: lane
// fragments + per-row fp16 scale/bias) to fp16 w = s*q + b, stored into
// tensor-memory lanes lane0 .. lane0 + 15 and 32 columns from col (the A operand
// of four k16 MMAs), with one .16x256b store.  The caller's warp must own
// those lanes (warp % 4 == lane0 / 32).  Per nibble pair: the nibbles as fp16
// 1024 + q (OR under the exponent of 1024), minus 1024 (exact q), then s*q + b
// (fp16 fma); lane (g, t4)'s word st of the fragment holds nibbles j (low
// half) and j + 4 (high half) for j = 0: row g, k 2t4..; 1: row g + 8, k 2t4..;
// 2: row g, k 2t4 + 8..; 3: row g + 8, k 2t4 + 8..; the store's registers of
// repetition st are (row g, col 2t4), (row g, col 2t4 + 1), (row g + 8, ...).
// One asm block, so the sixteen results go straight into the store's
// operand registers.
__device__ __forceinline__ void dequant_block_tmem(const uint8_t* blk, uint32_t taddr) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const uint4 q = *reinterpret_cast<const uint4*>(blk + lane * 16);
  const uint2 sb = *reinterpret_cast<const uint2*>(blk + kFragBytes + g * 8);
  const uint32_t s0 = (sb.x & 0xFFFFu) * 0x10001u, c0 = (sb.x >> 16) * 0x10001u;   // fp16 pairs (s, s), (b, b)
  const uint32_t s1 = (sb.y & 0xFFFFu) * 0x10001u, c1 = (sb.y >> 16) * 0x10001u;
  asm volatile(
      "{\n\t"
      ".reg .b32 t<16>, r<16>;\n\t"
      "lop3.b32 t0, %1, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t0, t0, %9;\n\t"
      "fma.rn.f16x2 r0, t0, %5, %6;\n\t"
      "shr.b32 t1, %1, 4;\n\t"
      "lop3.b32 t1, t1, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t1, t1, %9;\n\t"
      "fma.rn.f16x2 r2, t1, %7, %8;\n\t"
      "shr.b32 t2, %1, 8;\n\t"
      "lop3.b32 t2, t2, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t2, t2, %9;\n\t"
      "fma.rn.f16x2 r1, t2, %5, %6;\n\t"
      "shr.b32 t3, %1, 12;\n\t"
      "lop3.b32 t3, t3, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t3, t3, %9;\n\t"
      "fma.rn.f16x2 r3, t3, %7, %8;\n\t"
      "lop3.b32 t4, %2, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t4, t4, %9;\n\t"
      "fma.rn.f16x2 r4, t4, %5, %6;\n\t"
      "shr.b32 t5, %2, 4;\n\t"
      "lop3.b32 t5, t5, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t5, t5, %9;\n\t"
      "fma.rn.f16x2 r6, t5, %7, %8;\n\t"
      "shr.b32 t6, %2, 8;\n\t"
      "lop3.b32 t6, t6, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t6, t6, %9;\n\t"
      "fma.rn.f16x2 r5, t6, %5, %6;\n\t"
      "shr.b32 t7, %2, 12;\n\t"
      "lop3.b32 t7, t7, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t7, t7, %9;\n\t"
      "fma.rn.f16x2 r7, t7, %7, %8;\n\t"
      "lop3.b32 t8, %3, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t8, t8, %9;\n\t"
      "fma.rn.f16x2 r8, t8, %5, %6;\n\t"
      "shr.b32 t9, %3, 4;\n\t"
      "lop3.b32 t9, t9, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t9, t9, %9;\n\t"
      "fma.rn.f16x2 r10, t9, %7, %8;\n\t"
      "shr.b32 t10, %3, 8;\n\t"
      "lop3.b32 t10, t10, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t10, t10, %9;\n\t"
      "fma.rn.f16x2 r9, t10, %5, %6;\n\t"
      "shr.b32 t11, %3, 12;\n\t"
      "lop3.b32 t11, t11, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t11, t11, %9;\n\t"
      "fma.rn.f16x2 r11, t11, %7, %8;\n\t"
      "lop3.b32 t12, %4, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t12, t12, %9;\n\t"
      "fma.rn.f16x2 r12, t12, %5, %6;\n\t"
      "shr.b32 t13, %4, 4;\n\t"
      "lop3.b32 t13, t13, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t13, t13, %9;\n\t"
      "fma.rn.f16x2 r14, t13, %7, %8;\n\t"
      "shr.b32 t14, %4, 8;\n\t"
      "lop3.b32 t14, t14, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t14, t14, %9;\n\t"
      "fma.rn.f16x2 r13, t14, %5, %6;\n\t"
      "shr.b32 t15, %4, 12;\n\t"
      "lop3.b32 t15, t15, %10, %9, 0xEA;\n\t"
      "sub.f16x2 t15, t15, %9;\n\t"
      "fma.rn.f16x2 r15, t15, %7, %8;\n\t"
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {r0,r1,r2,r3,r4,r5,r6,r7,r8,r9,r10,r11,r12,r13,r14,r15};\n\t"
      "}"
      ::"r"(taddr), "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w), "r"(s0), "r"(c0), "r"(s1), "r"(c1), "r"(0x64006400u),
      "r"(0x000F000Fu)
      : "memory");
}

// ------------------------------------------------------------------ the GEMM

// Two CTAs share an SM, so one's epilogue overlaps the other's main loop.
template <int kN>
__global__ void __launch_bounds__(kThreads, 2) k_pf_gemm(const __grid_constant__ CUtensorMap tmap_b, PfGemm p) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  constexpr int kSlots = Tile<kN>::kSlots;
  constexpr int kRawStages = Tile<kN>::kRawStages;
  constexpr int kCols = Tile<kN>::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  GemmSmem<kN>& S = *reinterpret_cast<GemmSmem<kN>*>(smem_raw + pad);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x;
  const int item = blockIdx.y;
  const int n_items = p.n_items_dev ? *p.n_items_dev : p.n_items;
  if (item >= n_items) return;  // uniform over the CTA: nothing allocated yet
  if (threadIdx.x == 0) pf_stamp(p, 0);
  const int expert = p.items ? p.items[3 * item] : 0;
  const int row0 = p.items ? p.items[3 * item + 1] : item * kN;
  const int nrows = p.items ? p.items[3 * item + 2] : min(kN, p.rows_total - row0);
  const int nG = p.nG;
  const uint8_t* wbase = p.w + static_cast<long long>(expert) * p.w_stride +
                         static_cast<size_t>(8 * m_tile) * nG * kGroupBytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(&S.raw_full[i], 1);
      mbar_init(&S.raw_empty[i], kDqWarps);
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(&S.b_full[i], 1);
      mbar_init(&S.a_full[i], kDqWarps);
      mbar_init(&S.slot_empty[i], 1);
    }
    mbar_init(&S.acc_full, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {  // the whole warp allocates the accumulator and the A slots
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&S.tmem_base)),
                 "r"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp >= 2 && p.mode == PF_DN_ROUTED)
    for (int c = threadIdx.x - 64; c < kN; c += 32 * kDqWarps) S.row_info[c] = c < nrows ? p.pair_of_row[row0 + c] : 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  if (threadIdx.x == 0) pf_stamp(p, 1);

  if (warp == 0) {
    if (lane == 0) {
      // producer: the tile's weights go to L2 at once (HBM streams them at full rate while the
      // ring below is filled from L2), then raw int4 stages (every kRawG k steps) and one
      // token tile per k step
      for (int t = 0; t < 8; ++t)
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(wbase + static_cast<size_t>(t) * nG * kGroupBytes),
                     "r"(static_cast<uint32_t>(nG * kGroupBytes))
                     : "memory");
      uint32_t raw_issued = 0, b_issued = 0;
      for (int G = 0; G < nG && !S.abort; ++G) {
        if (G % kRawG == 0) {
          const int s = G / kRawG, rs = s % kRawStages;
          const int ng = min(kRawG, nG - G);
          if (!wait_or_abort(S, &S.raw_empty[rs], ((s / kRawStages) & 1) ^ 1, p.err)) break;
          const uint32_t bytes = static_cast<uint32_t>(8 * ng * kGroupBytes);
          fence_proxy_async_smem();
          mbar_arrive_expect_tx(&S.raw_full[rs], bytes);
          for (int t = 0; t < 8; ++t)
            bulk_g2s(S.raw[rs] + t * kRawStride, wbase + (static_cast<size_t>(t) * nG + G) * kGroupBytes,
                     static_cast<uint32_t>(ng * kGroupBytes), &S.raw_full[rs]);
          raw_issued = s + 1;
        }
        const int slot = G % kSlots;
        if (!wait_or_abort(S, &S.slot_empty[slot], ((G / kSlots) & 1) ^ 1, p.err)) break;
        mbar_arrive_expect_tx(&S.b_full[slot], Tile<kN>::kBBytes);
        tma_load_2d(S.b[slot], &tmap_b, 64 * G, row0, &S.b_full[slot]);
        b_issued = G + 1;
      }
      if (S.abort) {  // let the copies already issued land before the CTA leaves
        for (uint32_t s = raw_issued > kRawStages ? raw_issued - kRawStages : 0; s < raw_issued; ++s)
          mbar_wait_bounded(&S.raw_full[s % kRawStages], (s / kRawStages) & 1, p.err);
        for (uint32_t G = b_issued > kSlots ? b_issued - kSlots : 0; G < b_issued; ++G)
          mbar_wait_bounded(&S.b_full[G % kSlots], (G / kSlots) & 1, p.err);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = f16_idesc(kM, kN);
      for (int G = 0; G < nG; ++G) {
        const int slot = G % kSlots;
        const uint32_t par = (G / kSlots) & 1;
        if (!wait_or_abort(S, &S.a_full[slot], par, p.err)) break;
        if (G == 0) pf_stamp(p, 3);
        if (!wait_or_abort(S, &S.b_full[slot], par, p.err)) break;
        if (G == 0) pf_stamp(p, 4);
        if (G == p.nG - 1) pf_stamp(p, 5);
        tc_fence_after();
        const uint32_t a0 = tmem + kN + 32 * slot, b0 = smem_u32(S.b[slot]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)  // four k16 steps: 8 columns of A, +32 bytes inside B's swizzled rows
          tc_mma_ts(tmem, a0 + 8 * kk, sw128_desc(b0 + 32 * kk), idesc, (G | kk) != 0);
        tc_commit(&S.slot_empty[slot]);
      }
      tc_commit(&S.acc_full);  // fires once every MMA above has completed
    }
  } else {
    // dequant warps: warp w takes 16-row tile 2q + (w - 2) / 4 of each k step (q = w % 4: the
    // tensor-memory lanes 32q .. 32q + 31 its warp may access); in the epilogue it reads those
    // accumulator lanes and the column half (w - 2) / 4
    const int dw = warp - 2, q = warp & 3, b16 = 2 * q + (dw >> 2);
    // column range of this warp's epilogue: two halves of the kN columns, or all 32 for warps 2..5
    const int c_lo = kN >= 128 ? (dw >> 2) * (kN / 2) : 0;
    const int c_hi = kN >= 128 ? c_lo + kN / 2 : ((dw >> 2) == 0 ? 32 : 0);
    for (int G = 0; G < nG; ++G) {
      const int s = G / kRawG, rs = s % kRawStages, gi = G % kRawG;
      if (gi == 0 && !wait_or_abort(S, &S.raw_full[rs], (s / kRawStages) & 1, p.err)) break;
      if (G == 0 && threadIdx.x == 64) pf_stamp(p, 2);
      const int slot = G % kSlots;
      if (!wait_or_abort(S, &S.slot_empty[slot], ((G / kSlots) & 1) ^ 1, p.err)) break;
      dequant_block_tmem(S.raw[rs] + b16 * kRawStride + gi * kGroupBytes,
                         tmem + (static_cast<uint32_t>(16 * b16) << 16) + kN + 32 * slot);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbarrier_arrive(&S.a_full[slot]);
      if ((gi == kRawG - 1 || G == nG - 1) && lane == 0) mbarrier_arrive(&S.raw_empty[rs]);
    }
    // epilogue: this warp reads accumulator lanes 32q .. 32q + 31 (weight rows of the tile)
    if (threadIdx.x == 64) pf_stamp(p, 6);
    const bool ok = wait_or_abort(S, &S.acc_full, 0, p.err);
    if (threadIdx.x == 64) pf_stamp(p, 7);
    tc_fence_after();
    if (ok) {
      const int row_in_tile = 32 * q + lane;
      for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
        float v[32];
        tc_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + c0, v);
        if (p.mode == PF_GU) {
          // lanes 0-7 / 16-23 hold gate rows, lanes 8-15 / 24-31 the up rows of the same features
          const int feat = 8 * (8 * m_tile + 2 * q + (lane >> 4)) + (lane & 7);
          const bool gate_lane = (lane & 8) == 0;
          bool bad = false;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float up = __shfl_xor_sync(0xFFFFFFFFu, v[j], 8);
            const int c = c0 + j;
            if (gate_lane && c < nrows) {
              const float a = gelu_f(v[j], p.gelu) * up;
              if (!(fabsf(a) < 65504.f)) bad = true;
              p.out16[static_cast<size_t>(row0 + c) * p.f_out + k16_pos(feat)] = __half_as_ushort(__float2half_rn(a));
            }
          }
          if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(p.err, ERR_PF_RANGE);
        } else if (p.mode == PF_DN_ROUTED) {
          const int R = kM * m_tile + row_in_tile;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c = c0 + j;
            if (c < nrows) p.out32[static_cast<size_t>(S.row_info[c]) * p.d + R] = v[j];
          }
        } else {  // PF_DN_SHARED: the shared expert's output per token, fp32 [T][d]
          const int R = kM * m_tile + row_in_tile;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < nrows) p.out32[static_cast<size_t>(row0 + c0 + j) * p.d + R] = v[j];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) pf_stamp(p, 8);
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols) : "memory");
  }
}

// ------------------------------------------------------------------ token-side kernels

// A token's x row for the small-batch GEMVs (small_batch.cu): fp16 in their
// fragment order (for each 64-element group G and lane quarter t4, eight
// 32-bit words (k16 step st, half h) holding elements 64 G + 16 st + 8 h +
// 2 t4 + {0, 1}) and its per-group sums of the fp16 values (each the same
// warp-shuffle tree over the 32 element pairs); from the bf16 row x, by the
// eight warps of the CTA, a group per warp.
__device__ __forceinline__ void sg_token_row(const uint16_t* x, int d, uint16_t* xv, float* xg) {
  const uint32_t* src = reinterpret_cast<const uint32_t*>(x);
  uint32_t* dst = reinterpret_cast<uint32_t*>(xv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nG = d / 64;
  // lane holds elements 64 G + 2 lane, + 1: k16 step lane / 8, half (lane / 4) % 2, quarter lane % 4
  const int st = lane >> 3, h = (lane >> 2) & 1, t4 = lane & 3;
  for (int Gi = warp; Gi < nG; Gi += 8) {
    const uint32_t v = src[32 * Gi + lane];
    const __half a = __float2half_rn(bf16_bits_to_float(static_cast<uint16_t>(v & 0xFFFFu)));
    const __half b = __float2half_rn(bf16_bits_to_float(static_cast<uint16_t>(v >> 16)));
    dst[((Gi * 4 + t4) * 4 + st) * 2 + h] =
        static_cast<uint32_t>(__half_as_ushort(a)) | (static_cast<uint32_t>(__half_as_ushort(b)) << 16);
    float sum = __half2float(a) + __half2float(b);
#pragma unroll
    for (int m = 16; m; m >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, m);
    if (lane == 0) xg[Gi] = sum;
  }
}

// One CTA per token: x = RMSnorm(h) (or h) as bf16 and fp16; the sum of squares
// is taken in a fixed order.  fp16 overflow / underflow of x is flagged.
__global__ void __launch_bounds__(256) k_pf_prep(const uint16_t* h, int d, int prenorm, float eps, uint16_t* x_bf,
                                                 uint16_t* x16, uint16_t* dbg_x, float* xn2, float* xmax,
                                                 uint16_t* xv, float* xg, uint32_t* err) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  __shared__ float red[8], red2[8], redm[8];
  const int t = blockIdx.x;
  const uint16_t* hr = h + static_cast<size_t>(t) * d;
  float ss = 0.f;
  for (int i = threadIdx.x; i < d; i += 256) {
    const float a = bf16_bits_to_float(hr[i]);
    ss += a * a;
  }
#pragma unroll
  for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float r = 1.f;
  if (prenorm) {
    float tot = 0.f;
    for (int w = 0; w < 8; ++w) tot += red[w];
    r = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
  }
  bool bad = false;
  float s2 = 0.f, mx = 0.f;
  for (int i = threadIdx.x; i < d; i += 256) {
    const uint16_t hb = hr[i];
    const uint16_t xb = prenorm ? float_to_bf16_bits(bf16_bits_to_float(hb) * r) : hb;
    const float xf = bf16_bits_to_float(xb);
    s2 = fmaf(xf, xf, s2);
    mx = fmaxf(mx, fabsf(xf));   // NaN is dropped here but makes s2 NaN
    x_bf[static_cast<size_t>(t) * d + i] = xb;
    const __half xh = __float2half_rn(xf);   // exact unless |x| < 2^-14 (then off by < 2^-25)
    if (!(fabsf(xf) < 65504.f)) bad = true;
    x16[static_cast<size_t>(t) * d + k16_pos(i)] = __half_as_ushort(xh);   // operand order (k16_pos)
    if (dbg_x) dbg_x[static_cast<size_t>(t) * d + i] = xb;
  }
#pragma unroll
  for (int m = 16; m; m >>= 1) {
    s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, m);
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, m));
  }
  if ((threadIdx.x & 31) == 0) {
    red2[threadIdx.x >> 5] = s2;
    redm[threadIdx.x >> 5] = mx;
  }
  if (xv) {
    // small batches: the token's fp16 x row in the small-batch GEMVs' fragment
    // order, and its 64-element group sums, from the finished bf16 row
    __syncthreads();
    sg_token_row(x_bf + static_cast<size_t>(t) * d, d, xv + static_cast<size_t>(t) * d, xg + static_cast<size_t>(t) * (d / 64));
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(err, ERR_PF_RANGE);
  if (threadIdx.x == 0) {
    float a = 0.f, b = 0.f;
    for (int w = 0; w < 8; ++w) {
      a += red2[w];
      b = fmaxf(b, redm[w]);
    }
    xn2[t] = a;       // for the router's error bound
    xmax[t] = b;
  }
}

// |row|^2 and max |row_i| of fp16 rows (the router's rows, once per layer), one warp per row.
__global__ void __launch_bounds__(256) k_pf_row_stats(const uint16_t* rows, int n, int d, float* n2, float* mx) {
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= n) return;
  float ss = 0.f, m = 0.f;
  for (int i = lane; i < d; i += 32) {
    const float v = __half2float(__ushort_as_half(rows[static_cast<size_t>(r) * d + i]));
    ss = fmaf(v, v, ss);
    m = fmaxf(m, fabsf(v));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  }
  if (lane == 0) {
    n2[r] = ss;
    mx[r] = m;
  }
}

// Router, in two passes.
//
// Pass 1 (k_pf_logits_approx): every (token, expert) logit in fp32 with a
// rigorous error bound.  A CTA takes 32 tokens x 32 experts over one slice of
// d; each thread sums 2 x 2 logits with fused multiply-adds in 64-term chunks
// (the products are exact in fp32: 11-bit x 8-bit significands), so the sum
// differs from the exact one by at most about (64 + 2 * 44) u * sum|x_i w_i|
// with u = 2^-24 (chunk sums, slice sums and the adds across slices), and
// sum|x_i w_i| <= |x| |w| (Cauchy-Schwarz).  |x_t|^2 and max|x_t,i| come from
// k_pf_prep, |w_e|^2 and max|w_e,i| from k_pf_row_stats when the layer is loaded.
//
// Pass 2 (k_pf_route): one CTA per token.  With L~_e the approximate logit
// plus bias and eps_e its bound, tau = the k-th largest L~_e - eps_e is below
// the exact k-th largest logit, so an expert with L~_e + eps_e < tau cannot be
// selected.  An expert whose largest |x_i| |w_i| could leave the exact domain
// (|x_i w_i| < 2^11), or whose bound is not finite, is always a candidate, so
// the exact pass still flags such inputs.  The candidates (usually k or k + 1) get their exact
// fixed-point logits (products rounded onto the 2^-40 grid, summed exactly with
// Fix40), and the top-k (ties to the lower index) and the softmax gates are
// taken from those, so the result is the exact router's.
constexpr int kRE = 64;       // experts per CTA
constexpr int kApproxWavesBig = 3;   // grid target of the 128-token tiles, in SMs
constexpr int kRK = 64;       // k chunk (one partial sum per chunk)
// kTT tokens x 4 experts per thread, 16 kTT tokens x 64 experts per CTA: 4
// (64 tokens) for small batches, 8 (128 tokens: twice the multiply-adds per
// shared-memory read) for large ones, where shared-memory reads bound it.
template <int kTT>
__global__ void __launch_bounds__(256, kTT == 4 ? 4 : 2)
    k_pf_logits_approx(const uint16_t* x_bf, const uint16_t* router_w, int T, int d, int E, int k_slice,
                       float* approx) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  constexpr int kRT = 16 * kTT;                  // tokens per CTA
  __shared__ __align__(16) float xs[kRK][kRT];   // K-major, so a thread reads four tokens as one float4
  __shared__ __align__(16) float ws[kRK][kRE];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kRT, e0 = blockIdx.y * kRE, kb = blockIdx.z * k_slice;
  const int tx = tid & 15;             // experts e0 + 4 tx .. + 3
  const int ty = tid >> 4;             // tokens t0 + kTT ty .. + kTT - 1
  float acc[kTT][4];
#pragma unroll
  for (int a = 0; a < kTT; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;
  // staging: runs of eight columns, each thread's rows fixed over the chunks
  // (x: row tid % kRT; W_r: row tid % 64), so the 32 lanes of a warp store 32
  // consecutive rows of one column (no bank conflicts); several CTAs per SM
  // hide the loads (measured better than prefetching the next chunk into
  // registers)
  constexpr int kXR = kRT * kRK / 8 / 256;       // x runs per thread (2 or 4)
  const int rx = tid % kRT, cx = (tid / kRT) * 8, rw = tid & 63, cw = (tid >> 6) * 8;
  const bool tv = t0 + rx < T, ev = e0 + rw < E;
  uint4 xv[kXR], wv[2];
  auto load = [&](int k0) {
#pragma unroll
    for (int j = 0; j < kXR; ++j)
      xv[j] = tv ? *reinterpret_cast<const uint4*>(x_bf + static_cast<size_t>(t0 + rx) * d + k0 + cx + (64 / kXR) * j)
                 : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < 2; ++j)
      wv[j] = ev ? *reinterpret_cast<const uint4*>(router_w + static_cast<size_t>(e0 + rw) * d + k0 + cw + 32 * j)
                 : make_uint4(0u, 0u, 0u, 0u);
  };
  for (int k0 = kb; k0 < kb + k_slice; k0 += kRK) {
    load(k0);
    __syncthreads();   // the previous chunk's products are done
#pragma unroll
    for (int j = 0; j < kXR; ++j) {
      const uint32_t xa[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
      const int col = cx + (64 / kXR) * j;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        xs[col + 2 * u][rx] = bf16_bits_to_float(static_cast<uint16_t>(xa[u] & 0xFFFFu));
        xs[col + 2 * u + 1][rx] = bf16_bits_to_float(static_cast<uint16_t>(xa[u] >> 16));
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint32_t wa[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
      const int col = cw + 32 * j;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        ws[col + 2 * u][rw] = half_lo(wa[u]);
        ws[col + 2 * u + 1][rw] = half_hi(wa[u]);
      }
    }
    __syncthreads();
    float c[kTT][4];
#pragma unroll
    for (int a = 0; a < kTT; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) c[a][b] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < kRK; ++kk) {
      float xa[kTT];
#pragma unroll
      for (int q = 0; q < kTT / 4; ++q) {
        const float4 xf = *reinterpret_cast<const float4*>(&xs[kk][kTT * ty + 4 * q]);
        xa[4 * q] = xf.x;
        xa[4 * q + 1] = xf.y;
        xa[4 * q + 2] = xf.z;
        xa[4 * q + 3] = xf.w;
      }
      const float4 wf = *reinterpret_cast<const float4*>(&ws[kk][4 * tx]);
      const float wa[4] = {wf.x, wf.y, wf.z, wf.w};
#pragma unroll
      for (int a = 0; a < kTT; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) c[a][b] = fmaf(xa[a], wa[b], c[a][b]);
    }
#pragma unroll
    for (int a = 0; a < kTT; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) acc[a][b] += c[a][b];
  }
#pragma unroll
  for (int a = 0; a < kTT; ++a)
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int t = t0 + kTT * ty + a, e = e0 + 4 * tx + b;
      if (t < T && e < E) {
        float* dst = approx + static_cast<size_t>(t) * E + e;
        if (gridDim.z == 1) *dst = acc[a][b];
        else atomicAdd(dst, acc[a][b]);
      }
    }
}

// Eight products x_i w_i (bf16 x, fp16 w) onto the 2^-40 grid; a product
// outside |x_i w_i| < 2^11 is dropped and flagged.
constexpr int kRouteChunks = 12;   // 8-column chunks per lane: 256 * 12 = 3072 columns
__device__ __forceinline__ void exact_terms(const uint4& xv, const uint4& wv, Fix40& fx, bool& bad) {
  const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const float px = bf16_bits_to_float(static_cast<uint16_t>(hh ? (xa[u] >> 16) : (xa[u] & 0xFFFFu)));
      const float pw = hh ? half_hi(wa[u]) : half_lo(wa[u]);
      const float prod = pw * px;
      const bool ok = fabsf(prod) < 2048.f;
      bad |= !ok;
      fix40_add(fx, ok ? prod * 1099511627776.0f : 0.f);
    }
}

// Pass 2: candidates, their exact logits, top-k and gates.  A CTA takes tpc <= 8
// tokens (warp w < tpc takes the candidates and the top-k of token
// blockIdx.x * tpc + w); all eight warps share the exact dot products, so a
// small batch runs on one token per CTA and still spreads over the GPU.
template <int kHold>
__global__ void __launch_bounds__(256) k_pf_route(const uint16_t* x_bf, const uint16_t* router_w, float* approx,
                                                  const float* xn2, const float* wn2, const float* xmax,
                                                  const float* wmax, const float* bias, int T, int d,
                                                  int E, int k, int32_t* ids, float* gates, int32_t* dbg_ids,
                                                  float* dbg_gates, int64_t* dbg_logits, int tpc, uint32_t* err) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  __shared__ int cand_all[8][128];
  __shared__ long long exact_all[8][128];
  __shared__ int n_cand_all[8];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t = blockIdx.x * tpc + warp;
  const bool live = warp < tpc && t < T;         // warp-uniform
  int* cand = cand_all[warp];
  long long* exact = exact_all[warp];
  int& n_cand = n_cand_all[warp];
  if (lane == 0) n_cand = 0;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  if (live) {
    // candidates: L~_e + eps_e >= tau, tau = k-th largest of L~_e - eps_e
    const float u = 5.9604645e-8f;                                  // 2^-24
    const float xn = sqrtf(xn2[t]) * 1.01f;
    const float xm = xmax[t];
    float lo[4], hi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = lane + 32 * i;
      lo[i] = -INFINITY;
      hi[i] = -INFINITY;
      if (e < E) {
        const float s = approx[static_cast<size_t>(t) * E + e];
        approx[static_cast<size_t>(t) * E + e] = 0.f;   // zero again for the next accumulation
        const float b = bias ? bias[static_cast<size_t>(t) * E + e] : 0.f;
        const float L = s + b;
        const float eps = 160.f * u * xn * (sqrtf(wn2[e]) * 1.01f) + static_cast<float>(d + 1) * 4.5474735e-13f +
                          2.f * u * (fabsf(s) + fabsf(b)) + 1e-30f;
        lo[i] = L - eps * 1.01f;
        hi[i] = L + eps * 1.01f;
        if (!(xm * wmax[e] < 2048.f) || !(fabsf(lo[i]) < 3.0e38f) || !(fabsf(hi[i]) < 3.0e38f)) {
          lo[i] = -INFINITY;   // always a candidate: the exact pass decides (and flags the domain)
          hi[i] = INFINITY;
        }
        if (!(fabsf(b) < 1048576.f)) s_bad = 1;
      }
    }
    // tau: the k-th largest lower bound (repeated warp max, removing one entry each round)
    float tau = -INFINITY;
    {
      float v[4] = {lo[0], lo[1], lo[2], lo[3]};
      for (int j = 0; j < k; ++j) {
        float m = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
#pragma unroll
        for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        tau = m;
        // remove one occurrence of m: the lowest lane / slot that holds it
        int mine = -1;
#pragma unroll
        for (int i = 3; i >= 0; --i)
          if (v[i] == m) mine = i;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, mine >= 0);
        if (mine >= 0 && lane == __ffs(bal) - 1) v[mine] = -INFINITY;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = lane + 32 * i;
      const bool c = e < E && hi[i] >= tau;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, c);
      int base = 0;
      if (lane == 0) base = atomicAdd(&n_cand, __popc(bal));
      base = __shfl_sync(0xFFFFFFFFu, base, 0);
      if (c) cand[base + __popc(bal & ((1u << lane) - 1u))] = e;
    }
  }
  __syncthreads();
  // exact logits of every (token, candidate) of the CTA, one warp per pair
  int total = 0, first[9];
  for (int w = 0; w < 8; ++w) {
    first[w] = total;
    total += n_cand_all[w];
  }
  first[8] = total;
  bool bad = false;
  for (int pi = warp; pi < total; pi += 8) {
    int tw = 0;
    while (pi >= first[tw + 1]) ++tw;
    const int ci = pi - first[tw];
    const int tt = blockIdx.x * tpc + tw;
    const int e = cand_all[tw][ci];
    const uint16_t* xr = x_bf + static_cast<size_t>(tt) * d;
    const uint16_t* wr = router_w + static_cast<size_t>(e) * d;
    Fix40 fx;
    // eight products per lane per 256 columns (d <= 3072, checked when the
    // context is created: at most 96 terms); the loads of kHold chunks are
    // issued before their products, so with kHold = 12 a pair costs one
    // memory round trip (few tokens per launch: latency), with fewer the
    // kernel keeps more CTAs per SM (many tokens: throughput)
#pragma unroll
    for (int c0 = 0; c0 < kRouteChunks; c0 += kHold) {
      uint4 xv[kHold], wv[kHold];
#pragma unroll
      for (int c = 0; c < kHold; ++c)
        if (256 * (c0 + c) + 8 * lane < d) {
          xv[c] = *reinterpret_cast<const uint4*>(xr + 256 * (c0 + c) + 8 * lane);
          wv[c] = *reinterpret_cast<const uint4*>(wr + 256 * (c0 + c) + 8 * lane);
        }
#pragma unroll
      for (int c = 0; c < kHold; ++c)
        if (256 * (c0 + c) + 8 * lane < d) exact_terms(xv[c], wv[c], fx, bad);
    }
    long long v = fix40_value(fx);
#pragma unroll
    for (int m = 16; m; m >>= 1) v += shfl_xor_i64(v, m);
    if (lane == 0) {
      if (bias) {
        const float bv = bias[static_cast<size_t>(tt) * E + e];
        if (fabsf(bv) < 1048576.f) v += __float2ll_rn(bv * 1099511627776.0f);
      }
      exact_all[tw][ci] = v;
    }
  }
  if (__syncthreads_or(bad || s_bad) && tid == 0) atomicOr(err, ERR_ROUTER_DOMAIN);
  if (!live) return;
  if (dbg_logits) {
    // exact logits of the candidates; the experts the bound ruled out read LLONG_MIN
    int64_t* dl = dbg_logits + static_cast<size_t>(t) * E;
    for (int e = lane; e < E; e += 32) dl[e] = LLONG_MIN;
    __syncwarp();
    for (int ci = lane; ci < n_cand; ci += 32) dl[cand[ci]] = exact[ci];
  }
  // top-k over the candidates: a lane holds candidates lane, lane + 32, ...
  unsigned long long key[4];
  int idx[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ci = lane + 32 * i;
    key[i] = 0ull;
    idx[i] = 0x7fffffff;
    if (ci < n_cand) {
      key[i] = static_cast<unsigned long long>(exact[ci]) ^ 0x8000000000000000ull;
      idx[i] = cand[ci];
    }
  }
#pragma unroll
  for (int i = 1; i < 4; ++i)
#pragma unroll
    for (int j = i; j > 0; --j)
      if (key[j] > key[j - 1] || (key[j] == key[j - 1] && idx[j] < idx[j - 1])) {
        const unsigned long long tk = key[j];
        key[j] = key[j - 1];
        key[j - 1] = tk;
        const int ti = idx[j];
        idx[j] = idx[j - 1];
        idx[j - 1] = ti;
      }
  int head = 0, my_id = 0;
  long long my_v = 0;
  for (int j = 0; j < k; ++j) {
    unsigned long long hk = 0ull;
    int he = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i == head) {
        hk = key[i];
        he = idx[i];
      }
    const bool has = head < 4 && he != 0x7fffffff;
    const unsigned hi = has ? static_cast<unsigned>(hk >> 32) : 0u;
    const unsigned lo = has ? static_cast<unsigned>(hk) : 0u;
    const unsigned mh = __reduce_max_sync(0xFFFFFFFFu, hi);
    const bool c1 = has && hi == mh;
    const unsigned ml = __reduce_max_sync(0xFFFFFFFFu, c1 ? lo : 0u);
    const bool c2 = c1 && lo == ml;
    const unsigned me = __reduce_min_sync(0xFFFFFFFFu, c2 ? static_cast<unsigned>(he) : 0xFFFFFFFFu);
    if (c2 && static_cast<unsigned>(he) == me) ++head;
    if (lane == j) {
      my_id = static_cast<int>(me);
      my_v = static_cast<long long>((static_cast<unsigned long long>(mh) << 32 | ml) ^ 0x8000000000000000ull);
    }
  }
  const long long top = __shfl_sync(0xFFFFFFFFu, my_v, 0);
  float ex = 0.f;
  if (lane < k) ex = expf(__ll2float_rn(my_v - top) * 9.094947017729282e-13f);
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(0xFFFFFFFFu, ex, j);
  if (lane < k) {
    const size_t o = static_cast<size_t>(t) * k + lane;
    ids[o] = my_id;
    gates[o] = ex / sum;
    if (dbg_ids) dbg_ids[o] = my_id;
    if (dbg_gates) dbg_gates[o] = ex / sum;
  }
}

// Pairs per expert.  One CTA per expert scans every (token, position) pair.
__global__ void __launch_bounds__(256) k_pf_count(const int32_t* ids, int P, int32_t* cnt) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  const int e = blockIdx.x;
  int n = 0;
  for (int i = threadIdx.x; i < P; i += 256) n += ids[i] == e;
  __shared__ int red[8];
#pragma unroll
  for (int m = 16; m; m >>= 1) n += __shfl_xor_sync(0xFFFFFFFFu, n, m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int w = 0; w < 8; ++w) s += red[w];
    cnt[e] = s;
  }
}

// Stable placement: expert e's pairs in increasing pair order at
// [off_e, off_e + n_e), and its 128-row work items.
// With count_here (small P), every CTA first counts all pairs per expert in
// shared memory (and CTA e writes cnt[e]), so no counting launch precedes it.
__global__ void __launch_bounds__(256) k_pf_scatter(const int32_t* ids, int P, int E, int32_t* cnt, int tile,
                                                    int32_t* row_pair, int32_t* items, int32_t* n_items,
                                                    int count_here) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  const int e = blockIdx.x;
  __shared__ int s_off, s_base;
  __shared__ int wsum[8], wit[8];
  __shared__ int hist[256];
  if (count_here) {
    for (int i = threadIdx.x; i < E; i += 256) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < P; i += 256) atomicAdd(&hist[ids[i]], 1);
    __syncthreads();
    if (threadIdx.x == 0) cnt[e] = hist[e];
  }
  {
    // pairs and items of the experts before e (E <= 256: one per thread), summed over the CTA
    const int e2 = threadIdx.x;
    int c = e2 < e ? (count_here ? hist[e2] : cnt[e2]) : 0;
    int it2 = (c + tile - 1) / tile;
#pragma unroll
    for (int m = 16; m; m >>= 1) {
      c += __shfl_xor_sync(0xFFFFFFFFu, c, m);
      it2 += __shfl_xor_sync(0xFFFFFFFFu, it2, m);
    }
    if ((threadIdx.x & 31) == 0) {
      wsum[threadIdx.x >> 5] = c;
      wit[threadIdx.x >> 5] = it2;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    int off = 0, it = 0;
    for (int w = 0; w < 8; ++w) {
      off += wsum[w];
      it += wit[w];
    }
    s_off = off;
    s_base = 0;
    const int n_e = count_here ? hist[e] : cnt[e];
    for (int i = 0; i * tile < n_e; ++i) {
      items[3 * (it + i)] = e;
      items[3 * (it + i) + 1] = off + i * tile;
      items[3 * (it + i) + 2] = min(tile, n_e - i * tile);
    }
    if (e == E - 1) *n_items = it + (n_e + tile - 1) / tile;
  }
  __syncthreads();
  // 2048 pairs per pass, eight consecutive ones per thread, placed in pair
  // order; the next pass's ids are loaded before this pass's scan
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  auto load_ids = [&](int c0, int (&v)[8]) {
    const int i0 = c0 + 8 * threadIdx.x;
    if (i0 + 8 <= P) {   // ids is 256-byte aligned and i0 a multiple of 8
      const int4 a = *reinterpret_cast<const int4*>(ids + i0), b = *reinterpret_cast<const int4*>(ids + i0 + 4);
      v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = i0 + u < P ? ids[i0 + u] : -1;
    }
  };
  int cur[8];
  load_ids(0, cur);
  for (int c0 = 0; c0 < P; c0 += 2048) {
    const int i0 = c0 + 8 * threadIdx.x;
    int nxt[8] = {-1, -1, -1, -1, -1, -1, -1, -1};
    if (c0 + 2048 < P) load_ids(c0 + 2048, nxt);
    unsigned mask = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (cur[u] == e) mask |= 1u << u;
#pragma unroll
    for (int u = 0; u < 8; ++u) cur[u] = nxt[u];
    const int n = __popc(mask);
    int incl = n;   // inclusive scan over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    int before = incl - n, total = 0;
    for (int w2 = 0; w2 < 8; ++w2) {
      if (w2 < w) before += wsum[w2];
      total += wsum[w2];
    }
    int pos = s_off + s_base + before;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (mask & (1u << u)) row_pair[pos++] = i0 + u;
    __syncthreads();
    if (threadIdx.x == 0) s_base += total;
    __syncthreads();
  }
}

// y = shared + sum_j g_j * y_j in top-k order, h' = bf16(h + y): one CTA per
// token and block of 1024 output rows, four consecutive rows per thread
// (16-byte loads of the fp32 rows; d is a multiple of 64), each row's sum in
// the same order as one row per thread.
__global__ void __launch_bounds__(256) k_pf_combine(const float* ys, const float* ytok, const float* gates,
                                                    const uint16_t* hin, uint16_t* hout, float* y_last, float* dbg_y,
                                                    int d, int k) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  const int t = blockIdx.x;
  __shared__ float g[32];
  if (threadIdx.x < k) g[threadIdx.x] = gates[static_cast<size_t>(t) * k + threadIdx.x];
  __syncthreads();
  const float* yt = ytok + static_cast<size_t>(t) * k * d;
  const int R = (blockIdx.y * 256 + threadIdx.x) * 4;
  if (R >= d) return;
  const size_t o = static_cast<size_t>(t) * d + R;
  const float4 y0 = *reinterpret_cast<const float4*>(ys + o);
  float y[4] = {y0.x, y0.y, y0.z, y0.w};
  int j = 0;
  for (; j + 8 <= k; j += 8) {   // eight independent 16-byte loads in flight, summed in top-k order
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = __ldcs(reinterpret_cast<const float4*>(yt + static_cast<size_t>(j + u) * d + R));   // read once: stream
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      y[0] += g[j + u] * v[u].x;
      y[1] += g[j + u] * v[u].y;
      y[2] += g[j + u] * v[u].z;
      y[3] += g[j + u] * v[u].w;
    }
  }
  for (; j < k; ++j) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(yt + static_cast<size_t>(j) * d + R));
    y[0] += g[j] * v.x;
    y[1] += g[j] * v.y;
    y[2] += g[j] * v.z;
    y[3] += g[j] * v.w;
  }
  const uint2 hv = *reinterpret_cast<const uint2*>(hin + o);
  const uint16_t h4[4] = {static_cast<uint16_t>(hv.x & 0xFFFFu), static_cast<uint16_t>(hv.x >> 16),
                          static_cast<uint16_t>(hv.y & 0xFFFFu), static_cast<uint16_t>(hv.y >> 16)};
  uint16_t r4[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) r4[u] = float_to_bf16_bits(bf16_bits_to_float(h4[u]) + y[u]);
  *reinterpret_cast<uint2*>(hout + o) =
      make_uint2(r4[0] | (static_cast<uint32_t>(r4[1]) << 16), r4[2] | (static_cast<uint32_t>(r4[3]) << 16));
  const float4 yv = make_float4(y[0], y[1], y[2], y[3]);
  if (y_last) *reinterpret_cast<float4*>(y_last + o) = yv;
  if (dbg_y) *reinterpret_cast<float4*>(dbg_y + o) = yv;
}

// The same, one row per thread: for small batches (more CTAs) and for caller
// buffers that are not aligned for the vector form (h_in / h_out to 8 bytes,
// y to 16).
__global__ void __launch_bounds__(256) k_pf_combine1(const float* ys, const float* ytok, const float* gates,
                                                     const uint16_t* hin, uint16_t* hout, float* y_last, float* dbg_y,
                                                     int d, int k) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  const int t = blockIdx.x;
  __shared__ float g[32];
  if (threadIdx.x < k) g[threadIdx.x] = gates[static_cast<size_t>(t) * k + threadIdx.x];
  __syncthreads();
  const float* yt = ytok + static_cast<size_t>(t) * k * d;
  const int R = blockIdx.y * 256 + threadIdx.x;
  if (R >= d) return;
  const size_t o = static_cast<size_t>(t) * d + R;
  float y = ys[o];
  int j = 0;
  for (; j + 8 <= k; j += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcs(yt + static_cast<size_t>(j + u) * d + R);
#pragma unroll
    for (int u = 0; u < 8; ++u) y += g[j + u] * v[u];
  }
  for (; j < k; ++j) y += g[j] * __ldcs(yt + static_cast<size_t>(j) * d + R);
  hout[o] = float_to_bf16_bits(bf16_bits_to_float(hin[o]) + y);
  if (y_last) y_last[o] = y;
  if (dbg_y) dbg_y[o] = y;
}

// Row r of the expert-ordered matrix = fp16 x of the pair's token.
__global__ void __launch_bounds__(256) k_pf_gather(const uint16_t* x16, const int32_t* row_pair, int P, int d, int k,
                                                   uint16_t* xp) {
  pdl_wait();      // the previous kernel of the stream is complete (no-op without programmatic launch)
  pdl_trigger();
  // one warp per row, eight rows per CTA; a lane's loads (up to 12 of 16
  // bytes for d <= 3072) are all issued before its stores
  const int r = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (r >= P) return;
  const int t = row_pair[r] / k;
  const uint4* src = reinterpret_cast<const uint4*>(x16 + static_cast<size_t>(t) * d);
  uint4* dst = reinterpret_cast<uint4*>(xp + static_cast<size_t>(r) * d);
  const int n = d / 8;
  uint4 v[12];
#pragma unroll
  for (int u = 0; u < 12; ++u)
    if (lane + 32 * u < n) v[u] = src[lane + 32 * u];
#pragma unroll
  for (int u = 0; u < 12; ++u)
    if (lane + 32 * u < n) dst[lane + 32 * u] = v[u];
}

}  // namespace

size_t pf_gemm_smem(int n) {
  return (n == 32 ? sizeof(GemmSmem<32>) : n == 256 ? sizeof(GemmSmem<256>) : sizeof(GemmSmem<128>)) + 1024;
}

cudaError_t pf_set_attrs() {
  cudaError_t e = cudaFuncSetAttribute((const void*)k_pf_gemm<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(pf_gemm_smem(128)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute((const void*)k_pf_gemm<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(pf_gemm_smem(256)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute((const void*)k_pf_gemm<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(pf_gemm_smem(32)));
}

cudaError_t launch_pf_gemm(int n, const CUtensorMap& tmap_b, const PfGemm& p, int m_tiles, int max_items,
                           cudaStream_t s) {
  if (m_tiles <= 0 || max_items <= 0) return cudaSuccess;
  if (n == 32) return launch_chain(k_pf_gemm<32>, dim3(m_tiles, max_items), dim3(kThreads), pf_gemm_smem(32), s, tmap_b, p);
  if (n == 256)
    return launch_chain(k_pf_gemm<256>, dim3(m_tiles, max_items), dim3(kThreads), pf_gemm_smem(256), s, tmap_b, p);
  return launch_chain(k_pf_gemm<128>, dim3(m_tiles, max_items), dim3(kThreads), pf_gemm_smem(128), s, tmap_b, p);
}

cudaError_t launch_pf_prep(const uint16_t* h, int T, int d, int prenorm, float eps, uint16_t* x_bf, uint16_t* x16,
                           uint16_t* dbg_x, float* xn2, float* xmax, uint16_t* xv, float* xg, uint32_t* err,
                           cudaStream_t s) {
  return launch_chain(k_pf_prep, dim3(T), dim3(256), 0, s, h, d, prenorm, eps, x_bf, x16, dbg_x, xn2, xmax, xv, xg,
                      err);
}

cudaError_t launch_pf_row_stats(const uint16_t* rows, int n, int d, float* n2, float* mx, cudaStream_t s) {
  k_pf_row_stats<<<(n + 7) / 8, 256, 0, s>>>(rows, n, d, n2, mx);
  return cudaGetLastError();
}

cudaError_t launch_pf_router(const uint16_t* x_bf, const uint16_t* router_w, const float* bias, int T, int d, int E,
                             int k, float* approx, float* xn2, float* wn2, float* xmax, float* wmax, int32_t* ids,
                             float* gates, int32_t* dbg_ids, float* dbg_gates, int64_t* dbg_logits, uint32_t* err, int n_sm,
                             cudaStream_t s) {
  // 128-token tiles from 256 tokens on (kTT = 8), else 64
  const bool big = T >= 256;
  const int rt = big ? 128 : 64;
  const int tiles = ((T + rt - 1) / rt) * ((E + kRE - 1) / kRE);
  // slice d (in 64-wide chunks, a divisor of d/64) until the grid covers the
  // GPU's CTA slots about a few times over (each slice adds one atomic add
  // per logit)
  const int nc = d / kRK;
  const int target = (big ? kApproxWavesBig : 6) * n_sm;
  int slices = 1;
  for (int c = 1; c <= nc; ++c)
    if (nc % c == 0) {
      slices = c;
      if (tiles * c >= target) break;
    }
  // approx is all zeros here: zeroed when allocated, and k_pf_route zeroes what it reads
  const dim3 grid((T + rt - 1) / rt, (E + kRE - 1) / kRE, slices);
  cudaError_t e = big ? launch_chain(k_pf_logits_approx<8>, grid, dim3(256), 0, s, x_bf, router_w, T, d, E, d / slices,
                                     approx)
                      : launch_chain(k_pf_logits_approx<4>, grid, dim3(256), 0, s, x_bf, router_w, T, d, E, d / slices,
                                     approx);
  if (e != cudaSuccess) return e;
  // tokens per CTA: eight, or fewer when that leaves SMs idle
  const int tpc = std::max(1, std::min(8, (T + n_sm - 1) / n_sm));
  if (tpc == 1)
    return launch_chain(k_pf_route<kRouteChunks>, dim3((T + tpc - 1) / tpc), dim3(256), 0, s, x_bf, router_w, approx, xn2, wn2, xmax,
                        wmax, bias, T, d, E, k, ids, gates, dbg_ids, dbg_gates, dbg_logits, tpc, err);
  return launch_chain(k_pf_route<4>, dim3((T + tpc - 1) / tpc), dim3(256), 0, s, x_bf, router_w, approx, xn2, wn2, xmax,
                      wmax, bias, T, d, E, k, ids, gates, dbg_ids, dbg_gates, dbg_logits, tpc, err);
}

cudaError_t launch_pf_plan(const int32_t* ids, int P, int E, int tile, int32_t* cnt, int32_t* row_pair,
                           int32_t* items, int32_t* n_items, cudaStream_t s) {
  // small pair lists: one launch, each CTA counting them all itself
  const int count_here = P <= 4096 ? 1 : 0;
  if (!count_here) {
    const cudaError_t e = launch_chain(k_pf_count, dim3(E), dim3(256), 0, s, ids, P, cnt);
    if (e != cudaSuccess) return e;
  }
  return launch_chain(k_pf_scatter, dim3(E), dim3(256), 0, s, ids, P, E, cnt, tile, row_pair, items, n_items,
                      count_here);
}

cudaError_t launch_pf_combine(const float* ys, const float* ytok, const float* gates, const uint16_t* hin,
                              uint16_t* hout, float* y_last, float* dbg_y, int T, int d, int k, cudaStream_t s) {
  const auto al = [](const void* q, uintptr_t a) { return (reinterpret_cast<uintptr_t>(q) & (a - 1)) == 0; };
  // four rows per thread from 256 tokens on (small batches want the CTAs)
  if (T >= 256 && d % 4 == 0 && al(ys, 16) && al(ytok, 16) && al(hin, 8) && al(hout, 8) && al(y_last, 16) &&
      al(dbg_y, 16))
    return launch_chain(k_pf_combine, dim3(T, (d + 1023) / 1024), dim3(256), 0, s, ys, ytok, gates, hin, hout, y_last,
                        dbg_y, d, k);
  return launch_chain(k_pf_combine1, dim3(T, (d + 255) / 256), dim3(256), 0, s, ys, ytok, gates, hin, hout, y_last,
                      dbg_y, d, k);
}

cudaError_t launch_pf_gather(const uint16_t* x16, const int32_t* row_pair, int P, int d, int k, uint16_t* xp,
                             cudaStream_t s) {
  return launch_chain(k_pf_gather, dim3((P + 7) / 8), dim3(256), 0, s, x16, row_pair, P, d, k, xp);
}

bool g_chain_pdl = false;

}  // namespace moe
